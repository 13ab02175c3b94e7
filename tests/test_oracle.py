"""Pins of the CPU oracle against what the pages and plain mathematics fix.

Nothing here compares the oracle with itself: each pin checks it against a
hand-worked value from the pages' drawing, a library routine (numpy advanced
indexing, the pages' own `layer[block_ids]` gather), a closed-form invariant or
the independent brute-force enumeration in oracle/brute.py.  The mutation test
at the end plants plausible mistakes in a copy of the oracle's C source and
checks that every one of them fails at least one pin.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from oracle import brute
from paged_kv_cache_81_gb300 import workloads as W
from tests import helpers as H

LAYOUTS = ("separate", "blocks_first", "kv_first", "mla")


def natural_rows(geom: W.CacheGeom, tensor: np.ndarray) -> np.ndarray:
    """[num_blocks, planes, bs, row_bytes] copy of a tensor, from the pages' layer shapes."""
    nb, bs, row = geom.num_blocks, geom.block_size, geom.row_bytes
    b = tensor.reshape(-1).view(np.uint8)
    if geom.layout == "blocks_first":  # (num_blocks, 2, bs, H, D)
        return b.reshape(nb, 2, bs, row).copy()
    if geom.layout == "kv_first":  # (2, num_blocks, bs, H, D)
        return np.moveaxis(b.reshape(2, nb, bs, row), 0, 1).copy()
    return b.reshape(nb, 1, bs, row).copy()  # separate K or V, or MLA latent


def small_geom(layout, nb=7, bs=4, heads=2, head_dim=8):
    if layout == "mla":
        return W.CacheGeom("mla", nb, bs, 1, heads * head_dim)
    return W.CacheGeom(layout, nb, bs, heads, head_dim)


# ---------------------------------------------------------------------------
# pins (each takes the oracle library so the mutation test can swap it)
# ---------------------------------------------------------------------------
def pin_slot_golden(lib):
    for case, bs, table, pos, want in H.read_slot_golden():
        got, bad = oracle.slot_mapping(np.array([table], np.int32), [0], [pos], bs, lib=lib)
        assert got[0] == want, (case, bs, table, pos, got[0], want)
        assert bad == (1 if want < 0 else 0)


def pin_slot_brute(lib):
    rng = np.random.default_rng(7)
    for bs in (1, 2, 3, 16):
        nb, R, M = 40, 5, 6
        table = np.stack([rng.permutation(nb)[:M] for _ in range(R)]).astype(np.int32)
        T = 60
        req = rng.integers(0, R, T).astype(np.int32)
        pos = rng.integers(0, M * bs, T).astype(np.int32)
        got, bad = oracle.slot_mapping(table, req, pos, bs, lib=lib)
        assert bad == 0
        want = brute.slot_mapping(table, req, pos, nb, bs)
        np.testing.assert_array_equal(got, want)


def pin_reshape_indexing(lib):
    for layout in LAYOUTS:
        g = small_geom(layout)
        nt = 2
        tensors = H.random_cache(g, nt, seed=11)
        before = [natural_rows(g, t) for t in tensors]
        rng = np.random.default_rng(12)
        T = 13
        slots = rng.choice(g.num_blocks * g.block_size, size=T, replace=False).astype(np.int64)
        slots[[2, 9]] = -1  # padding tokens
        new = H.random_rows(T, g.row_bytes, nt * g.n_planes, seed=13)
        c = H.ora_cache(g, tensors)
        assert oracle.reshape_and_cache(c, new, slots, lib=lib) == 0
        keep = slots >= 0
        for t in range(nt):
            # slots number the rows of a [num_blocks * bs] flattening of each plane
            want = before[t].transpose(1, 0, 2, 3).reshape(g.n_planes, -1, g.row_bytes).copy()
            for p in range(g.n_planes):
                want[p, slots[keep]] = new[t * g.n_planes + p][keep]
            got = natural_rows(g, c.tensors[t]).transpose(1, 0, 2, 3).reshape(g.n_planes, -1, g.row_bytes)
            np.testing.assert_array_equal(got, want, err_msg=layout)


def pin_pack_indexing(lib):
    """stage(t, r) == layer[block_ids] (or layer[:, block_ids] for kv-first), sliced per row."""
    for layout in LAYOUTS:
        g = small_geom(layout, nb=9)
        nt = 3
        tensors = H.random_cache(g, nt, seed=21)
        rng = np.random.default_rng(22)
        lists = [rng.permutation(g.num_blocks)[:k] for k in (3, 0, 5, 1)]
        off, ids = W.csr(lists)
        for s_off, s_len in ((0, g.row_bytes), (g.row_bytes // 2, g.row_bytes // 4)):
            stage = oracle.pack(H.ora_cache(g, tensors), off, ids, s_off, s_len, lib=lib)
            parts = []
            for t in range(nt):
                nat = tensors[t].reshape(-1).view(np.uint8)
                for l in lists:
                    if layout == "blocks_first":
                        sel = nat.reshape(g.num_blocks, 2, g.block_size, g.row_bytes)[l]
                    elif layout == "kv_first":
                        sel = np.moveaxis(nat.reshape(2, g.num_blocks, g.block_size, g.row_bytes)[:, l], 0, 1)
                    else:
                        sel = nat.reshape(g.num_blocks, g.block_size, g.row_bytes)[l]
                    parts.append(np.ascontiguousarray(sel[..., s_off:s_off + s_len]).reshape(-1))
            np.testing.assert_array_equal(stage, np.concatenate(parts), err_msg=f"{layout} {s_off}")


def pin_pack_brute(lib):
    case = W.make_case(W.TINY)
    g = W.TINY.src
    tensors = H.random_cache(g, W.TINY.n_tensors, seed=31)
    stage = oracle.pack(H.ora_cache(g, tensors), case.req_offsets, case.src_ids, lib=lib)
    views = [H.rows_view(g, t) for t in tensors]
    want = brute.pack(views, H.req_lists(case.req_offsets, case.src_ids), g.block_size, 0, g.row_bytes)
    np.testing.assert_array_equal(stage, want)


def pin_unpack_roundtrip(lib):
    """pack then unpack to the same ids: listed blocks restored, every other block untouched."""
    for layout in LAYOUTS:
        g = small_geom(layout, nb=11)
        nt = 2
        src = H.random_cache(g, nt, seed=41)
        dst = H.random_cache(g, nt, seed=42)
        dst_before = [natural_rows(g, t) for t in dst]
        rng = np.random.default_rng(43)
        perm = rng.permutation(g.num_blocks)
        lists = [perm[0:4], perm[4:4], perm[4:7]]
        off, ids = W.csr(lists)
        stage = oracle.pack(H.ora_cache(g, src), off, ids, lib=lib)
        dc = H.ora_cache(g, dst)
        assert oracle.unpack(dc, stage, off, off, ids, g.block_size, g.row_bytes, lib=lib) == 0
        listed = set(int(x) for x in ids)
        for t in range(nt):
            got, s_rows = natural_rows(g, dc.tensors[t]), natural_rows(g, src[t])
            for b in range(g.num_blocks):
                want = s_rows[b] if b in listed else dst_before[t][b]
                np.testing.assert_array_equal(got[b], want, err_msg=f"{layout} block {b}")


def pin_unpack_other_ids(lib):
    """Equal geometry: dst block dst_ids[i] receives src block src_ids[i]; the rest is untouched."""
    g = small_geom("blocks_first", nb=12)
    nt = 2
    src = H.random_cache(g, nt, seed=51)
    dst = H.random_cache(g, nt, seed=52)
    dst_before = [natural_rows(g, t) for t in dst]
    rng = np.random.default_rng(53)
    s_perm, d_perm = rng.permutation(g.num_blocks), rng.permutation(g.num_blocks)
    off, ids = W.csr([s_perm[:3], s_perm[3:8]])
    _, dids = W.csr([d_perm[:3], d_perm[3:8]])
    stage = oracle.pack(H.ora_cache(g, src), off, ids, lib=lib)
    dc = H.ora_cache(g, dst)
    assert oracle.unpack(dc, stage, off, off, dids, g.block_size, g.row_bytes, lib=lib) == 0
    pairs = dict(zip(dids.tolist(), ids.tolist()))
    for t in range(nt):
        got, s_rows = natural_rows(g, dc.tensors[t]), natural_rows(g, src[t])
        for b in range(g.num_blocks):
            want = s_rows[pairs[b]] if b in pairs else dst_before[t][b]
            np.testing.assert_array_equal(got[b], want)


def pin_unpack_remap_handworked(lib):
    """block_size 16 -> 64: four staged source blocks fill one destination block in order.

    Source list [5, 2, 7, 1, 3] (80 tokens) lands in destination list [4, 0]:
    dst block 4 slots 0-15 <- src 5, 16-31 <- src 2, 32-47 <- src 7, 48-63 <- src 1;
    dst block 0 slots 0-15 <- src 3; dst block 0 slots 16-63 keep their old bytes.
    """
    sg = W.CacheGeom("separate", 8, 16, 1, 8)  # 16-byte rows
    dg = W.CacheGeom("separate", 6, 64, 1, 8)
    src = H.random_cache(sg, 1, seed=61)
    dst = H.random_cache(dg, 1, seed=62)
    old = dst[0].reshape(-1).view(np.uint8).reshape(6, 64, 16).copy()
    s = src[0].reshape(-1).view(np.uint8).reshape(8, 16, 16)
    off, ids = W.csr([[5, 2, 7, 1, 3]])
    doff, dids = W.csr([[4, 0]])
    stage = oracle.pack(H.ora_cache(sg, src), off, ids, lib=lib)
    dc = H.ora_cache(dg, dst)
    assert oracle.unpack(dc, stage, off, doff, dids, 16, 16, lib=lib) == 0
    d = dc.tensors[0].reshape(-1).view(np.uint8).reshape(6, 64, 16)
    np.testing.assert_array_equal(d[4, 0:16], s[5])
    np.testing.assert_array_equal(d[4, 16:32], s[2])
    np.testing.assert_array_equal(d[4, 32:48], s[7])
    np.testing.assert_array_equal(d[4, 48:64], s[1])
    np.testing.assert_array_equal(d[0, 0:16], s[3])
    np.testing.assert_array_equal(d[0, 16:64], old[0, 16:64])
    for b in (1, 2, 3, 5):
        np.testing.assert_array_equal(d[b], old[b])


def pin_unpack_brute(lib):
    """Head slice plus block-size change (4 -> 8 and the non-multiple 4 -> 6) vs brute force.

    The last variant lands the slice in the upper half of a wider destination row
    (a TP 2 -> 1 merge)."""
    for dbs, dheads, d_off in ((8, 2, 0), (6, 2, 0), (8, 4, 16)):
        sg = W.CacheGeom("blocks_first", 10, 4, 4, 4)  # row 32 B: 4 heads of 8 B
        dg = W.CacheGeom("blocks_first", 9, dbs, dheads, 4)
        src = H.random_cache(sg, 2, seed=71)
        dst = H.random_cache(dg, 2, seed=72)
        dst_b = [t.copy() for t in dst]
        rng = np.random.default_rng(73)
        s_lists = [rng.permutation(10)[:k] for k in (3, 1, 2)]
        need = [-(-len(l) * 4 // dbs) for l in s_lists]
        dperm = rng.permutation(9)
        d_lists = [dperm[sum(need[:i]):sum(need[:i]) + need[i]] for i in range(3)]
        off, ids = W.csr(s_lists)
        doff, dids = W.csr(d_lists)
        stage = oracle.pack(H.ora_cache(sg, src), off, ids, 16, 16, lib=lib)
        dc = H.ora_cache(dg, dst)
        assert oracle.unpack(dc, stage, off, doff, dids, 4, 16, d_off, lib=lib) == 0
        views = [H.rows_view(dg, t) for t in dst_b]
        brute.unpack(views, stage, [len(l) for l in s_lists], d_lists, 4, dbs, 2, 16, d_off)
        for t in range(2):
            np.testing.assert_array_equal(dc.tensors[t], dst_b[t], err_msg=f"dst bs {dbs}")


def pin_xfer_golden(lib):
    for c in H.read_xfer_golden():
        off, ids = W.csr(c["src_lists"])
        dids = None if c["dst_lists"] is None else W.csr(c["dst_lists"])[1]
        got = oracle.build_xfer_list(off, ids, dids, c["cap"], lib=lib)
        rows = np.stack([got["req"], got["src_block"], got["dst_block"], got["n_blocks"],
                         got["stage_block"]], axis=1).tolist() if got["req"].size else []
        assert rows == c["runs"], (c["name"], rows)


def pin_xfer_random(lib):
    """Runs cover the list exactly, are maximal under the cap, and equal brute-force grouping."""
    rng = np.random.default_rng(81)
    for trial in range(40):
        q = W.fragmented_queue(rng, 300, int(rng.integers(1, 12)), float(rng.random()))
        counts = rng.integers(0, 25, size=int(rng.integers(1, 9)))
        lists = W.pop_lists(q, counts)
        dq = W.fragmented_queue(rng, 300, 6, 0.7) if trial % 2 else None
        dlists = W.pop_lists(dq, counts) if dq is not None else None
        cap = int(rng.choice([0, 1, 2, 3, 7]))
        off, ids = W.csr(lists)
        dids = None if dlists is None else W.csr(dlists)[1]
        got = oracle.build_xfer_list(off, ids, dids, cap, lib=lib)
        n = got["n_blocks"]
        assert int(n.sum()) == ids.shape[0]
        if cap:
            assert n.size == 0 or n.max() <= cap
        # expansion reproduces the lists
        exp = np.concatenate([np.arange(s, s + k) for s, k in zip(got["src_block"], n)]) if n.size else ids[:0]
        np.testing.assert_array_equal(exp, ids)
        np.testing.assert_array_equal(got["stage_block"], np.concatenate([[0], np.cumsum(n)[:-1]]) if n.size else [])
        # maximality: adjacent runs in one request that could merge only where the cap was hit
        for k in range(1, n.size):
            if got["req"][k] == got["req"][k - 1] and got["src_block"][k] == got["src_block"][k - 1] + n[k - 1] \
                    and (dids is None or got["dst_block"][k] == got["dst_block"][k - 1] + n[k - 1]):
                assert cap and n[k - 1] == cap
        want = brute.xfer_runs(lists, dlists, cap)
        rows = np.stack([got["req"], got["src_block"], got["dst_block"], n, got["stage_block"]], axis=1).tolist() \
            if n.size else []
        assert rows == want


def pin_clip_golden(lib):
    for c in H.read_clip_golden():
        off, ids = W.csr([c["ids"]])
        o, got = oracle.clip_block_lists(off, ids, [c["n"]], c["window"], c["bs"], lib=lib)
        assert got.tolist() == c["want"], c
        assert o.tolist() == [0, len(c["want"])]


def pin_clip_brute(lib):
    """The blocks holding the last `window` tokens, found by enumerating block filling."""
    rng = np.random.default_rng(91)
    for trial in range(60):
        bs = int(rng.choice([1, 2, 3, 16]))
        R = int(rng.integers(1, 6))
        lens = rng.integers(0, 9, size=R)
        perm = rng.permutation(200)
        lists = W.pop_lists(perm, lens)
        n_tok = [int(rng.integers(0, l * bs + 1)) for l in lens]
        window = int(rng.choice([0, 1, 3, 5, 17, 1000]))
        off, ids = W.csr(lists)
        o, got = oracle.clip_block_lists(off, ids, n_tok, window, bs, lib=lib)
        want = []
        for l, n in zip(lists, n_tok):
            slots = brute.token_slots(l, n, 200, bs)
            first = max(0, n - window) if window > 0 else 0
            seen = []
            for s_ in slots[first:]:
                b = int(np.unravel_index(s_, (200, bs))[0])
                if b not in seen:
                    seen.append(b)
            want.extend(seen)
        assert got.tolist() == want, (bs, window, n_tok, lists)
        assert o[-1] == len(want)


def pin_fnv_vectors(lib):
    for data, want in H.read_fnv_golden():
        assert oracle.fnv1a64(data, lib=lib) == want, data


def pin_hash_chain(lib):
    """Chain structure: h0 = hash(seed ‖ block 0), h_i = hash(h_(i-1) ‖ block i), full blocks only;
    equal prefixes give equal hashes and a changed token changes its block's hash and every later one."""
    rng = np.random.default_rng(7)
    bs, seed = 4, 0x1234_5678_9ABC_DEF0
    a = rng.integers(0, 128000, size=23).astype(np.int32)  # 5 full blocks and a partial one
    b = a.copy()
    b[13] += 1  # inside block 3
    c = a[:9].copy()  # 2 full blocks and a partial
    off, toks = W.csr([a, b, c])
    o, h = oracle.block_hashes(off, toks, bs, seed, lib=lib)
    assert o.tolist() == [0, 5, 10, 12]  # floor(23/4), floor(23/4), floor(9/4)
    # explicit serialisation: parent as 8 little-endian bytes, then each token id as 4 little-endian bytes
    h0 = oracle.fnv1a64(np.array([seed], "<u8").tobytes() + a[0:4].astype("<u4").tobytes(), lib=lib)
    h1 = oracle.fnv1a64(np.array([h0], "<u8").tobytes() + a[4:8].astype("<u4").tobytes(), lib=lib)
    assert int(h[0]) == h0 and int(h[1]) == h1
    ha, hb, hc = h[0:5], h[5:10], h[10:12]
    np.testing.assert_array_equal(ha[:3], hb[:3])  # shared prefix, shared hashes
    assert all(int(x) != int(y) for x, y in zip(ha[3:], hb[3:]))  # the changed block and all after it
    np.testing.assert_array_equal(hc, ha[:2])
    _, h2 = oracle.block_hashes(off, toks, bs, seed + 1, lib=lib)
    assert all(int(x) != int(y) for x, y in zip(h, h2))  # another seed changes every hash


PINS = [pin_slot_golden, pin_slot_brute, pin_reshape_indexing, pin_pack_indexing, pin_pack_brute,
        pin_unpack_roundtrip, pin_unpack_other_ids, pin_unpack_remap_handworked, pin_unpack_brute,
        pin_xfer_golden, pin_xfer_random, pin_clip_golden, pin_clip_brute, pin_fnv_vectors, pin_hash_chain]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(None)


# ---------------------------------------------------------------------------
# rejection behaviour and workload pins
# ---------------------------------------------------------------------------
def test_reshape_range_and_duplicates():
    g = small_geom("separate")
    tensors = H.random_cache(g, 1, seed=91)
    before = tensors[0].copy()
    new = H.random_rows(3, g.row_bytes, 1, seed=92)
    c = H.ora_cache(g, tensors)
    nslots = g.num_blocks * g.block_size
    assert oracle.reshape_and_cache(c, new, np.array([0, nslots, nslots + 5]), ) == 2  # two out of range
    np.testing.assert_array_equal(natural_rows(g, c.tensors[0])[0, 0, 0], new[0][0])
    c2 = H.ora_cache(g, [before.copy()])
    assert oracle.reshape_and_cache(c2, new, np.array([4, 4, -1])) == -1  # duplicate slot
    np.testing.assert_array_equal(c2.tensors[0], before)


def test_unpack_rejects_bad_lists():
    g = small_geom("separate", nb=6)
    src = H.random_cache(g, 1, seed=93)
    dst = H.random_cache(g, 1, seed=94)
    before = dst[0].copy()
    off, ids = W.csr([[0, 1], [2]])
    stage = oracle.pack(H.ora_cache(g, src), off, ids)
    dc = H.ora_cache(g, dst)
    assert oracle.unpack(dc, stage, off, off, [3, 3, 4], g.block_size, g.row_bytes) == -1  # duplicate dst
    assert oracle.unpack(dc, stage, off, [0, 1, 2], [3, 4], g.block_size, g.row_bytes) == -1  # list too short
    assert oracle.unpack(dc, stage, off, off, [3, 4, 6], g.block_size, g.row_bytes) == -1  # out of range
    np.testing.assert_array_equal(dc.tensors[0], before)
    with pytest.raises(ValueError):
        oracle.pack(H.ora_cache(g, src), off, [0, 1, 6])
    with pytest.raises(ValueError):
        oracle.build_xfer_list([0, 2, 1], [0, 1, 2])  # decreasing offsets


def test_page_layout_sizes():
    """Drawing, per-layer tensor panel: 48 layer tensors of 147456 blocks, 1.125 GB each;
    "Paged kv cache": 16 slots per block; "scheduler(step)": 8 prompts -> 576 x 8 blocks."""
    g = W.PAGE.src
    assert g.tensor_shape() == (147456, 2, 16, 1, 128)
    assert g.block_payload_bytes == 8192
    assert g.tensor_bytes == 1_207_959_552 == int(1.125 * 2 ** 30)
    assert W.PAGE.n_tensors * g.tensor_bytes == 54 * 2 ** 30
    case = W.make_case(W.PAGE)
    assert case.n_reqs == 8 and case.n_blocks == 576 * 8 == 4608
    assert case.n_tokens == 8 * 9216 and 576 * 16 == 9216
    assert len(set(case.src_ids.tolist())) == 4608 and len(set(case.dst_ids.tolist())) == 4608


def test_other_presets():
    assert W.TINY.n_tensors == 4 and W.TINY.src.row_bytes == 256
    assert W.MID.n_tensors == 64 and W.MID.src.tensor_bytes == 512 * 2 ** 20
    assert W.MLA.src.row_bytes == (512 + 64) * 2 and W.MLA.src.tensor_shape() == (8192, 64, 576)
    assert W.ASYM.n_tensors == 80 and W.ASYM.slice_off == 1024 and W.ASYM.slice_bytes == 1024
    assert W.ASYM.dst.row_bytes == 1024 and not W.ASYM.equal_geometry and W.PAGE.equal_geometry

    t = W.make_case(W.TINY)
    assert t.n_reqs == 3 and all(1 <= l <= 100 for l in t.info["lens"]) and t.n_tokens == 24
    assert len(set(t.src_ids.tolist())) == t.n_blocks and len(set(t.dst_ids.tolist())) == t.n_blocks

    m = W.make_case(W.MID)
    assert m.n_blocks == 16 * 128
    runs = oracle.build_xfer_list(m.req_offsets, m.src_ids)
    frac = float(runs["n_blocks"][runs["n_blocks"] > 1].sum()) / m.n_blocks
    assert 0.3 < frac < 0.7, frac  # about half of the blocks sit in contiguous runs

    a = W.make_case(W.MLA)
    cur = a.block_table[np.arange(256), a.token_pos // 64]
    assert len(set(cur.tolist())) == 256  # distinct current blocks: no slot collides
    assert a.n_reqs == 32 and all(1024 <= l <= 32768 for l in a.info["lens"])

    s = W.make_case(W.ASYM)
    assert s.n_reqs == 24
    for r, l in enumerate(s.info["lens"]):
        assert s.req_offsets[r + 1] - s.req_offsets[r] == -(-l // 16)
        assert s.dst_req_offsets[r + 1] - s.dst_req_offsets[r] == -(-l // 64)


def test_cases_are_seeded():
    a, b = W.make_case(W.MID), W.make_case(W.MID)
    np.testing.assert_array_equal(a.src_ids, b.src_ids)
    np.testing.assert_array_equal(a.dst_ids, b.dst_ids)


def test_bf16_generator():
    rng = np.random.default_rng(5)
    u = W.normal_bf16_bytes(rng, 4096)
    import torch
    f = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).float()
    finite = torch.isfinite(f)
    assert 0.8 < float(f[finite].std()) < 1.2
    assert (~finite).sum() > 0 and (u == 0x8000).any()


# ---------------------------------------------------------------------------
# mutation test: every planted mistake must fail at least one pin
# ---------------------------------------------------------------------------
MUTANTS = [
    ("slot uses // for the offset", "+ position % block_size;", "+ position / block_size;"),
    ("slot drops the block factor", "slot[i] = (int64_t)block * block_size + position", "slot[i] = (int64_t)block + position"),
    ("reshape swaps block and offset", "int64_t block = slot[i] / c->block_size;", "int64_t block = slot[i] % c->block_size;"),
    ("plane stride dropped", "(int64_t)plane * c->plane_stride", "(int64_t)0 * c->plane_stride"),
    ("pack ignores slice offset", "row_addr(src, t, src_ids[i], p, o) + slice_off", "row_addr(src, t, src_ids[i], p, o)"),
    ("xfer treats equal ids as contiguous", "(src_ids[i] != src_ids[i - 1] + 1)", "(src_ids[i] != src_ids[i - 1] + 1 && src_ids[i] != src_ids[i - 1])"),
    ("xfer ignores request boundary", "int fresh = (i == req_offsets[r])", "int fresh = (i == 0)"),
    ("xfer cap off by one", "cur_len == max_run_blocks", "cur_len > max_run_blocks"),
    ("xfer ignores dst contiguity", "(dst_ids != NULL && dst_ids[i] != dst_ids[i - 1] + 1)", "(0)"),
    ("unpack uses src block size for dst slot", "j % dst->block_size) + dst_slice_off", "j % src_block_size) + dst_slice_off"),
    ("unpack wrong dst block index", "dst_ids[dst_req_offsets[r] + j / dst->block_size]", "dst_ids[dst_req_offsets[r] + q]"),
    ("unpack ignores dst slice offset", ") + dst_slice_off,\n", "),\n"),
    ("clip keeps one token too many", "? n - window : 0;", "? n - window - 1 : 0;"),
    ("clip drops the partial last block", "int64_t end = (n + block_size - 1) / block_size;", "int64_t end = n / block_size;"),
    ("clip ignores the window", "int64_t first = first_token / block_size;", "int64_t first = 0;"),
    ("hash is FNV-1 (multiply before xor)", "h ^= data[i];\n        h *= 0x100000001b3ull;", "h *= 0x100000001b3ull;\n        h ^= data[i];"),
    ("hash drops the parent", "buf[j] = (uint8_t)(parent >> (8 * j));", "buf[j] = 0;"),
    ("hash big-endian token bytes", "buf[8 + 4 * t + j] = (uint8_t)(id >> (8 * j));", "buf[8 + 4 * t + j] = (uint8_t)(id >> (8 * (3 - j)));"),
    ("hash covers the partial block", "for (int64_t b = 0; b < n / block_size; b++) {", "for (int64_t b = 0; b < (n + block_size - 1) / block_size; b++) {"),
]


_RUN_PINS = """
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import test_oracle as T
lib = oracle._get({so!r})
failed = []
for pin in T.PINS:
    try:
        pin(lib)
    except (AssertionError, ValueError, IndexError):
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    """Each mutant runs the pins in a child process: a planted index mistake may also
    corrupt memory, and a crash of the child counts as caught."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pagedkv_oracle.c"), encoding="utf-8").read()
    assert old in src, f"mutation site missing: {old!r}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new), encoding="utf-8")
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(mut)], check=True)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RUN_PINS.format(root=root, so=str(so))], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught mutant: {name}"
