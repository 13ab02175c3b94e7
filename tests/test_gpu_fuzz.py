"""Seeded random geometries through the whole step, bit-exact against the oracle.

Each case draws a cache geometry and a list structure and runs all five calls:
- geometry: layout pair (separate/separate, latent/latent, or any mix of blocks-first and
  kv-first), block sizes, heads and head dims, an optional head slice;
- an optional remap onto another block size and row offset;
- the run cap, and staging in HBM or in pinned host memory;
- lists: fragmented id queues, empty requests, requests sharing a prefix of block ids (prefix
  caching: the shared blocks are read more than once), new tokens at random positions of each
  request's own blocks.
The presets cover the configurations of the pages; this covers the combinations between
them.  Two more fuzzes drive the builder alone (lists up to 120K entries) and the prefix hash
(block sizes 1 to 700) against the oracle.  Every output is compared: slots, run records, the staging buffer, the source cache
after the token write and the destination cache after unpack.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from tests import gpu_support as G
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()


MAX_REQS, MAX_BLOCKS_PER_REQ = 5, 24


def _geom(layout, bs, row, num_blocks):
    """A geometry of `row` bytes per token row (a multiple of 16)."""
    if layout == "mla":
        return W.CacheGeom("mla", num_blocks, bs, 1, row // 2)
    return W.CacheGeom(layout, num_blocks, bs, row // 16, 8)


def fuzz_workload(seed: int) -> tuple:
    rng = np.random.default_rng(seed)
    two_planes = bool(rng.integers(0, 2))
    if two_planes:
        src_layout, dst_layout = rng.choice(["blocks_first", "kv_first"], size=2)
    else:
        src_layout = dst_layout = str(rng.choice(["separate", "mla"]))
    bs = int(rng.choice([1, 2, 3, 8, 16, 32]))
    head_dim = int(rng.choice([8, 16, 24, 64, 128]))
    heads = 1 if src_layout == "mla" else int(rng.integers(1, 5))
    row = heads * head_dim * 2
    slice_off, slice_bytes = 0, 0
    if heads > 1 and rng.random() < 0.5:
        h0 = int(rng.integers(0, heads))
        hn = int(rng.integers(1, heads - h0 + 1))
        slice_off, slice_bytes = h0 * head_dim * 2, hn * head_dim * 2
    moved = slice_bytes or row
    src_blocks = MAX_REQS * MAX_BLOCKS_PER_REQ + int(rng.integers(4, 64))
    if rng.random() < 0.5:  # whole blocks onto the same geometry (a head slice keeps only that slice)
        dst_bs, dst_row, dst_off = bs, moved, 0
    else:  # token-granular remap: another block size, the slice somewhere inside a wider row
        dst_bs = int(rng.choice([1, 2, 4, 8, 16, 32]))
        extra = 16 * int(rng.integers(0, 4))
        dst_row, dst_off = moved + extra, 16 * int(rng.integers(0, extra // 16 + 1))
    dst_blocks = -(-MAX_REQS * MAX_BLOCKS_PER_REQ * bs // dst_bs) + int(rng.integers(2, 32))
    wl = W.Workload(f"fuzz{seed}", 100 + seed, "tiny", n_layers=int(rng.integers(1, 4)),
                    src=_geom(str(src_layout), bs, row, src_blocks),
                    dst=_geom(str(dst_layout), dst_bs, dst_row, dst_blocks),
                    slice_off=slice_off, slice_bytes=slice_bytes, dst_slice_off=dst_off)
    cap = [None, 0, 1, 2, 5, 16][int(rng.integers(0, 6))]
    return wl, cap, rng


def fuzz_host_stage(seed: int) -> bool:
    """A quarter of the cases stage in pinned host memory (the spill target) instead of HBM."""
    return seed % 4 == 3


def fuzz_case(wl: W.Workload, rng) -> W.Case:
    bs = wl.src.block_size
    n = int(rng.integers(1, MAX_REQS + 1))
    counts = [int(rng.integers(0, MAX_BLOCKS_PER_REQ + 1)) for _ in range(n)]
    if n > 1 and rng.random() < 0.5:
        counts[int(rng.integers(0, n))] = 0  # an empty request
    q = W.fragmented_queue(rng, wl.src.num_blocks, int(rng.integers(1, 9)), float(rng.random()))
    src_lists = [list(l) for l in W.pop_lists(q, counts)]
    # prefix caching: some requests start with request 0's first blocks (shared source ids)
    shared = [0] * n
    if n > 1 and counts[0] > 0 and rng.random() < 0.3:
        for r in range(1, n):
            if counts[r] > 0 and rng.random() < 0.5:
                k = int(rng.integers(1, min(counts[0], counts[r]) + 1))
                src_lists[r][:k] = src_lists[0][:k]
                shared[r] = k
    off, ids = W.csr(src_lists)
    if wl.equal_geometry:
        dst_counts = counts
    else:
        dst_counts = [W.blocks_for(c * bs, wl.dst.block_size) for c in counts]
    qd = W.fragmented_queue(rng, wl.dst.num_blocks, int(rng.integers(1, 9)), float(rng.random()))
    doff, dids = W.csr(W.pop_lists(qd, dst_counts))
    width = max(1, max(counts))
    table = np.full((n, width), -1, dtype=np.int32)
    for r, l in enumerate(src_lists):
        table[r, :len(l)] = l
    token_req, token_pos = [], []
    for r, c in enumerate(counts):
        own = (c - shared[r]) * bs  # new tokens only in the request's own blocks: slots stay distinct
        if own <= 0:
            continue
        k = int(rng.integers(0, min(6, own) + 1))
        pos = shared[r] * bs + rng.choice(own, size=k, replace=False)
        token_req += [r] * k
        token_pos += [int(p) for p in pos]
    tr = np.asarray(token_req, dtype=np.int32) if token_req else None
    tp = np.asarray(token_pos, dtype=np.int32) if token_pos else None
    return W.Case(wl, off, ids, doff, dids, table if tr is not None else None, tr, tp,
                  req_tokens=np.asarray([c * bs for c in counts], dtype=np.int32))


@pytest.mark.parametrize("seed", range(400))
def test_fuzz_step_matches_oracle(seed):
    wl, cap, rng = fuzz_workload(seed)
    case = fuzz_case(wl, rng)
    src, dst, new = G.host_inputs(wl, case, seed=seed + 5000)
    host_stage = fuzz_host_stage(seed)
    gpu = G.run_gpu(wl, case, src, dst, new, max_run_blocks=cap, host_stage=host_stage)
    ora = G.run_oracle(wl, case, src, dst, new, gpu["max_run_blocks"])
    what = (f"seed {seed}: {wl.src.layout}->{wl.dst.layout} bs {wl.src.block_size}->{wl.dst.block_size} "
            f"row {wl.src.row_bytes}->{wl.dst.row_bytes} slice {wl.slice_off}+{wl.moved_slice}@{wl.dst_slice_off} "
            f"layers {wl.n_layers} cap {cap} blocks {case.n_blocks} tokens {case.n_tokens} host stage {host_stage}")
    G.compare(gpu, ora, what)


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_builder_matches_oracle(seed):
    """Random lists from 1 to 120K entries, across the single-CTA / look-back boundary and many
    look-back tiles: request count and lengths, id contiguity, destination ids, the cap, and the
    workspace or static entry point."""
    rng = np.random.default_rng(10_000 + seed)
    n = int(rng.choice([int(rng.integers(1, 6000)), int(rng.integers(5000, 12000)), int(rng.integers(1, 120_000))]))
    lens, left = [], n
    while left > 0:
        k = int(min(left, rng.integers(0, max(2, n // int(rng.integers(1, 64)) + 2))))
        lens.append(k)
        left -= k
    q = W.fragmented_queue(rng, n + int(rng.integers(0, 50)), int(rng.integers(1, 40)), float(rng.random()))
    off, ids = W.csr(W.pop_lists(q, lens))
    dids = W.fragmented_queue(rng, n + 9, int(rng.integers(1, 40)), float(rng.random()))[:n].astype(np.int32)
    cap = int(rng.choice([0, 1, 2, 3, 7, 32, 1000]))
    with_dst = bool(rng.integers(0, 2))
    builder = K.kv_build_xfer_list_static if rng.integers(0, 2) else K.kv_build_xfer_list
    x = builder(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda(),
                torch.from_numpy(dids).cuda() if with_dst else None, cap)
    torch.cuda.synchronize()
    got = x.host()
    want = oracle.build_xfer_list(off, ids, dids if with_dst else None, cap)
    assert got["count"] == want["req"].shape[0]
    for key in want:
        np.testing.assert_array_equal(got[key], want[key], err_msg=f"{key}: n {n} cap {cap} dst {with_dst}")
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_hashes_match_oracle(seed):
    """Random token batches: block sizes 1 to 700, up to 39 requests of any length, any token
    values and seed; both device paths."""
    rng = np.random.default_rng(20_000 + seed)
    bs = int(rng.choice([1, 2, 3, 5, 16, 17, 64, 80, 512, 700]))
    lens = rng.integers(0, bs * int(rng.integers(1, 40)) + 1, size=int(rng.integers(1, 40)))
    toks = [rng.integers(-2 ** 31, 2 ** 31, size=int(l), dtype=np.int64).astype(np.int32) for l in lens]
    off, flat = W.csr(toks)
    hseed = int(rng.integers(0, 2 ** 63))
    want_o, want = oracle.block_hashes(off, flat, bs, hseed)
    for ws in ("auto", None):
        o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(flat).cuda(), bs, hseed, workspace=ws)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(o.cpu().numpy(), want_o)
        np.testing.assert_array_equal(h[:int(want_o[-1])].cpu().numpy().view(np.uint64), want, err_msg=f"ws {ws}")
    assert K.kv_get_last_error() == 0


def fuzz_write_case(seed: int):
    """A random token write: geometry (any layout, block sizes 1-32, 1-4 heads of 8-200 elements,
    so rows of 1 to 50 chunks and both row kernels), 1-3 layers, a block table with holes, tokens
    at distinct slots plus a few invalid ones, and the batch size (one token to several passes)."""
    rng = np.random.default_rng(30_000 + seed)
    layout = str(rng.choice(["separate", "blocks_first", "kv_first", "mla"]))
    bs = int(rng.choice([1, 2, 3, 8, 16, 32]))
    hd = int(rng.choice([8, 16, 24, 64, 72, 128, 136, 200]))
    heads = 1 if layout == "mla" else int(rng.integers(1, 5))
    n_reqs, width = int(rng.integers(1, 6)), int(rng.integers(1, 9))
    nb = n_reqs * width + int(rng.integers(1, 16))
    g = W.CacheGeom(layout, nb, bs, 1, heads * hd) if layout == "mla" else W.CacheGeom(layout, nb, bs, heads, hd)
    table = rng.permutation(nb)[:n_reqs * width].astype(np.int32).reshape(n_reqs, width)
    table[rng.random(table.shape) < 0.1] = -1  # holes
    # distinct (request, position) pairs, so distinct slots; some invalid requests or positions
    pairs = [(r, p) for r in range(n_reqs) for p in range(width * bs)]
    T = int(rng.integers(1, min(len(pairs), int(rng.choice([8, 64, 4000]))) + 1))
    pick = rng.choice(len(pairs), size=T, replace=False)
    req = np.array([pairs[i][0] for i in pick], dtype=np.int32)
    pos = np.array([pairs[i][1] for i in pick], dtype=np.int32)
    bad = rng.random(T) < 0.05
    req[bad & (rng.random(T) < 0.5)] = n_reqs
    pos[bad & (req < n_reqs)] = width * bs + int(rng.integers(0, 3))
    return rng, g, int(rng.integers(1, 4)), table, req, pos, bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(80))
def test_fuzz_write_tokens_match_oracle(seed):
    """kv_write_tokens on random geometries and batches == the oracle's slot_mapping +
    reshape_and_cache: every cache tensor, slot_out when given, and the error bits."""
    rng, g, layers, table, req, pos, with_slot_out = fuzz_write_case(seed)
    T = req.shape[0]
    nt = layers * g.tensors_per_layer
    src = W.host_cache_tensors(g, nt, rng)
    new = [W.normal_bf16_bytes(rng, T * g.row_bytes // 2).reshape(T, g.row_bytes // 2) for _ in range(nt * g.n_planes)]
    s_dev = W.to_device_bf16(src, "cuda")
    n_dev = [x.reshape(G._new_shape(g, T)) for x in W.to_device_bf16(new, "cuda")]
    cache = K.PagedCache.from_tensors(s_dev, g.layout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((T,), -7, dtype=torch.int64, device="cuda") if with_slot_out else None
    K.kv_get_last_error(clear=True)
    K.kv_write_tokens(cache, n_dev, t(table), t(req), t(pos), out)
    torch.cuda.synchronize()
    err = K.kv_get_last_error(clear=True)
    want_slot, n_bad = oracle.slot_mapping(table, req, pos, g.block_size)
    assert ((err & K.KV_DERR_TABLE) != 0) == (n_bad > 0), f"error word {err:#x}, {n_bad} invalid tokens"
    assert (err & ~K.KV_DERR_TABLE) == 0, f"error word {err:#x}"
    if out is not None:
        np.testing.assert_array_equal(out.cpu().numpy(), want_slot)
    sc = H.ora_cache(g, [a.copy() for a in src])
    assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], want_slot) == 0
    what = f"seed {seed}: {g.layout} bs {g.block_size} row {g.row_bytes} planes {g.n_planes} T {T} tensors {nt}"
    for a, b in zip(s_dev, sc.tensors):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b, err_msg=what)
