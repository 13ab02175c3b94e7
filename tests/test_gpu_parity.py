"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit-exact.

Every output is compared element by element: slots, run records, the staging buffer,
the source cache after reshape_and_cache and the destination cache after unpack.
Cases: the five presets at reduced sizes (several builder tiles, ragged last
blocks), the Tiny preset in full, and edge cases (empty lists, capacity overflow,
out-of-range ids, padding slots, every cache layout and address mode).
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


PRESETS = [W.TINY, W.small(W.MID), W.small(W.PAGE), W.small(W.MLA), W.small(W.ASYM), W.small(W.PAGE_KV_FIRST)]


@pytest.mark.parametrize("wl", PRESETS, ids=lambda w: w.name)
def test_preset_parity(wl):
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 1000)
    gpu = G.run_gpu(wl, case, src, dst, new)
    ora = G.run_oracle(wl, case, src, dst, new, gpu["max_run_blocks"])
    G.compare(gpu, ora, wl.name)


@pytest.mark.parametrize("cap", [0, 1, 3])
@pytest.mark.parametrize("wl", [W.small(W.MID), W.small(W.ASYM)], ids=lambda w: w.name)
def test_run_cap_variants(wl, cap):
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=7)
    gpu = G.run_gpu(wl, case, src, dst, new, max_run_blocks=cap)
    ora = G.run_oracle(wl, case, src, dst, new, cap)
    G.compare(gpu, ora, f"{wl.name} cap {cap}")


def _builder_case(n_reqs, lens, rng, frag=(12, 0.6), n_ids=None):
    n_ids = n_ids or int(sum(lens)) + 7
    q = W.fragmented_queue(rng, n_ids, *frag)
    return W.csr(W.pop_lists(q, lens))


@pytest.mark.parametrize("n", [1, 64, 639, 640, 641, 2047, 2048, 2049, 4096, 5119, 5120, 5121, 6145, 20000, 100003])
@pytest.mark.parametrize("cap", [0, 1, 2, 7, 32])
@pytest.mark.parametrize("req_len", [3000, 1], ids=["long_requests", "one_block_requests"])
def test_builder_tiles(n, cap, req_len):
    """Runs across tile boundaries, long runs, empty requests, all cap variants.

    Lists of up to 640 entries go to the 128-thread single-CTA builder, up to 5120 to the
    1024-thread one (one tile each), longer ones to the look-back builder (tiles of 2048); the
    sizes straddle the three limits and the look-back tile edges.  Requests are up to 3000
    entries long, or one entry each (as many requests as entries)."""
    rng = np.random.default_rng(n * 31 + cap + req_len)
    lens = []
    left = n
    while left > 0:
        k = int(min(left, rng.integers(0, req_len + 1) if req_len > 1 else 1))
        lens.append(k)
        left -= k
    lens.insert(len(lens) // 2, 0)  # an empty request in the middle
    off, ids = _builder_case(len(lens), lens, rng, frag=(int(rng.integers(1, 64)), 0.8))
    dq = W.fragmented_queue(rng, n + 9, 40, 0.9)
    dids = dq[:n].astype(np.int32)
    for with_dst in (False, True):
        d = torch.from_numpy(dids).cuda() if with_dst else None
        x = K.kv_build_xfer_list(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda(), d, cap)
        torch.cuda.synchronize()
        got = x.host()
        want = oracle.build_xfer_list(off, ids, dids if with_dst else None, cap)
        assert got["count"] == want["req"].shape[0]
        for key in want:
            np.testing.assert_array_equal(got[key], want[key], err_msg=f"{key} n={n} cap={cap} dst={with_dst}")
    assert K.kv_get_last_error() == 0


def test_builder_empty_and_capacity():
    off = torch.zeros(4, dtype=torch.int32, device="cuda")
    ids = torch.zeros(0, dtype=torch.int32, device="cuda")
    x = K.kv_build_xfer_list(off, ids)
    torch.cuda.synchronize()
    assert x.host()["count"] == 0 and K.kv_get_last_error() == 0
    # more runs than capacity: the count is exact, the first `capacity` runs are written, the error bit is set
    o, s = W.csr([[5, 9, 11, 12, 3], [4]])
    want = oracle.build_xfer_list(o, s)
    out = K.XferList(2, "cuda", 0)
    K.kv_build_xfer_list(torch.from_numpy(o).cuda(), torch.from_numpy(s).cuda(), out=out)
    torch.cuda.synchronize()
    got = out.host()
    assert got["count"] == 5
    np.testing.assert_array_equal(got["src_block"], want["src_block"][:2])
    assert K.kv_get_last_error() & K.KV_DERR_CAPACITY


@pytest.mark.parametrize("n", [4, 70000])
def test_builder_bad_offsets_flagged(n):
    o = torch.tensor([0, 3, n + 1], dtype=torch.int32, device="cuda")  # claims n + 1 entries, list has n
    s = torch.arange(1, n + 1, dtype=torch.int32, device="cuda")
    K.kv_build_xfer_list(o, s)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_LIST


def test_slot_mapping_golden_and_invalid():
    """The hand-worked golden cases (padded to one table) and invalid tokens -> -1 + error bit."""
    for case, bs, table, pos, want in H.read_slot_golden():
        bt = torch.tensor([table], dtype=torch.int32, device="cuda")
        got = K.kv_slot_mapping(bt, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                torch.tensor([pos], dtype=torch.int32, device="cuda"), bs)
        torch.cuda.synchronize()
        assert int(got.item()) == want, (case, bs, table, pos)
        err = K.kv_get_last_error()
        assert bool(err & K.KV_DERR_TABLE) == (want < 0)
    bt = torch.tensor([[3, 7], [8, 9]], dtype=torch.int32, device="cuda")
    req = torch.tensor([0, 2, -1, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([1, 0, 0, -3], dtype=torch.int32, device="cuda")
    got = K.kv_slot_mapping(bt, req, pos, 2).cpu().numpy()
    np.testing.assert_array_equal(got, [7, -1, -1, -1])
    assert K.kv_get_last_error() & K.KV_DERR_TABLE


def test_slot_mapping_large_random():
    rng = np.random.default_rng(3)
    R, M, bs, nb = 300, 70, 16, 50000
    table = rng.integers(0, nb, size=(R, M)).astype(np.int32)
    T = 100000
    req = rng.integers(0, R, T).astype(np.int32)
    pos = rng.integers(0, M * bs, T).astype(np.int32)
    got = K.kv_slot_mapping(torch.from_numpy(table).cuda(), torch.from_numpy(req).cuda(),
                            torch.from_numpy(pos).cuda(), bs).cpu().numpy()
    want, bad = oracle.slot_mapping(table, req, pos, bs)
    assert bad == 0
    np.testing.assert_array_equal(got, want)
    assert K.kv_get_last_error() == 0


def _layout_case(layout, nb=40, bs=16, heads=4, hd=32, seed=0):
    g = W.CacheGeom(layout, nb, bs, heads, hd) if layout != "mla" else W.CacheGeom("mla", nb, bs, 1, heads * hd)
    rng = np.random.default_rng(seed)
    host = W.host_cache_tensors(g, 3, rng)
    perm = rng.permutation(nb)
    lists = [perm[0:5], perm[5:5], np.array([perm[5], perm[5] + 1 if perm[5] + 1 < nb else perm[6]]), perm[7:20]]
    off, ids = W.csr(lists)
    return g, host, off, ids


@pytest.mark.parametrize("layout", ["separate", "blocks_first", "kv_first", "mla"])
@pytest.mark.parametrize("sl", [None, (32, 64)])
def test_pack_layouts(layout, sl):
    """Every layout and address mode: MERGED (dense), ROWS (kv-first planes, head slice)."""
    g, host, off, ids = _layout_case(layout, seed=W.LAYOUTS.index(layout) + 17)
    s_off, s_len = (0, g.row_bytes) if sl is None else sl
    dev = W.to_device_bf16(host, "cuda")
    cache = K.PagedCache.from_tensors(dev, layout)
    x = K.kv_build_xfer_list(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda(), None, 4)
    stage = K.kv_pack_blocks(cache, x, ids.shape[0], slice_off=s_off, slice_bytes=s_len)
    want = oracle.pack(H.ora_cache(g, host), off, ids, s_off, s_len)
    np.testing.assert_array_equal(stage.cpu().numpy(), want)
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("layout,heads,engine", [("kv_first", 1, "warp"), ("kv_first", 2, "tma"), ("kv_first", 8, "tma"),
                                                 ("separate", 1, "warp"), ("blocks_first", 1, "tma"),
                                                 ("blocks_first", 4, "tma")],
                         ids=["kv_first_2KiB_planes_spans_warp", "kv_first_4KiB_planes_spans_tma",
                              "kv_first_16KiB_planes_spans_tma", "separate_2KiB_blocks_merged_warp",
                              "blocks_first_4KiB_blocks_merged_tma", "blocks_first_16KiB_blocks_merged_tma"])
def test_copy_engine_layouts(layout, heads, engine):
    """Whole steps on both copy engines, against the oracle.  Contiguous spans (a whole block, or
    one plane of a kv-first block) of 4 KiB and more take the TMA bulk engine (SPANS: one bulk
    copy per plane of a block; MERGED: one per run), smaller spans the register-staged warp
    engine."""
    from dataclasses import replace
    g = W.CacheGeom(layout, 64, 16, heads, 64)
    span = g.block_payload_bytes // (g.n_planes if layout == "kv_first" else 1)
    assert (span >= 4 * 1024) == (engine == "tma")
    wl = replace(W.TINY, name=f"tma_{layout}", src=g, dst=g)
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 41)
    gpu = G.run_gpu(wl, case, src, dst, new)
    ora = G.run_oracle(wl, case, src, dst, new, gpu["max_run_blocks"])
    G.compare(gpu, ora, wl.name)


@pytest.mark.parametrize("layout,dst_layout,bs,dst_bs,head_dim,extra,engine", [
    ("separate", "separate", 16, 64, 128, 0, "tma"),          # 4 KiB staged blocks landing whole in 64-slot blocks
    ("blocks_first", "blocks_first", 16, 32, 128, 0, "tma"),  # two planes: a span per (staged block, plane)
    ("kv_first", "kv_first", 16, 64, 128, 0, "tma"),          # planes a whole cache apart
    ("blocks_first", "kv_first", 32, 64, 64, 0, "tma"),       # the two layer layouts of the drawing, mixed
    ("separate", "separate", 16, 64, 128, 32, "warp"),        # the slice inside a wider destination row
    ("separate", "separate", 16, 24, 128, 0, "warp"),         # 24 is not a multiple of 16: staged blocks straddle
    ("separate", "separate", 8, 32, 64, 0, "warp"),           # 8 x 128 B = 1 KiB spans: below the TMA engine's 4 KiB
], ids=["tma_1plane", "tma_2planes", "tma_kv_first", "tma_mixed_layouts", "warp_wider_row", "warp_straddle",
        "warp_small_span"])
def test_remap_engines(layout, dst_layout, bs, dst_bs, head_dim, extra, engine):
    """Unpack onto another block size on both copy engines, against the oracle.  A remap whose
    staged blocks land whole inside destination blocks (the destination block size a multiple of
    the staged one) on rows the slice fills takes the TMA engine when a (block, plane) span is 4 KiB
    or more; any other remap takes the warp engine's token-granular path."""
    from dataclasses import replace
    row = head_dim * 2
    src = W.CacheGeom(layout, 160, bs, 1, head_dim)
    dst = W.CacheGeom(dst_layout, 160 * bs // dst_bs + 8, dst_bs, 1, head_dim + extra // 2)
    span = bs * row
    assert ((span >= 4096 and dst_bs % bs == 0 and extra == 0) == (engine == "tma"))
    wl = replace(W.TINY, name=f"remap_{layout}_{bs}_{dst_bs}_{extra}", src=src, dst=dst,
                 dst_slice_off=16 if extra else 0)  # the slice 16 bytes into a wider destination row
    case = W.make_case(wl)
    srch, dsth, new = G.host_inputs(wl, case, seed=wl.seed + 53)
    gpu = G.run_gpu(wl, case, srch, dsth, new)
    ora = G.run_oracle(wl, case, srch, dsth, new, gpu["max_run_blocks"])
    G.compare(gpu, ora, wl.name)


def test_pack_unpack_strided_blocks():
    """BLOCKS mode: each block contiguous, blocks further apart than their size (a padded view)."""
    nb, bs, heads, hd = 30, 8, 2, 16
    rng = np.random.default_rng(5)
    full = [torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(nb, 2 * bs, heads, hd), dtype=np.int16)).cuda()
            for _ in range(2)]
    views = [f.view(torch.bfloat16)[:, :bs] for f in full]  # block_stride = 2 * bs * row
    cache = K.PagedCache.from_tensors(views, "separate")
    assert cache.block_stride == 2 * bs * heads * hd * 2
    off, ids = W.csr([[3, 4, 5, 9], [0, 1]])
    x = K.kv_build_xfer_list(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda(), None, 3)
    stage = K.kv_pack_blocks(cache, x, ids.shape[0])
    host = [v.cpu().view(torch.int16).numpy() for v in views]
    want = np.concatenate([np.concatenate([h[i].reshape(-1).view(np.uint8) for i in ids]) for h in host])
    np.testing.assert_array_equal(stage.cpu().numpy(), want)
    # unpack back into other blocks of the padded views: the padding rows must stay untouched
    before = [f.clone() for f in full]
    d_off, d_ids = W.csr([[10, 11, 12, 20], [21, 22]])
    x2 = K.kv_build_xfer_list(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda(),
                              torch.from_numpy(d_ids).cuda(), 3)
    K.kv_unpack_blocks(cache, stage, x2, ids.shape[0], bs)
    torch.cuda.synchronize()
    for f, b, h in zip(full, before, host):
        fh, bh = f.cpu().numpy(), b.cpu().numpy()
        np.testing.assert_array_equal(fh[:, bs:], bh[:, bs:])  # padding untouched
        for s_, d_ in zip(ids, d_ids):
            np.testing.assert_array_equal(fh[d_, :bs], h[s_])
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("dbs,dheads,d_off", [(64, 4, 0), (24, 4, 0), (16, 8, 512)])
def test_unpack_remap_variants(dbs, dheads, d_off):
    """Token-granular unpack: 16 -> 64, the non-multiple 16 -> 24, and a slice landing mid-row."""
    sg = W.CacheGeom("separate", 256, 16, 8, 64)  # 1 KiB rows
    dg = W.CacheGeom("separate", 200, dbs, dheads, 64)
    rng = np.random.default_rng(dbs)
    src = W.host_cache_tensors(sg, 2, rng)
    dst = W.host_cache_tensors(dg, 2, rng)
    lens = [37, 1, 130, 64]
    s_lists = W.pop_lists(rng.permutation(256).astype(np.int32), [-(-l // 16) for l in lens])
    need = [-(-len(l) * 16 // dbs) for l in s_lists]
    d_lists = W.pop_lists(rng.permutation(200).astype(np.int32), need)
    off, ids = W.csr(s_lists)
    doff, dids = W.csr(d_lists)
    s_off, s_len = 256, 512  # heads 2..5 of the source row
    dd = W.to_device_bf16(dst, "cuda")
    scache = K.PagedCache.from_tensors(W.to_device_bf16(src, "cuda"), "separate")
    dcache = K.PagedCache.from_tensors(dd, "separate")
    t = lambda a: torch.from_numpy(a).cuda()
    x = K.kv_build_xfer_list(t(off), t(ids), None, 2)
    stage = K.kv_pack_blocks(scache, x, ids.shape[0], slice_off=s_off, slice_bytes=s_len)
    K.kv_unpack_blocks(dcache, stage, x, ids.shape[0], 16, s_len, d_off, t(off), t(doff), t(dids))
    torch.cuda.synchronize()
    st = oracle.pack(H.ora_cache(sg, src), off, ids, s_off, s_len)
    np.testing.assert_array_equal(stage.cpu().numpy(), st)
    dh = [a.copy() for a in dst]
    assert oracle.unpack(H.ora_cache(dg, dh), st, off, doff, dids, 16, s_len, d_off) == 0
    for a, b in zip(dd, dh):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)
    assert K.kv_get_last_error() == 0


def test_reshape_padding_and_range():
    g = W.CacheGeom("blocks_first", 12, 4, 2, 32)
    rng = np.random.default_rng(9)
    host = W.host_cache_tensors(g, 2, rng)
    dev = W.to_device_bf16(host, "cuda")
    cache = K.PagedCache.from_tensors(dev, "blocks_first")
    T = 6
    new = [torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(T, 2, 32), dtype=np.int16)).cuda().view(
        torch.bfloat16) for _ in range(4)]
    slot = torch.tensor([5, -1, 47, 48, 0, 1000], dtype=torch.int64, device="cuda")  # 48 slots in the cache
    K.kv_reshape_and_cache(cache, new, slot)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_SLOT
    hc = [h.copy() for h in host]
    rows = [n.cpu().view(torch.int16).numpy().view(np.uint8).reshape(T, -1) for n in new]
    assert oracle.reshape_and_cache(H.ora_cache(g, hc), rows, np.array([5, -1, 47, -1, 0, -1])) == 0
    for a, b in zip(dev, hc):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


def test_out_of_range_run_skipped():
    """A run naming blocks past the cache is skipped and flagged; the other runs still land."""
    g = W.CacheGeom("separate", 16, 4, 1, 64)
    rng = np.random.default_rng(11)
    host = W.host_cache_tensors(g, 1, rng)
    cache = K.PagedCache.from_tensors(W.to_device_bf16(host, "cuda"), "separate")
    off, ids = W.csr([[2, 3], [15, 16], [7]])  # 15,16 runs past the 16-block cache
    x = K.kv_build_xfer_list(torch.from_numpy(off).cuda(), torch.from_numpy(ids).cuda())
    stage = K.kv_pack_blocks(cache, x, ids.shape[0])
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_BLOCK
    s = stage.cpu().numpy().reshape(5, -1)
    h = host[0].reshape(16, -1).view(np.uint8)
    np.testing.assert_array_equal(s[0], h[2])
    np.testing.assert_array_equal(s[1], h[3])
    np.testing.assert_array_equal(s[4], h[7])


def test_host_argument_errors():
    g = W.CacheGeom("separate", 8, 4, 1, 64)
    dev = W.device_cache(g, 1, "cuda", seed=1)
    cache = K.PagedCache.from_tensors(dev, "separate")
    x = K.kv_build_xfer_list(torch.zeros(2, dtype=torch.int32, device="cuda").index_fill_(0, torch.tensor([1], device="cuda"), 1),
                             torch.zeros(1, dtype=torch.int32, device="cuda"))
    with pytest.raises(K.KvError) as e:
        K.kv_pack_blocks(cache, x, 1, slice_off=8, slice_bytes=32)  # slice offset not 16-byte aligned
    assert e.value.status == K.KV_ERR_ALIGN
    with pytest.raises(K.KvError) as e:
        K.kv_pack_blocks(cache, x, 1, slice_off=64, slice_bytes=128)  # slice past the row
    assert e.value.status == K.KV_ERR_RANGE
    with pytest.raises(K.KvError) as e:
        K.kv_pack_blocks(cache, x, 1, stage=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == K.KV_ERR_RANGE
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("heads", [1, 4, 8], ids=["2KiB_blocks_warp_engine", "8KiB_blocks_tma_engine",
                                                   "16KiB_blocks_tma_engine"])
def test_run_past_the_staging_buffer_flagged(heads):
    """Runs built for four blocks, pack and unpack told the staging buffer holds three: the run
    staged past the end is skipped and flagged (KV_DERR_STAGE); the other runs still move."""
    g = W.CacheGeom("separate", 16, 16, heads, 64)  # heads * 128 B rows; 2, 8 or 16 KiB blocks
    rng = np.random.default_rng(31)
    src = W.to_device_bf16(W.host_cache_tensors(g, 1, rng), "cuda")
    dst = W.to_device_bf16(W.host_cache_tensors(g, 1, rng), "cuda")
    dst_before = dst[0].clone()
    scache, dcache = K.PagedCache.from_tensors(src, "separate"), K.PagedCache.from_tensors(dst, "separate")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    off, ids = W.csr([[3, 4], [9, 10]])
    dids = np.array([1, 2, 6, 7], dtype=np.int32)
    x = K.kv_build_xfer_list(t(off), t(ids), t(dids), 1)  # cap 1: one run per block, staged 0..3
    K.kv_get_last_error(clear=True)
    stage = K.kv_pack_blocks(scache, x, 3)
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) & K.KV_DERR_STAGE
    blk = g.block_payload_bytes
    s_bytes = src[0].view(torch.uint8).reshape(g.num_blocks, blk)
    np.testing.assert_array_equal(stage.cpu().numpy().reshape(3, blk), s_bytes[[3, 4, 9]].cpu().numpy())
    K.kv_unpack_blocks(dcache, stage, x, 3, g.block_size, g.row_bytes, 0)
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) & K.KV_DERR_STAGE
    want = dst_before.view(torch.uint8).reshape(g.num_blocks, blk).clone()
    want[[1, 2, 6]] = s_bytes[[3, 4, 9]]
    np.testing.assert_array_equal(dst[0].view(torch.uint8).reshape(g.num_blocks, blk).cpu().numpy(), want.cpu().numpy())


def test_empty_remap_step():
    """A remap step (another block size on the receiver) whose requests are all empty: every call
    succeeds and nothing is written, although the empty destination list reaches the library as a
    null pointer."""
    src_g, dst_g = W.CacheGeom("separate", 16, 4, 1, 64), W.CacheGeom("separate", 8, 8, 1, 64)
    wl = W.Workload("empty_remap", 95, "tiny", n_layers=1, src=src_g, dst=dst_g)
    assert not wl.equal_geometry
    z = np.zeros(3, dtype=np.int32)
    case = W.Case(wl, z, np.zeros(0, np.int32), z.copy(), np.zeros(0, np.int32),
                  req_tokens=np.zeros(2, np.int32))
    src, dst, new = G.host_inputs(wl, case, seed=96)
    gpu = G.run_gpu(wl, case, src, dst, new)
    ora = G.run_oracle(wl, case, src, dst, new, gpu["max_run_blocks"])
    G.compare(gpu, ora, "empty remap step")


@pytest.mark.parametrize("write", ["reshape", "write_tokens"])
@pytest.mark.parametrize("layout", ["separate", "blocks_first"])
def test_more_tensors_than_one_launch_carries(layout, write):
    """130 and 257 cache tensors: the token write, pack and unpack split into several launches
    (128 tensor bases per launch); the staging offsets of later launches must continue.  The
    token write is kv_reshape_and_cache, or kv_write_tokens through an identity block table
    (slot = position), whose slot_out must come back whole from the first launch alone."""
    for n_tensors in (130, 257):
        g = W.CacheGeom(layout, 24, 4, 1, 16)  # 32-byte rows, tiny tensors
        rng = np.random.default_rng(n_tensors)
        src = W.host_cache_tensors(g, n_tensors, rng)
        dst = W.host_cache_tensors(g, n_tensors, rng)
        lists = [rng.permutation(24)[:5], rng.permutation(24)[:3]]
        off, ids = W.csr(lists)
        dids = rng.permutation(24)[:8].astype(np.int32)  # distinct destination blocks
        T = 6
        slot = rng.choice(24 * 4, size=T, replace=False).astype(np.int64)
        new = [rng.integers(-2 ** 15, 2 ** 15, size=(T, 16), dtype=np.int16) for _ in range(n_tensors * g.n_planes)]
        s_dev, d_dev = W.to_device_bf16(src, "cuda"), W.to_device_bf16(dst, "cuda")
        scache = K.PagedCache.from_tensors(s_dev, layout)
        dcache = K.PagedCache.from_tensors(d_dev, layout)
        n_dev = [torch.from_numpy(x).cuda().view(torch.bfloat16).reshape(T, 1, 16) for x in new]
        if write == "reshape":
            K.kv_reshape_and_cache(scache, n_dev, torch.from_numpy(slot).cuda())
        else:
            table = torch.arange(24, dtype=torch.int32, device="cuda").reshape(1, 24)
            out = torch.full((T,), -7, dtype=torch.int64, device="cuda")
            K.kv_write_tokens(scache, n_dev, table, torch.zeros(T, dtype=torch.int32, device="cuda"),
                              torch.from_numpy(slot.astype(np.int32)).cuda(), out)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(out.cpu().numpy(), slot)
        t = lambda a: torch.from_numpy(a).cuda()
        x = K.kv_build_xfer_list(t(off), t(ids), t(dids), 2)
        stage = K.kv_pack_blocks(scache, x, ids.shape[0])
        K.kv_unpack_blocks(dcache, stage, x, ids.shape[0], 4)
        torch.cuda.synchronize()
        assert K.kv_get_last_error() == 0
        sh = [a.copy() for a in src]
        sc = H.ora_cache(g, sh)
        assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], slot) == 0
        want = oracle.pack(sc, off, ids)
        np.testing.assert_array_equal(stage.cpu().numpy(), want)
        dh = [a.copy() for a in dst]
        assert oracle.unpack(H.ora_cache(g, dh), want, off, off, dids, 4, g.row_bytes) == 0
        for a, b in zip(s_dev, sh):
            np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)
        for a, b in zip(d_dev, dh):
            np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


def test_remap_with_offsets_that_do_not_match_the_runs():
    """Unpack remap given source offsets that disagree with the runs (a request said to start past
    its runs): those runs are skipped and flagged, nothing is read or written out of place."""
    sg = W.CacheGeom("separate", 16, 4, 1, 64)  # 128-byte rows
    dg = W.CacheGeom("separate", 64, 1, 1, 64)  # destination block size 1
    rng = np.random.default_rng(12)
    src = W.host_cache_tensors(sg, 1, rng)
    dst = W.host_cache_tensors(dg, 1, rng)
    off, ids = W.csr([[3, 4], [9]])
    doff, dids = W.csr([list(range(0, 8)), list(range(8, 12))])  # 8 and 4 one-slot blocks
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    d_dev = W.to_device_bf16(dst, "cuda")
    scache = K.PagedCache.from_tensors(W.to_device_bf16(src, "cuda"), "separate")
    dcache = K.PagedCache.from_tensors(d_dev, "separate")
    x = K.kv_build_xfer_list(t(off), t(ids), None, 2)
    stage = K.kv_pack_blocks(scache, x, 3)
    bad_off = t([0, 3, 3])  # request 1 "starts" at entry 3, after its run at entry 2
    K.kv_unpack_blocks(dcache, stage, x, 3, 4, None, 0, bad_off, t(doff), t(dids))
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_DST_TABLE
    # request 0's run still lands in slots 0..7; the rest of the destination is untouched
    got = d_dev[0].cpu().view(torch.int16).numpy().view(np.uint16).reshape(64, -1)
    want = dst[0].reshape(64, -1).copy()
    st = stage.cpu().numpy().reshape(3 * 4, -1).view(np.uint16)
    want[0:8] = st[0:8]
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("wl", [W.small(W.PAGE), W.small(W.MID), W.small(W.ASYM)], ids=lambda w: w.name)
def test_staging_guard_canaries(wl):
    """Canary bytes before and after the staging region survive pack (both copy engines' paths)."""
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=99)
    scache = K.PagedCache.from_tensors(W.to_device_bf16(src, "cuda"), wl.src.layout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    cap = K.default_max_run_blocks(wl.src.n_planes * wl.src.block_size * wl.moved_slice)
    x = K.kv_build_xfer_list(t(case.req_offsets), t(case.src_ids), None, cap)
    n = G._stage_len(wl, case)
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    K.kv_pack_blocks(scache, x, case.n_blocks, buf[guard:guard + n], wl.slice_off, wl.moved_slice)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    b = buf.cpu().numpy()
    assert (b[:guard] == 0xA5).all() and (b[guard + n:] == 0xA5).all()
    want = oracle.pack(H.ora_cache(wl.src, src), case.req_offsets, case.src_ids, wl.slice_off, wl.moved_slice)
    np.testing.assert_array_equal(b[guard:guard + n], want)


@pytest.mark.parametrize("with_slot_out", [True, False], ids=["two_launches", "fused"])
@pytest.mark.parametrize("wl", [W.TINY, W.small(W.MLA), W.small(W.PAGE), W.small(W.PAGE_KV_FIRST)],
                         ids=lambda w: w.name)
def test_write_tokens_matches_oracle(wl, with_slot_out):
    """kv_write_tokens == oracle slot_mapping + reshape_and_cache: with slot_out (slot_mapping, then
    the row copy) and without (the slot lookup fused into the row copy)."""
    case = W.make_case(wl)
    src, _, new = G.host_inputs(wl, case, seed=wl.seed + 17)
    s_dev = W.to_device_bf16(src, "cuda")
    n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
    cache = K.PagedCache.from_tensors(s_dev, wl.src.layout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    slot = torch.full((case.n_tokens,), -7, dtype=torch.int64, device="cuda") if with_slot_out else None
    K.kv_get_last_error(clear=True)
    K.kv_write_tokens(cache, n_dev, t(case.block_table), t(case.token_req), t(case.token_pos), slot)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    want_slot, bad = oracle.slot_mapping(case.block_table, case.token_req, case.token_pos, wl.src.block_size)
    assert bad == 0
    if with_slot_out:
        np.testing.assert_array_equal(slot.cpu().numpy(), want_slot)
    sc = H.ora_cache(wl.src, [a.copy() for a in src])
    assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], want_slot) == 0
    for a, b in zip(s_dev, sc.tensors):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


@pytest.mark.parametrize("with_slot_out", [True, False], ids=["split", "fused"])
def test_write_tokens_large_batch(with_slot_out):
    """A 48-layer prefill of 8192 tokens through kv_write_tokens: slot_mapping and the row copy as
    two launches when it may write slot_out; without slot_out the fused kernel, several grid-stride
    passes per thread."""
    g = W.CacheGeom("blocks_first", 1024, 16, 1, 128)
    wl = W.Workload("write_large", 90, "page", n_layers=48, src=g, dst=g)
    rng = np.random.default_rng(91)
    ids = rng.choice(g.num_blocks, size=4 * 128, replace=False).astype(np.int32)
    table = ids.reshape(4, 128)
    token_req = np.repeat(np.arange(4, dtype=np.int32), 2048)
    token_pos = np.tile(np.arange(2048, dtype=np.int32), 4)
    src = W.host_cache_tensors(g, wl.n_tensors, rng)
    new = [W.normal_bf16_bytes(rng, 8192 * g.row_bytes // 2).reshape(8192, g.row_bytes // 2)
           for _ in range(wl.n_tensors * g.n_planes)]
    s_dev = W.to_device_bf16(src, "cuda")
    n_dev = [x.reshape(8192, g.heads, g.head_dim) for x in W.to_device_bf16(new, "cuda")]
    cache = K.PagedCache.from_tensors(s_dev, g.layout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    slot = torch.full((8192,), -7, dtype=torch.int64, device="cuda") if with_slot_out else None
    K.kv_get_last_error(clear=True)
    K.kv_write_tokens(cache, n_dev, t(table), t(token_req), t(token_pos), slot)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    want_slot, bad = oracle.slot_mapping(table, token_req, token_pos, g.block_size)
    assert bad == 0
    if with_slot_out:
        np.testing.assert_array_equal(slot.cpu().numpy(), want_slot)
    sc = H.ora_cache(g, [a.copy() for a in src])
    assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], want_slot) == 0
    for a, b in zip(s_dev, sc.tensors):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


@pytest.mark.parametrize("entry", ["reshape", "write_slot_out", "write"])
def test_decode_write_one_wave(entry):
    """A decode step of 256 tokens into 61 latent-layout layers (576 bf16 per row, 18 CTAs a layer:
    1098 CTAs, a wave and a tail on 152 SMs).  Padding tokens (slot -1), a table hole and a
    partial last CTA are included; every tensor is compared with the oracle's slot_mapping +
    reshape_and_cache, and slot_out when it is asked for."""
    g = W.CacheGeom("mla", 8, 64, 1, 576)
    nt, T = 61, 256
    rng = np.random.default_rng(95)
    table = rng.permutation(g.num_blocks).astype(np.int32).reshape(4, 2)
    table[3, 1] = -1  # a hole: tokens of request 3 past position 63 have no block
    token_req = rng.integers(0, 4, T).astype(np.int32)
    token_pos = np.empty(T, dtype=np.int32)
    for r in range(4):  # distinct positions per request, so slots are distinct
        k = int((token_req == r).sum())
        token_pos[token_req == r] = rng.choice(128, size=k, replace=False)
    want_slot, bad = oracle.slot_mapping(table, token_req, token_pos, g.block_size)
    src = W.host_cache_tensors(g, nt, rng)
    new = [W.normal_bf16_bytes(rng, T * g.row_bytes // 2).reshape(T, g.row_bytes // 2) for _ in range(nt)]
    s_dev = W.to_device_bf16(src, "cuda")
    n_dev = [x.reshape(T, 1, g.row_bytes // 2) for x in W.to_device_bf16(new, "cuda")]
    cache = K.PagedCache.from_tensors(s_dev, "mla")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    K.kv_get_last_error(clear=True)
    if entry == "reshape":
        slot = want_slot.copy()
        slot[::37] = -1  # padding tokens are skipped
        K.kv_reshape_and_cache(cache, n_dev, t(slot))
        torch.cuda.synchronize()
        assert K.kv_get_last_error() == 0
    else:
        assert bad > 0
        slot = want_slot
        out = torch.full((T,), -7, dtype=torch.int64, device="cuda") if entry == "write_slot_out" else None
        K.kv_write_tokens(cache, n_dev, t(table), t(token_req), t(token_pos), out)
        torch.cuda.synchronize()
        assert K.kv_get_last_error() & K.KV_DERR_TABLE
        if out is not None:
            np.testing.assert_array_equal(out.cpu().numpy(), want_slot)
    sc = H.ora_cache(g, [a.copy() for a in src])
    assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], slot) == 0
    for a, b in zip(s_dev, sc.tensors):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


@pytest.mark.parametrize("entry", ["reshape", "write_tokens", "fused"])
@pytest.mark.parametrize("layout,hd", [("separate", 136), ("blocks_first", 136), ("mla", 200), ("mla", 288),
                                       ("kv_first", 24), ("mla", 8)],
                         ids=["sep_17_chunks", "bf_2x17_chunks", "mla_25_chunks", "mla_36_chunks", "kvf_2x3_chunks",
                              "mla_1_chunk"])
def test_row_write_chunk_counts(layout, hd, entry):
    """Row writes whose chunk count per token (planes x 16-byte chunks of a row) does or does not
    divide a whole number of 256-thread CTAs within 16 CTAs: 17, 34 and 25 chunks take the general
    kernel, 36, 6 and 1 the token-strided one.  Token counts leave ragged tails; padding tokens
    (slot -1) are skipped.  Entries: kv_reshape_and_cache, kv_write_tokens with slot_out (two
    launches) and without (the fused kernel)."""
    g = W.CacheGeom(layout, 24, 8, 1, hd)
    rng = np.random.default_rng(hd + len(layout))
    src = W.host_cache_tensors(g, 3, rng)
    T = 70
    table = rng.permutation(g.num_blocks).astype(np.int32).reshape(3, 8)
    token_req = rng.integers(0, 3, T).astype(np.int32)
    token_pos = np.empty(T, dtype=np.int32)
    for r in range(3):
        k = int((token_req == r).sum())
        token_pos[token_req == r] = rng.choice(64, size=k, replace=False)
    want_slot, bad = oracle.slot_mapping(table, token_req, token_pos, g.block_size)
    assert bad == 0
    new = [W.normal_bf16_bytes(rng, T * g.row_bytes // 2).reshape(T, g.row_bytes // 2)
           for _ in range(3 * g.n_planes)]
    s_dev = W.to_device_bf16(src, "cuda")
    n_dev = [x.reshape(G._new_shape(g, T)) for x in W.to_device_bf16(new, "cuda")]
    cache = K.PagedCache.from_tensors(s_dev, layout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    K.kv_get_last_error(clear=True)
    slot = want_slot.copy()
    if entry != "reshape":
        out = torch.full((T,), -7, dtype=torch.int64, device="cuda") if entry == "write_tokens" else None
        K.kv_write_tokens(cache, n_dev, t(table), t(token_req), t(token_pos), out)
        torch.cuda.synchronize()
        if out is not None:
            np.testing.assert_array_equal(out.cpu().numpy(), want_slot)
    else:
        slot[::9] = -1
        K.kv_reshape_and_cache(cache, n_dev, t(slot))
        torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    sc = H.ora_cache(g, [a.copy() for a in src])
    assert oracle.reshape_and_cache(sc, [r.view(np.uint8) for r in new], slot) == 0
    for a, b in zip(s_dev, sc.tensors):
        np.testing.assert_array_equal(a.cpu().view(torch.int16).numpy().view(np.uint16), b)


def test_write_tokens_invalid_tokens():
    g = W.CacheGeom("separate", 8, 4, 1, 64)
    host = W.host_cache_tensors(g, 1, np.random.default_rng(2))
    dev = W.to_device_bf16(host, "cuda")
    cache = K.PagedCache.from_tensors(dev, "separate")
    table = torch.tensor([[1, 2], [3, -1]], dtype=torch.int32, device="cuda")
    req = torch.tensor([0, 1, 1, 5], dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, 2, 6, 0], dtype=torch.int32, device="cuda")  # 2nd ok, 3rd hits -1, 4th bad req
    rows = torch.arange(4 * 64, dtype=torch.int16, device="cuda").view(torch.bfloat16).reshape(4, 1, 64)
    slot = torch.empty(4, dtype=torch.int64, device="cuda")
    K.kv_write_tokens(cache, [rows], table, req, pos, slot)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_TABLE
    np.testing.assert_array_equal(slot.cpu().numpy(), [9, 14, -1, -1])
    got = dev[0].cpu().view(torch.int16).numpy().reshape(32, 64)
    want = host[0].view(np.int16).reshape(32, 64).copy()
    r = rows.view(torch.int16).cpu().numpy().reshape(4, 64)
    want[9], want[14] = r[0], r[1]
    np.testing.assert_array_equal(got, want)
