"""Full-size parity: each preset at its full size, in the launch configuration bench.py times.

For every preset the whole step runs once through the C ABI (TransferStep, default run
cap and copy engine, as in the benchmark).  Then:
  * index outputs (slots, the run list) are compared with the oracle in full;
  * three sampled cache tensors (first, last, one seeded pick) are recomputed by the oracle
    from host snapshots taken before the step and compared byte for byte: the source tensor
    after reshape_and_cache, its staging slice after pack, the destination tensor after unpack;
  * every tensor is checked on the device against properties that hold at any size: the
    staging equals torch advanced indexing of the source (the pages' layer[block_ids]), the
    destination blocks equal the staged ones, and every block or slot the step must not touch
    still holds its seeded fill (regenerated on the device);
  * then fresh rows go through kv_write_tokens (the fused call, with slot_out): its slots equal
    the oracle's, and every tensor's rows at those slots equal the fresh rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep
from tests import helpers as H

pytestmark = pytest.mark.gpu

FULL = [W.MID, W.PAGE, W.MLA, W.ASYM, W.PAGE_KV_FIRST]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()
    yield
    torch.cuda.empty_cache()


def rows_dev(t: torch.Tensor, g: W.CacheGeom) -> torch.Tensor:
    """[num_blocks, planes, bs, row_bytes] uint8 view of a device cache tensor (its natural layout)."""
    b = t.view(torch.uint8).reshape(-1)
    if g.layout == "blocks_first":
        return b.view(g.num_blocks, 2, g.block_size, g.row_bytes)
    if g.layout == "kv_first":
        return b.view(2, g.num_blocks, g.block_size, g.row_bytes).transpose(0, 1)
    return b.view(g.num_blocks, 1, g.block_size, g.row_bytes)


def regen(g: W.CacheGeom, seed: int, t: int, device) -> torch.Tensor:
    """Tensor t of W.device_cache(g, ..., seed) regenerated alone."""
    x = torch.empty(g.tensor_shape(), dtype=torch.bfloat16, device=device)
    return W.fill_random_(x, seed * 1000003 + t)


def needed_bytes(wl: W.Workload, case: W.Case) -> int:
    b = wl.n_tensors * wl.src.tensor_bytes
    if wl.kind != "mla":
        b += wl.n_tensors * wl.dst.tensor_bytes
    b += wl.n_tensors * case.n_blocks * wl.src.n_planes * wl.src.block_size * wl.moved_slice
    b += wl.n_tensors * wl.src.n_planes * case.n_tokens * wl.src.row_bytes
    return b + (4 << 30)


@pytest.mark.parametrize("wl", FULL, ids=lambda w: w.name)
def test_full_size(wl):
    dev = torch.device("cuda")
    case = W.make_case(wl)
    torch.cuda.empty_cache()
    if torch.cuda.mem_get_info()[0] < needed_bytes(wl, case):
        pytest.skip("not enough free device memory for the full-size preset")
    has_dst = wl.kind != "mla"
    seed = 4242 + wl.index
    src = W.device_cache(wl.src, wl.n_tensors, dev, seed=seed)
    dst = W.device_cache(wl.dst, wl.n_tensors, dev, seed=seed + 1) if has_dst else None
    new = W.new_token_rows(wl.src, wl.n_tensors, case.n_tokens, dev, seed=seed + 2)
    rng = np.random.default_rng(seed)
    sample = sorted({0, wl.n_tensors - 1, int(rng.integers(1, wl.n_tensors - 1))})
    snap = {t: (src[t].view(torch.uint8).cpu().numpy(), dst[t].view(torch.uint8).cpu().numpy() if has_dst else None)
            for t in sample}

    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, src, dst, new, device=dev)
    step.run()
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) == 0

    g, N = wl.src, case.n_blocks
    sl, s_off = wl.moved_slice, wl.slice_off
    # --- index outputs, whole, against the oracle ---------------------------
    slot = None
    if case.n_tokens:
        slot, bad = oracle.slot_mapping(case.block_table, case.token_req, case.token_pos, g.block_size)
        assert bad == 0
        np.testing.assert_array_equal(step.slot.cpu().numpy(), slot)
    equal = wl.equal_geometry and has_dst
    runs = oracle.build_xfer_list(case.req_offsets, case.src_ids, case.dst_ids if equal else None,
                                  step.max_run_blocks)
    got = step.xfer.host()
    assert got["count"] == runs["req"].shape[0]
    for k in runs:
        np.testing.assert_array_equal(got[k], runs[k], err_msg=k)

    per = N * g.n_planes * g.block_size * sl
    stage = step.stage[:wl.n_tensors * per]

    # --- sampled tensors, element by element, against the oracle ------------
    for t in sample:
        s_host, d_host = snap[t]
        sc = H.ora_cache(g, [s_host])
        if case.n_tokens:
            rows = [new[t * g.n_planes + p].reshape(case.n_tokens, -1).view(torch.uint8).cpu().numpy()
                    for p in range(g.n_planes)]
            assert oracle.reshape_and_cache(sc, rows, slot) == 0
            assert np.array_equal(src[t].view(torch.uint8).cpu().numpy().reshape(-1), sc.tensors[0].reshape(-1)), \
                f"tensor {t}: reshape_and_cache differs from the oracle"
        want_stage = oracle.pack(sc, case.req_offsets, case.src_ids, s_off, sl)
        got_stage = stage[t * per:(t + 1) * per].cpu().numpy()
        diff = np.flatnonzero(got_stage != want_stage)
        assert diff.size == 0, f"tensor {t}: staging differs at {diff.size} bytes"
        if has_dst:
            dc = H.ora_cache(wl.dst, [d_host])
            assert oracle.unpack(dc, want_stage, case.req_offsets, case.dst_req_offsets, case.dst_ids,
                                 g.block_size, sl, wl.dst_slice_off) == 0
            assert np.array_equal(dst[t].view(torch.uint8).cpu().numpy().reshape(-1), dc.tensors[0].reshape(-1)), \
                f"tensor {t}: unpack differs from the oracle"
        del sc, s_host, d_host
    snap.clear()

    # --- every tensor: properties on the device ------------------------------
    src_ids = torch.from_numpy(case.src_ids.astype(np.int64)).to(dev)
    if case.n_tokens:
        blk = torch.from_numpy(slot // g.block_size).to(dev)
        off = torch.from_numpy(slot % g.block_size).to(dev)
        written = torch.ones(g.num_blocks, g.block_size, dtype=torch.bool, device=dev)
        written[blk, off] = False  # True = slot untouched by reshape_and_cache
    if has_dst:
        d = wl.dst
        if equal:
            dst_ids = torch.from_numpy(case.dst_ids.astype(np.int64)).to(dev)
            keep = torch.ones(d.num_blocks, dtype=torch.bool, device=dev)
            keep[dst_ids] = False
        else:  # token-granular destination of every staged token
            db, ds = [], []
            for r in range(case.n_reqs):
                n_tok = int(case.req_offsets[r + 1] - case.req_offsets[r]) * g.block_size
                j = np.arange(n_tok)
                db.append(case.dst_ids[case.dst_req_offsets[r] + j // d.block_size])
                ds.append(j % d.block_size)
            db = torch.from_numpy(np.concatenate(db).astype(np.int64)).to(dev)
            ds = torch.from_numpy(np.concatenate(ds).astype(np.int64)).to(dev)
            keep2 = torch.ones(d.num_blocks, d.block_size, dtype=torch.bool, device=dev)
            keep2[db, ds] = False
    for t in range(wl.n_tensors):
        sr = rows_dev(src[t], g)
        st_t = stage[t * per:(t + 1) * per].view(N, g.n_planes, g.block_size, sl)
        assert torch.equal(sr[src_ids][..., s_off:s_off + sl], st_t), f"tensor {t}: staging != layer[block_ids]"
        base = rows_dev(regen(g, seed, t, dev), g)
        if case.n_tokens:
            for p in range(g.n_planes):
                nr = new[t * g.n_planes + p].reshape(case.n_tokens, -1).view(torch.uint8)
                assert torch.equal(sr[blk, p, off], nr), f"tensor {t} plane {p}: new rows not at their slots"
                assert torch.equal(sr[:, p][written], base[:, p][written]), f"tensor {t}: untouched slots changed"
        else:
            assert torch.equal(sr, base), f"tensor {t}: source changed without new tokens"
        del base
        if has_dst:
            dr = rows_dev(dst[t], d)
            dbase = rows_dev(regen(d, seed + 1, t, dev), d)
            o = wl.dst_slice_off
            if equal:
                assert torch.equal(dr[dst_ids][..., o:o + sl], st_t), f"tensor {t}: dst blocks != staged blocks"
                assert torch.equal(dr[keep], dbase[keep]), f"tensor {t}: unlisted dst blocks changed"
            else:
                toks = st_t.reshape(N * g.block_size, sl)  # one plane: staged tokens in order
                assert torch.equal(dr[db, 0, ds, o:o + sl], toks), f"tensor {t}: remapped tokens misplaced"
                assert torch.equal(dr[:, 0][keep2], dbase[:, 0][keep2]), f"tensor {t}: untouched dst slots changed"
            del dbase

    # --- kv_write_tokens at full size: fresh rows through the fused call -----
    if case.n_tokens:
        del new
        new2 = W.new_token_rows(g, wl.n_tensors, case.n_tokens, dev, seed=seed + 3)
        out = torch.full((case.n_tokens,), -7, dtype=torch.int64, device=dev)
        K.kv_write_tokens(step.src, new2, step.block_table, step.token_req, step.token_pos, out)
        torch.cuda.synchronize()
        assert K.kv_get_last_error(clear=True) == 0
        np.testing.assert_array_equal(out.cpu().numpy(), slot)
        for t in range(wl.n_tensors):
            sr = rows_dev(src[t], g)
            for p in range(g.n_planes):
                nr = new2[t * g.n_planes + p].reshape(case.n_tokens, -1).view(torch.uint8)
                assert torch.equal(sr[blk, p, off], nr), f"tensor {t} plane {p}: kv_write_tokens rows not at their slots"
        del new2
    else:
        del new
    del step, src, dst, stage
    torch.cuda.empty_cache()
