"""Running one workload through the CUDA path and through the oracle, on identical inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep
from tests import helpers as H


def has_dst(wl: W.Workload) -> bool:
    return wl.kind != "mla"  # the MLA preset packs only


def host_inputs(wl: W.Workload, case: W.Case, seed: int):
    """Seeded host inputs: src cache, dst cache (or None), new token rows per (tensor, plane)."""
    rng = np.random.default_rng(seed)
    src = W.host_cache_tensors(wl.src, wl.n_tensors, rng)
    dst = W.host_cache_tensors(wl.dst, wl.n_tensors, rng) if has_dst(wl) else None
    g = wl.src
    new = [W.normal_bf16_bytes(rng, case.n_tokens * g.row_bytes // 2).reshape(case.n_tokens, g.row_bytes // 2)
           for _ in range(wl.n_tensors * g.n_planes)]
    return src, dst, new


def _new_shape(g: W.CacheGeom, T: int):
    return (T, 1, g.heads * g.head_dim) if g.layout == "mla" else (T, g.heads, g.head_dim)


def run_gpu(wl, case, src, dst, new, max_run_blocks=None, device="cuda", host_stage=False):
    s_dev = W.to_device_bf16(src, device)
    d_dev = W.to_device_bf16(dst, device) if dst is not None else None
    n_dev = [x.reshape(_new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, device)]
    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, s_dev, d_dev, n_dev, max_run_blocks=max_run_blocks, device=device,
                        host_stage=host_stage)
    step.run()
    torch.cuda.synchronize()
    out = dict(
        err=K.kv_get_last_error(clear=True),
        slot=step.slot.cpu().numpy() if case.n_tokens else None,
        runs=step.xfer.host(),
        stage=step.stage[:_stage_len(wl, case)].cpu().numpy(),
        src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
        dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev] if d_dev is not None else None,
        max_run_blocks=step.max_run_blocks,
    )
    return out


def _stage_len(wl, case):
    return wl.n_tensors * case.n_blocks * wl.src.n_planes * wl.src.block_size * wl.moved_slice


def run_oracle(wl, case, src, dst, new, max_run_blocks):
    src = [a.copy() for a in src]
    dst = [a.copy() for a in dst] if dst is not None else None
    out = dict(slot=None)
    sc = H.ora_cache(wl.src, src)
    if case.n_tokens:
        slot, bad = oracle.slot_mapping(case.block_table, case.token_req, case.token_pos, wl.src.block_size)
        assert bad == 0
        rows = [r.view(np.uint8) for r in new]
        assert oracle.reshape_and_cache(sc, rows, slot) == 0
        out["slot"] = slot
    equal = wl.equal_geometry and dst is not None
    out["runs"] = oracle.build_xfer_list(case.req_offsets, case.src_ids, case.dst_ids if equal else None,
                                         max_run_blocks)
    out["stage"] = oracle.pack(sc, case.req_offsets, case.src_ids, wl.slice_off, wl.moved_slice)
    out["src"] = sc.tensors
    if dst is not None:
        dc = H.ora_cache(wl.dst, dst)
        st = oracle.unpack(dc, out["stage"], case.req_offsets, case.dst_req_offsets, case.dst_ids,
                           wl.src.block_size, wl.moved_slice, wl.dst_slice_off)
        assert st == 0
        out["dst"] = dc.tensors
    else:
        out["dst"] = None
    return out


def compare(gpu: dict, ora: dict, what: str = ""):
    """Bit-exact comparison of every output; raises AssertionError naming the first difference."""
    assert gpu["err"] == 0, f"{what}: device error word {gpu['err']:#x}"
    if ora["slot"] is not None:
        np.testing.assert_array_equal(gpu["slot"], ora["slot"], err_msg=f"{what}: slot")
    g, o = gpu["runs"], ora["runs"]
    assert g["count"] == o["req"].shape[0], f"{what}: run count {g['count']} vs {o['req'].shape[0]}"
    for key in ("req", "src_block", "dst_block", "n_blocks", "stage_block"):
        np.testing.assert_array_equal(g[key], o[key], err_msg=f"{what}: runs.{key}")
    assert gpu["stage"].shape == ora["stage"].shape
    diff = np.flatnonzero(gpu["stage"] != ora["stage"])
    assert diff.size == 0, f"{what}: staging differs at {diff.size} bytes, first at {diff[:4]}"
    for t, (a, b) in enumerate(zip(gpu["src"], ora["src"])):
        assert np.array_equal(a, b), f"{what}: src tensor {t} after reshape_and_cache"
    if ora["dst"] is not None:
        for t, (a, b) in enumerate(zip(gpu["dst"], ora["dst"])):
            assert np.array_equal(a, b), f"{what}: dst tensor {t} after unpack"
