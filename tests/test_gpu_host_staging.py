"""Pack into, and unpack from, a staging buffer in pinned host memory.

The NCCL page's receiver spills a received tensor to pinned host memory when its
device buffer is past a threshold ("0. vllm 如何使用 nccl 传输 kv cache", section 2.3).
Here the copy kernels write the staging buffer straight into pinned host memory over
the host link, and read it back from there; results must equal the oracle's bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep
from tests import gpu_support as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()


@pytest.mark.parametrize("wl", [W.TINY, W.small(W.PAGE), W.small(W.MID), W.small(W.ASYM)], ids=lambda w: w.name)
def test_host_staging_parity(wl):
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 77)
    s_dev = W.to_device_bf16(src, "cuda")
    d_dev = W.to_device_bf16(dst, "cuda")
    n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, s_dev, d_dev, n_dev, host_stage=True)
    assert not step.stage.is_cuda and step.stage.is_pinned()
    step.run()
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) == 0
    gpu = dict(err=0, slot=step.slot.cpu().numpy() if case.n_tokens else None, runs=step.xfer.host(),
               stage=step.stage[:G._stage_len(wl, case)].numpy().copy(),
               src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
               dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev])
    ora = G.run_oracle(wl, case, src, dst, new, step.max_run_blocks)
    G.compare(gpu, ora, wl.name + " host staging")


def test_unregistered_host_staging_rejected():
    g = W.CacheGeom("separate", 8, 4, 1, 64)
    cache = K.PagedCache.from_tensors(W.device_cache(g, 1, "cuda", seed=3), "separate")
    off = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    ids = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    x = K.kv_build_xfer_list(off, ids)
    pageable = torch.empty(2 * 4 * 128, dtype=torch.uint8)  # not pinned
    lib = K.load()
    d = cache.desc()
    sd = K.stage_desc(2, 1, 1, 4, 128)
    import ctypes
    st = lib.kv_pack_blocks(ctypes.byref(d), 0, ctypes.byref(sd), K._ptr(x.runs), K._ptr(x.n_runs), x.capacity, 0,
                            ctypes.c_void_p(pageable.data_ptr()), pageable.numel(), K._stream())
    assert st == K.KV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
