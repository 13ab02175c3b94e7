"""Completion signals: unpack posts a counter increment once its rows have landed; a
bounded device-side wait releases the stream when the counter reaches the expected value.

Protocol of the FlagCX connector ("5. flagcx connector design & dev & test", section 1.2):
the sender adds 1 with the last put of each transfer; the receiver waits for the largest
expected value.  Every wait here either follows the signalling call on the same stream
or waits on a counter nothing sets and must time out, reporting KV_ERR_TIMEOUT.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

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


def _signalled_unpack(step: TransferStep, signal, add):
    wl = step.wl
    if step.equal:
        K.kv_unpack_blocks(step.dst, step.stage, step.xfer, step.case.n_blocks, wl.src.block_size, step.slice_bytes,
                           wl.dst_slice_off, signal=signal, signal_add=add)
    else:
        K.kv_unpack_blocks(step.dst, step.stage, step.xfer, step.case.n_blocks, wl.src.block_size, step.slice_bytes,
                           wl.dst_slice_off, step.req_offsets, step.dst_req_offsets, step.dst_ids, signal=signal,
                           signal_add=add)


# small page and small mid: TMA bulk engine (8 and 32 KiB blocks); small asym: token remap (warp engine)
@pytest.mark.parametrize("wl", [W.small(W.PAGE), W.small(W.MID), W.small(W.ASYM)], ids=lambda w: w.name)
def test_unpack_signal_then_wait(wl):
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 55)
    s_dev, d_dev = W.to_device_bf16(src, "cuda"), W.to_device_bf16(dst, "cuda")
    n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, s_dev, d_dev, n_dev)
    step.write_tokens()
    step.build()
    step.pack()
    sig = K.new_signal()
    _signalled_unpack(step, sig, 1)
    status = K.kv_wait_signal(sig, 1, 1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == K.KV_OK
    assert K.signal_value(sig) == 1 and int(sig[1].item()) == 0  # arrival count reset for reuse
    # two more transfers: the waiter asks for the largest expected value
    _signalled_unpack(step, sig, 1)
    _signalled_unpack(step, sig, 2)
    status = K.kv_wait_signal(sig, 4, 1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == K.KV_OK and K.signal_value(sig) == 4
    assert K.kv_get_last_error(clear=True) == 0
    # the scatter itself is still exact (unpacking the same staging again is idempotent)
    gpu = dict(err=0, slot=step.slot.cpu().numpy() if case.n_tokens else None, runs=step.xfer.host(),
               stage=step.stage[:G._stage_len(wl, case)].cpu().numpy(),
               src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
               dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev])
    G.compare(gpu, G.run_oracle(wl, case, src, dst, new, step.max_run_blocks), wl.name + " signalled")


def test_wait_times_out_on_a_counter_nothing_sets():
    K.kv_get_last_error(clear=True)
    sig = K.new_signal()
    status = K.kv_wait_signal(sig, 1, 20_000)  # 20 ms
    torch.cuda.synchronize()
    assert int(status.item()) == K.KV_ERR_TIMEOUT
    assert K.kv_get_last_error(clear=True) & K.KV_DERR_TIMEOUT
    # the context is still usable: a satisfied wait right after succeeds
    sig[0] = 3
    status = K.kv_wait_signal(sig, 3, 20_000)
    torch.cuda.synchronize()
    assert int(status.item()) == K.KV_OK and K.kv_get_last_error() == 0


def test_zero_work_unpack_still_signals():
    g = W.CacheGeom("separate", 8, 4, 1, 64)
    cache = K.PagedCache.from_tensors(W.device_cache(g, 1, "cuda", seed=5), "separate")
    off = torch.zeros(2, dtype=torch.int32, device="cuda")
    ids = torch.zeros(0, dtype=torch.int32, device="cuda")
    x = K.kv_build_xfer_list(off, ids)
    stage = torch.empty(16, dtype=torch.uint8, device="cuda")
    sig = K.new_signal()
    K.kv_unpack_blocks(cache, stage, x, 0, 4, signal=sig, signal_add=7)
    torch.cuda.synchronize()
    assert K.signal_value(sig) == 7


def test_wait_argument_checks():
    sig = K.new_signal()
    lib = K.load()
    import ctypes
    assert lib.kv_wait_signal(K._ptr(sig), 1, 0, None, K._stream()) == K.KV_ERR_RANGE
    assert lib.kv_wait_signal(K._ptr(sig), 1, 60_000_001, None, K._stream()) == K.KV_ERR_RANGE
    assert lib.kv_wait_signal(ctypes.c_void_p(sig.data_ptr() + 8), 1, 10, None, K._stream()) == K.KV_ERR_ALIGN
    assert lib.kv_wait_signal(None, 1, 10, None, K._stream()) == K.KV_ERR_INVALID_ARG


@pytest.mark.parametrize("row", [128, 256], ids=["2KiB_blocks_warp_engine", "4KiB_blocks_tma_engine"])
def test_wait_then_copy_leaves_room_for_the_producer(row):
    """Stream A waits for a counter that a signalled unpack on stream B sets, then packs: a
    persistent grid that fills every SM.  The pack must not be scheduled while the wait polls, or
    it would hold the SM space the unpack needs and the wait would run out.  B starts late (a
    sleep kernel), so A's wait is already polling when the unpack is queued.  The pack reads the
    blocks the unpack wrote, ordered by the counter, and must return the staged bytes."""
    n, bs = 40, 16
    g = W.CacheGeom("separate", 256, bs, 1, row // 2)  # 2 KiB blocks: the warp engine; 4 KiB: the TMA engine
    rng = np.random.default_rng(31)
    cache = K.PagedCache.from_tensors(W.device_cache(g, 2, "cuda", seed=31), "separate")
    ids = rng.permutation(256)[:n].astype(np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    off = t([0, n])
    x_in = K.kv_build_xfer_list(off, t(ids), t(ids), 0)  # runs carry the ids as destination blocks
    x_out = K.kv_build_xfer_list(off, t(ids), None, 0)
    stage_in = torch.from_numpy(rng.integers(0, 256, size=2 * n * bs * row, dtype=np.uint8)).cuda()
    stage_out = torch.zeros_like(stage_in)
    sig = K.new_signal()
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda._sleep(1000)  # the sleep kernel is this test's own producer-side kernel: load it before the poll
    torch.cuda.synchronize()
    K.kv_get_last_error(clear=True)
    with torch.cuda.stream(a):
        status = K.kv_wait_signal(sig, 1, 2_000_000)
        K.kv_pack_blocks(cache, x_out, n, stage_out)
    with torch.cuda.stream(b):
        torch.cuda._sleep(50_000_000)
        K.kv_unpack_blocks(cache, stage_in, x_in, n, bs, signal=sig, signal_add=1)
    torch.cuda.synchronize()
    assert int(status.item()) == K.KV_OK
    assert K.kv_get_last_error() == 0
    assert torch.equal(stage_out, stage_in)


_FRESH_PROCESS = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, ".")
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
K.load()
n, bs, row = 40, 16, 256
g = W.CacheGeom("separate", 256, bs, 1, row // 2)
rng = np.random.default_rng(32)
cache = K.PagedCache.from_tensors(W.device_cache(g, 2, "cuda", seed=32), "separate")
ids = rng.permutation(256)[:n].astype(np.int32)
t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
x = K.kv_build_xfer_list(t([0, n]), t(ids), t(ids), 0)
stage_in = torch.from_numpy(rng.integers(0, 256, size=2 * n * bs * row, dtype=np.uint8)).cuda()
sig = K.new_signal()
a, b = torch.cuda.Stream(), torch.cuda.Stream()
torch.cuda.synchronize()
with torch.cuda.stream(a):
    status = K.kv_wait_signal(sig, 1, 2_000_000)
with torch.cuda.stream(b):  # the unpack kernel's first use in this process
    K.kv_unpack_blocks(cache, stage_in, x, n, bs, signal=sig, signal_add=1)
torch.cuda.synchronize()
got = torch.stack([c.view(torch.uint8).reshape(256, -1)[torch.from_numpy(ids.astype(np.int64)).cuda()]
                   for c in cache.tensors]).reshape(-1)
print(json.dumps({"status": int(status.item()), "err": K.kv_get_last_error(),
                  "data_ok": bool(torch.equal(got, stage_in))}))
"""


def test_wait_does_not_hold_a_producer_kernel_loaded_after_it():
    """In a fresh process, queue a wait on stream A, then the first signalled unpack of the
    process on stream B.  The unpack's kernel must already be loaded: loading it while the wait
    polls may synchronise the context, which would hold the unpack until the wait runs out."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d == {"status": K.KV_OK, "err": 0, "data_ok": True}
