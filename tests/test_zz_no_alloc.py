"""kv_build_xfer_list_static: the transfer-list builder for callers that cannot allocate.

Some callers cannot allocate device memory when they build a transfer list: a
transport's progress thread (cudaMalloc / cudaFree may synchronise the device and
stall the model's stream) or a serving process whose KV-cache pool already took
nearly all free device memory.  This entry point keeps its scratch in a fixed array
inside the library.  The test calls it through the C ABI on four different lists,
twice in a row, and checks every result bit-exactly against the oracle's run walk
and against kv_build_xfer_list (the workspace variant) on the same input.  Between
the two rounds it reads the device's free memory and the caching allocator's
reserved bytes: the second round (after the first round's per-device set-up) must
leave both unchanged.  It also checks the size limit.

The file name sorts last so that a run stopping at the first failure has already run
every other test; it needs nothing from the other tests and runs alone too.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FIELDS = ("req", "src_block", "dst_block", "n_blocks", "stage_block")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()


def _lists(seed, n, max_piece):
    rng = np.random.default_rng(seed)
    lens, left = [], n
    while left > 0:
        k = int(min(left, rng.integers(0, 2500)))
        lens.append(k)
        left -= k
    q = W.fragmented_queue(rng, n + 11, max_piece, 0.7)
    off, ids = W.csr(W.pop_lists(q, lens))
    dids = W.fragmented_queue(rng, n + 5, 9, 0.8)[:n].astype(np.int32)
    return off, ids, dids


def _host(x: K.XferList):
    h = x.host()
    return h["count"], [h[k] for k in FIELDS]


def _assert_same(got, want, what):
    gc, gr = got
    wc, wr = want
    assert gc == wc, f"{what}: {gc} runs, expected {wc}"
    for name, a, b in zip(FIELDS, gr, wr):
        np.testing.assert_array_equal(a, b, err_msg=f"{what}: runs.{name}")


def test_static_builder_matches_oracle_and_allocates_nothing():
    # different lists; those longer than 5120 entries take the look-back builder, which uses the
    # library's scratch array; the 3000-entry list takes the single-CTA kernel
    cases = [(_lists(1, 9000, 17), 2), (_lists(2, 100000, 3), 0), (_lists(3, 3000, 4), 1), (_lists(4, 70001, 5), 7)]
    oracle_runs = []
    for (off, ids, dids), cap in cases:
        r = oracle.build_xfer_list(off, ids, dids, cap)
        oracle_runs.append((int(r["req"].shape[0]), [r[k] for k in FIELDS]))
    dev = [tuple(torch.from_numpy(a).cuda() for a in lists) + (cap,) for lists, cap in cases]
    workspace_runs = [_host(K.kv_build_xfer_list(o, s, d, cap)) for o, s, d, cap in dev]
    # every output list of both rounds exists before the first reading of device memory
    outs = [[K.XferList(s.shape[0], s.device, cap) for o, s, d, cap in dev] for _ in range(2)]
    torch.cuda.synchronize()

    def round_of_calls(k):
        # calls in a row on one stream: each look-back call reuses the scratch the one before left behind
        for (o, s, d, cap), out in zip(dev, outs[k]):
            K.kv_build_xfer_list_static(o, s, d, cap, out=out)
        torch.cuda.synchronize()

    round_of_calls(0)  # the first call on this device looks up the scratch array's address
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    round_of_calls(1)
    free1, reserved1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    assert free1 == free0, f"device free memory changed by {free1 - free0} bytes across the calls"
    assert reserved1 == reserved0, "the caching allocator reserved memory during the calls"
    for k in range(2):
        for i, out in enumerate(outs[k]):
            got = _host(out)
            _assert_same(got, oracle_runs[i], f"round {k}, list {i}: vs the oracle")
            _assert_same(got, workspace_runs[i], f"round {k}, list {i}: vs kv_build_xfer_list")
    assert K.kv_get_last_error() == 0


def test_static_builder_rejects_oversized_list():
    lib = K.load()
    n = K.KV_XFER_STATIC_MAX_BLOCKS + 1
    # rejected before anything is queued, so placeholder pointers are never touched
    st = lib.kv_build_xfer_list_static(ctypes.c_void_p(16), 1, ctypes.c_void_p(32), None, n, 0,
                                       ctypes.c_void_p(64), n, ctypes.c_void_p(128), None)
    assert st == K.KV_ERR_RANGE
