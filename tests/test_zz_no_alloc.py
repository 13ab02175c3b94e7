"""kv_build_xfer_list_static: the transfer-list builder for callers that cannot allocate.

Some callers cannot allocate device memory when they build a transfer list: a
transport's progress thread (cudaMalloc / cudaFree may synchronise the device and
stall the model's stream) or a serving process whose KV-cache pool already took
nearly all free device memory.  This entry point keeps its scratch in a fixed array
inside the library.  The test calls it through the C ABI four times in a row, on
different lists, and checks each result bit-exactly against kv_build_xfer_list
(the workspace variant) on the same input.  It also checks the size limit.

The file name sorts last so that a run stopping at the first failure has already run
every other test; it needs nothing from the other tests and runs alone too.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W

pytestmark = pytest.mark.gpu


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
    return h["count"], [h[k] for k in ("req", "src_block", "dst_block", "n_blocks", "stage_block")]


def test_static_builder_matches_workspace_builder_twice():
    # different lists; those longer than 5120 entries take the look-back builder, which uses the scratch
    cases = [(_lists(1, 9000, 17), 2), (_lists(2, 100000, 3), 0), (_lists(3, 3000, 4), 1), (_lists(4, 70001, 5), 7)]
    dev = [tuple(torch.from_numpy(a).cuda() for a in lists) + (cap,) for lists, cap in cases]
    want = [_host(K.kv_build_xfer_list(o, s, d, cap)) for o, s, d, cap in dev]
    # calls in a row on one stream: each look-back call reuses the scratch the one before left behind
    got = [K.kv_build_xfer_list_static(o, s, d, cap) for o, s, d, cap in dev]
    torch.cuda.synchronize()
    for (wc, wr), g in zip(want, got):
        gc, gr = _host(g)
        assert gc == wc
        for a, b in zip(gr, wr):
            np.testing.assert_array_equal(a, b)
    assert K.kv_get_last_error() == 0


def test_static_builder_rejects_oversized_list():
    lib = K.load()
    n = K.KV_XFER_STATIC_MAX_BLOCKS + 1
    # rejected before anything is queued, so placeholder pointers are never touched
    st = lib.kv_build_xfer_list_static(ctypes.c_void_p(16), 1, ctypes.c_void_p(32), None, n, 0,
                                       ctypes.c_void_p(64), n, ctypes.c_void_p(128), None)
    assert st == K.KV_ERR_RANGE
