"""kv_block_hashes (prefix hash chain over full token blocks) against the oracle, bit-exact.

Drawing "vllm v1 调度逻辑 和 distributed 分布式原理", hash-table labels: h0 = hash(seed, [t0..t1]),
h_i = hash(h_(i-1), ...).  The hash is read as FNV-1a 64 (the oracle's pins fix it).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
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


def _gpu(off, toks, bs, seed):
    o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(toks).cuda(), bs, seed)
    o = o.cpu().numpy()
    return o, h[:o[-1]].cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("bs", [1, 2, 16, 64])
def test_hashes_match_oracle(bs):
    rng = np.random.default_rng(bs)
    lens = rng.integers(0, 40 * bs, size=300)
    lens[[3, 17]] = 0
    toks = [rng.integers(0, 128000, size=n).astype(np.int32) for n in lens]
    toks[5] = toks[4][: len(toks[5])].copy() if len(toks[5]) <= len(toks[4]) else toks[5]  # a shared prefix
    off, flat = W.csr(toks)
    for seed in (0, 0xDEADBEEFCAFEF00D):
        want_o, want = oracle.block_hashes(off, flat, bs, seed)
        got_o, got = _gpu(off, flat, bs, seed)
        np.testing.assert_array_equal(got_o, want_o)
        np.testing.assert_array_equal(got, want)
    assert K.kv_get_last_error() == 0


def test_page_shaped_prompts():
    """8 prompts of 9216 tokens, block size 16: 576 hashes each."""
    rng = np.random.default_rng(83)
    toks = [rng.integers(0, 128000, size=9216).astype(np.int32) for _ in range(8)]
    off, flat = W.csr(toks)
    want_o, want = oracle.block_hashes(off, flat, 16, 81)
    got_o, got = _gpu(off, flat, 16, 81)
    assert got_o[-1] == 8 * 576
    np.testing.assert_array_equal(got, want)


def test_inconsistent_offsets_flagged():
    off = torch.tensor([0, 40, 20, 60], dtype=torch.int32, device="cuda")
    toks = torch.arange(60, dtype=torch.int32, device="cuda")
    o, h = K.kv_block_hashes(off, toks, 4, 1)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_LIST
    assert h.shape[0] == 15  # capacity; the kernel bounds every write
