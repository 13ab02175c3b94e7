"""kv_block_hashes (prefix hash chain over full token blocks) against the oracle, bit-exact.

Drawing "vllm v1 调度逻辑 和 distributed 分布式原理", hash-table labels: h0 = hash(seed, [t0..t1]),
h_i = hash(h_(i-1), ...).  The hash is read as FNV-1a 64 (the oracle's pins fix it).  Both
device paths are compared: the table split with a workspace and the plain byte chain without.
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


PATHS = ["table", "chain"]


def _gpu(off, toks, bs, seed, path="table"):
    o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(toks).cuda(), bs, seed,
                             workspace="auto" if path == "table" else None)
    o = o.cpu().numpy()
    return o, h[:o[-1]].cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bs", [1, 2, 3, 16, 64, 600])
def test_hashes_match_oracle(bs, path):
    rng = np.random.default_rng(bs)
    lens = rng.integers(0, 40 * bs if bs < 100 else 5 * bs, size=300 if bs < 100 else 24)
    lens[[3, 17]] = 0
    toks = [rng.integers(0, 128000, size=n).astype(np.int32) for n in lens]
    toks[5] = toks[4][: len(toks[5])].copy() if len(toks[5]) <= len(toks[4]) else toks[5]  # a shared prefix
    off, flat = W.csr(toks)
    for seed in (0, 0xDEADBEEFCAFEF00D):
        want_o, want = oracle.block_hashes(off, flat, bs, seed)
        got_o, got = _gpu(off, flat, bs, seed, path)
        np.testing.assert_array_equal(got_o, want_o)
        np.testing.assert_array_equal(got, want)
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("path", PATHS)
def test_page_shaped_prompts(path):
    """8 prompts of 9216 tokens, block size 16: 576 hashes each."""
    rng = np.random.default_rng(83)
    toks = [rng.integers(0, 128000, size=9216).astype(np.int32) for _ in range(8)]
    off, flat = W.csr(toks)
    want_o, want = oracle.block_hashes(off, flat, 16, 81)
    got_o, got = _gpu(off, flat, 16, 81, path)
    assert got_o[-1] == 8 * 576
    np.testing.assert_array_equal(got, want)


def test_extreme_token_values_and_reused_workspace():
    """Token ids with every byte value (negative ids too), and one workspace reused by calls in turn."""
    rng = np.random.default_rng(84)
    toks = [rng.integers(-2**31, 2**31, size=int(n), dtype=np.int64).astype(np.int32) for n in (64, 200, 33, 1000)]
    toks[1][:16] = [-1, 0, 1, 2**31 - 1, -2**31, 255, 256, -256, 0x01020304, 0x7f7f7f7f, -0x7f7f7f80, 65535, 65536,
                    -65536, 0xff00ff, -0xff0100]
    off, flat = W.csr(toks)
    ws = torch.empty(K.kv_block_hashes_workspace_bytes(flat.shape[0], 8), dtype=torch.uint8, device="cuda")
    for seed in (3, 2**64 - 1):
        o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(flat).cuda(), 8, seed, workspace=ws)
        want_o, want = oracle.block_hashes(off, flat, 8, seed)
        np.testing.assert_array_equal(h[:int(want_o[-1])].cpu().numpy().view(np.uint64), want)
    assert K.kv_get_last_error() == 0


def test_workspace_checked():
    off = torch.tensor([0, 32], dtype=torch.int32, device="cuda")
    toks = torch.arange(32, dtype=torch.int32, device="cuda")
    need = K.kv_block_hashes_workspace_bytes(32, 4)
    assert need == 8 * 256 * 8
    with pytest.raises(RuntimeError):
        K.kv_block_hashes(off, toks, 4, 1, workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(RuntimeError):  # not 16-byte aligned
        K.kv_block_hashes(off, toks, 4, 1, workspace=torch.empty(need + 16, dtype=torch.uint8, device="cuda")[8:])


@pytest.mark.parametrize("path", PATHS)
def test_inconsistent_offsets_flagged(path):
    off = torch.tensor([0, 40, 20, 60], dtype=torch.int32, device="cuda")
    toks = torch.arange(60, dtype=torch.int32, device="cuda")
    o, h = K.kv_block_hashes(off, toks, 4, 1, workspace="auto" if path == "table" else None)
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) & K.KV_DERR_LIST
    assert h.shape[0] == 15  # capacity; the kernel bounds every write
