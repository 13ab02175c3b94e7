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


# "table": the full workspace (tables and walk in one cooperative launch when the walk is the
# longer part, else a table kernel first); "two": a workspace of the tables alone (always a table
# kernel, then the walk); "chain": no workspace (the plain byte chain).
PATHS = ["table", "two", "chain"]


def _workspace(path, n_tokens, bs):
    if path == "chain":
        return None
    if path == "table":
        return "auto"
    return torch.empty(max(16, (n_tokens // bs) * 2048), dtype=torch.uint8, device="cuda")


def _gpu(off, toks, bs, seed, path="table"):
    o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(toks).cuda(), bs, seed,
                             workspace=_workspace(path, toks.shape[0], bs))
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
    assert need == 8 * (256 * 8 + 4)  # 16416: tables and flags, a multiple of 16
    want_o, want = oracle.block_hashes(np.array([0, 32], np.int32), np.arange(32, dtype=np.int32), 4, 1)
    for size in (need, 8 * 2048):  # the full size, and the tables alone
        o, h = K.kv_block_hashes(off, toks, 4, 1, workspace=torch.empty(size, dtype=torch.uint8, device="cuda"))
        np.testing.assert_array_equal(h.cpu().numpy().view(np.uint64), want)
    with pytest.raises(RuntimeError):  # smaller than the tables
        K.kv_block_hashes(off, toks, 4, 1, workspace=torch.empty(8 * 2048 - 16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(RuntimeError):  # not 16-byte aligned
        K.kv_block_hashes(off, toks, 4, 1, workspace=torch.empty(need + 16, dtype=torch.uint8, device="cuda")[8:])
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("bs", [1, 3, 16, 64, 600])
@pytest.mark.parametrize("n_reqs", [1, 2, 5, 8, 30])
def test_few_long_requests_every_path(bs, n_reqs):
    """Few requests of many blocks, the case the cooperative launch serves (here: every case with
    one or two requests, up to 8 requests of blocks up to 64 tokens, 30 requests of blocks up to
    3 tokens; the others run the table kernel first), lengths with partial last blocks, an empty
    request and a shared prefix; every path against the oracle, twice on one reused workspace."""
    rng = np.random.default_rng(1000 * bs + n_reqs)
    lens = rng.integers(0, 120 * bs if bs < 100 else 12 * bs, size=n_reqs)
    if n_reqs > 2:
        lens[1] = 0
    toks = [rng.integers(-2 ** 31, 2 ** 31, size=int(n), dtype=np.int64).astype(np.int32) for n in lens]
    if n_reqs > 4 and len(toks[3]) <= len(toks[4]):
        toks[3] = toks[4][: len(toks[3])].copy()
    off, flat = W.csr(toks)
    want_o, want = oracle.block_hashes(off, flat, bs, 7)
    ws = torch.empty(max(16, K.kv_block_hashes_workspace_bytes(flat.shape[0], bs)), dtype=torch.uint8, device="cuda")
    for path in PATHS:
        for _ in range(2):
            o, h = K.kv_block_hashes(torch.from_numpy(off).cuda(), torch.from_numpy(flat).cuda(), bs, 7,
                                     workspace=ws if path == "table" else _workspace(path, flat.shape[0], bs))
            np.testing.assert_array_equal(o.cpu().numpy(), want_o)
            np.testing.assert_array_equal(h[: int(want_o[-1])].cpu().numpy().view(np.uint64), want, err_msg=path)
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("path", PATHS)
def test_inconsistent_offsets_flagged(path):
    off = torch.tensor([0, 40, 20, 60], dtype=torch.int32, device="cuda")
    toks = torch.arange(60, dtype=torch.int32, device="cuda")
    o, h = K.kv_block_hashes(off, toks, 4, 1, workspace=_workspace(path, 60, 4))
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) & K.KV_DERR_LIST
    assert h.shape[0] == 15  # capacity; the kernel bounds every write


@pytest.mark.parametrize("path", ["table", "two"])
def test_hashes_replayed_from_a_cuda_graph(path):
    """Both workspace paths captured in a CUDA graph (with the full workspace this batch of four
    requests takes the cooperative launch: a memset of the flags, then the fused kernel) and
    replayed after new token values are written in place, each replay against the oracle."""
    rng = np.random.default_rng(99)
    bs, lens = 8, [600, 1000, 37, 800]  # 75, 125, 4 and 100 full blocks
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(off[-1])
    off_d = torch.from_numpy(off).cuda()
    toks_d = torch.empty(n, dtype=torch.int32, device="cuda")
    out_o = torch.empty_like(off_d)
    out_h = torch.empty(n // bs, dtype=torch.int64, device="cuda")
    ws = _workspace(path, n, bs)
    if ws == "auto":
        ws = torch.empty(K.kv_block_hashes_workspace_bytes(n, bs), dtype=torch.uint8, device="cuda")
    toks_d.copy_(torch.from_numpy(rng.integers(-2 ** 31, 2 ** 31, size=n, dtype=np.int64).astype(np.int32)))
    K.kv_block_hashes(off_d, toks_d, bs, 5, out_o, out_h, workspace=ws)  # eager first: per-device set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        K.kv_block_hashes(off_d, toks_d, bs, 5, out_o, out_h, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(3):
        flat = rng.integers(-2 ** 31, 2 ** 31, size=n, dtype=np.int64).astype(np.int32)
        toks_d.copy_(torch.from_numpy(flat))
        g.replay()
        torch.cuda.synchronize()
        want_o, want = oracle.block_hashes(off, flat, bs, 5)
        np.testing.assert_array_equal(out_o.cpu().numpy(), want_o)
        np.testing.assert_array_equal(out_h[: int(want_o[-1])].cpu().numpy().view(np.uint64), want,
                                      err_msg=f"{path} replay {rep}")
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("path", ["table", "two"])
@pytest.mark.parametrize("n_reqs", [2000, 5000])
def test_many_requests(n_reqs, path):
    """More requests than a table CTA keeps offsets for (1024: the slot search reads them from
    global memory), and more than the table kernel's CTA 0 scans (4096: a separate count launch
    first); lengths from 0 to 70 tokens at block size 4, shared prefixes among them."""
    rng = np.random.default_rng(n_reqs)
    lens = rng.integers(0, 71, size=n_reqs)
    toks = [rng.integers(-2 ** 31, 2 ** 31, size=int(n), dtype=np.int64).astype(np.int32) for n in lens]
    for i in range(1, n_reqs, 7):  # every seventh request shares the previous one's prefix
        m = min(len(toks[i]), len(toks[i - 1]))
        toks[i][:m] = toks[i - 1][:m]
    off, flat = W.csr(toks)
    want_o, want = oracle.block_hashes(off, flat, 4, 123)
    got_o, got = _gpu(off, flat, 4, 123, path)
    np.testing.assert_array_equal(got_o, want_o)
    np.testing.assert_array_equal(got, want)
    assert K.kv_get_last_error() == 0
