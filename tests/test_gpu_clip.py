"""kv_clip_block_lists (sliding-window clip) against the oracle, and a clipped step.

Page "vLLM PD 分离 源码级机制", section 3.1: the sender ships get_sw_clipped_blocks(block_ids).
Reading (stated in the oracle): keep the entries that hold the last `window` tokens.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep
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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _gpu_clip(off, ids, n_tok, window, bs):
    o, out = K.kv_clip_block_lists(_dev(off), _dev(ids), _dev(n_tok), window, bs)
    o = o.cpu().numpy()
    return o, out.cpu().numpy()[:o[-1]]


def test_clip_golden():
    for c in H.read_clip_golden():
        off, ids = W.csr([c["ids"]])
        o, got = _gpu_clip(off, ids, [c["n"]], c["window"], c["bs"])
        assert got.tolist() == c["want"], c
    assert K.kv_get_last_error() == 0


@pytest.mark.parametrize("seed", range(6))
def test_clip_random_against_oracle(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 3000))
    bs = int(rng.choice([1, 16, 64]))
    lens = rng.integers(0, 80, size=R)
    lens[rng.integers(0, R)] = 0
    off, ids = W.csr(W.pop_lists(rng.permutation(int(lens.sum()) + 5).astype(np.int32), lens))
    n_tok = np.array([int(rng.integers(0, l * bs + 3 * bs + 1)) for l in lens], np.int32)  # some beyond the list
    for window in (0, 1, 37, 4096):
        want_o, want = oracle.clip_block_lists(off, ids, n_tok, window, bs)
        got_o, got = _gpu_clip(off, ids, n_tok, window, bs)
        np.testing.assert_array_equal(got_o, want_o)
        np.testing.assert_array_equal(got, want)
    assert K.kv_get_last_error() == 0


def test_clip_inconsistent_offsets_flagged_and_contained():
    off = _dev([0, 10, 5, 15])  # decreasing: lengths 10, -5, 10 over 15 entries
    ids = _dev(np.arange(15))
    n_tok = _dev([1000, 1000, 1000])
    out_o, out = K.kv_clip_block_lists(off, ids, n_tok, 0, 1)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() & K.KV_DERR_LIST
    assert out.shape[0] == 15  # nothing was written past the capacity (the kernel checks every index)


@pytest.mark.parametrize("wl", [W.small(W.PAGE), W.small(W.MID)], ids=lambda w: w.name)
def test_clipped_step_against_oracle(wl):
    """slot_mapping -> reshape -> clip -> xfer_list -> pack -> unpack, with a sliding window."""
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 31)
    s_dev, d_dev = W.to_device_bf16(src, "cuda"), W.to_device_bf16(dst, "cuda")
    n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
    window = 1000
    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, s_dev, d_dev, n_dev, sw_window=window)
    step.run()
    torch.cuda.synchronize()
    assert K.kv_get_last_error(clear=True) == 0
    # the oracle: the same step on the clipped lists
    c_off, c_ids = oracle.clip_block_lists(case.req_offsets, case.src_ids, case.req_tokens, window,
                                           wl.src.block_size)
    _, c_dids = oracle.clip_block_lists(case.req_offsets, case.dst_ids, case.req_tokens, window, wl.src.block_size)
    assert step.n_listed == c_ids.shape[0] < case.n_blocks
    clipped = W.Case(wl, c_off, c_ids, c_off, c_dids, case.block_table, case.token_req, case.token_pos,
                     case.req_tokens)
    ora = G.run_oracle(wl, clipped, src, dst, new, step.max_run_blocks)
    gpu = dict(err=0, slot=step.slot.cpu().numpy() if case.n_tokens else None, runs=step.xfer.host(),
               stage=step.stage[:G._stage_len(wl, clipped)].cpu().numpy(),
               src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
               dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev])
    G.compare(gpu, ora, wl.name + " clipped")
