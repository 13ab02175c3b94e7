"""A whole step captured in a CUDA graph and replayed gives the oracle's results.

Every entry point of the path is asynchronous and allocation-free, so after one eager step
(which does the per-device setup) the five calls capture into one graph; replaying it is how
a launch-bound step, such as a decode step's cache write, is issued without per-call host cost.
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


@pytest.mark.parametrize("wl", [W.TINY, W.small(W.MLA), W.small(W.MID), W.small(W.ASYM)], ids=lambda w: w.name)
def test_graph_replay_matches_oracle(wl):
    case = W.make_case(wl)
    src, dst, new = G.host_inputs(wl, case, seed=wl.seed + 404)
    s_dev = W.to_device_bf16(src, "cuda")
    d_dev = W.to_device_bf16(dst, "cuda") if dst is not None else None
    n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
    s_before = [x.clone() for x in s_dev]
    d_before = [x.clone() for x in d_dev] if d_dev is not None else None
    K.kv_get_last_error(clear=True)
    step = TransferStep(wl, case, s_dev, d_dev, n_dev)
    step.run()  # eager first call: per-device setup happens here, outside the capture
    torch.cuda.synchronize()
    graph = step.capture()
    for _ in range(2):  # restore the inputs, replay, compare: the replay redoes the whole step
        for x, b in zip(s_dev, s_before):
            x.copy_(b)
        if d_dev is not None:
            for x, b in zip(d_dev, d_before):
                x.copy_(b)
        step.stage.zero_()
        step.xfer.runs.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert K.kv_get_last_error(clear=True) == 0
        gpu = dict(err=0, slot=step.slot.cpu().numpy() if case.n_tokens else None, runs=step.xfer.host(),
                   stage=step.stage[:G._stage_len(wl, case)].cpu().numpy(),
                   src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
                   dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev] if d_dev else None)
        G.compare(gpu, G.run_oracle(wl, case, src, dst, new, step.max_run_blocks), wl.name + " graph replay")
