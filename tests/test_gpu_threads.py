"""Two host threads driving the library at once, each on its own stream and caches.

The library keeps per-device state on the host (device info, occupancy and launch attributes,
the static builder scratch's address), set up on first use under a lock.  Here two threads
make their first calls at the same moment, then run whole steps concurrently, and each
thread's results are compared with the oracle bit-exactly.
"""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from paged_kv_cache_81_gb300.step import TransferStep
from tests import gpu_support as G

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_two_threads_run_steps_concurrently():
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()
    workloads = [W.small(W.PAGE), W.small(W.ASYM)]
    cases = [W.make_case(wl) for wl in workloads]
    inputs = [G.host_inputs(wl, case, seed=700 + i) for i, (wl, case) in enumerate(zip(workloads, cases))]
    results, errors = [None, None], []
    start = threading.Barrier(2)

    def worker(i):
        try:
            wl, case = workloads[i], cases[i]
            src, dst, new = inputs[i]
            s_dev = W.to_device_bf16(src, "cuda")
            d_dev = W.to_device_bf16(dst, "cuda")
            n_dev = [x.reshape(G._new_shape(wl.src, case.n_tokens)) for x in W.to_device_bf16(new, "cuda")]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                step = TransferStep(wl, case, s_dev, d_dev, n_dev)
                start.wait()  # both threads make their first library calls together
                for _ in range(3):  # the same step again: it rewrites the same bytes
                    step.run(stream)
            stream.synchronize()
            results[i] = dict(slot=step.slot.cpu().numpy() if case.n_tokens else None, runs=step.xfer.host(),
                              stage=step.stage[:G._stage_len(wl, case)].cpu().numpy(),
                              src=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in s_dev],
                              dst=[x.cpu().view(torch.int16).numpy().view(np.uint16) for x in d_dev],
                              max_run_blocks=step.max_run_blocks, err=0)
        except BaseException as e:  # reported below
            errors.append(e)
            start.abort()

    K.kv_get_last_error(clear=True)
    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=300)
    assert not errors, errors[0]
    assert K.kv_get_last_error() == 0
    for i, (wl, case) in enumerate(zip(workloads, cases)):
        src, dst, new = inputs[i]
        ora = G.run_oracle(wl, case, src, dst, new, results[i]["max_run_blocks"])
        G.compare(results[i], ora, f"thread {i} ({wl.name})")
