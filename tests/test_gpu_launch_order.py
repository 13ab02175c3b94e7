"""Stream order around the library's launches.

Every kernel of libpagedkv may be scheduled while the previous work on its stream still runs
(programmatic dependent launch); each waits for that work before touching memory.  These tests
interleave the library's calls with torch's own work on one stream, each iteration with fresh
data, so any read that moved ahead of the work before it would see stale bytes:
  torch copy kernel into the source cache -> kv_pack_blocks (must see the new bytes)
  -> torch copy of the staging buffer (must see the packed bytes)
  -> torch fill of the destination cache -> stage.zero_() (a memset)
  -> kv_unpack_blocks (must see the zeros, and land after the fill)
  -> torch copy kernel into the new-token rows -> kv_slot_mapping + kv_reshape_and_cache
  -> torch copy of the written cache.
The expected bytes are computed on the host with the oracle.  The same sequence also runs
replayed from a CUDA graph.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_81_gb300 import pagedkv as K
from paged_kv_cache_81_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

NB, BS, HEADS, HD = 64, 16, 2, 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_81_gb300 import build
    build.build()
    K.load()


class Case:
    """One separate-K/V cache pair of 2 tensors, a block list, new tokens, and the patterns."""

    def __init__(self, iters: int, seed: int):
        rng = np.random.default_rng(seed)
        self.g = W.CacheGeom("separate", NB, BS, HEADS, HD)
        self.src = [torch.zeros(self.g.tensor_shape(), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        self.dst = [torch.zeros(self.g.tensor_shape(), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        self.scache = K.PagedCache.from_tensors(self.src, "separate")
        self.dcache = K.PagedCache.from_tensors(self.dst, "separate")
        lists = [rng.permutation(NB)[:10], rng.permutation(NB)[:7]]
        lists[1] = np.setdiff1d(lists[1], lists[0])[:5]  # distinct blocks across requests
        self.off, self.ids = W.csr(lists)
        self.n = int(self.ids.shape[0])
        dids = rng.permutation(NB)[:self.n].astype(np.int32)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.x = K.kv_build_xfer_list(t(self.off), t(self.ids), t(dids), 4)
        self.stage = torch.empty(2 * self.n * BS * self.g.row_bytes, dtype=torch.uint8, device="cuda")
        # new tokens: 12 positions of request 0's blocks
        self.table = t(np.array([lists[0], np.pad(lists[1], (0, 10 - len(lists[1])), constant_values=-1)],
                                dtype=np.int32))
        self.T = 12
        self.req = t(np.zeros(self.T, dtype=np.int32))
        self.pos = t(rng.choice(10 * BS, size=self.T, replace=False).astype(np.int32))
        self.slot = torch.empty(self.T, dtype=torch.int64, device="cuda")
        self.rows = [torch.zeros((self.T, HEADS, HD), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        # per-iteration patterns, already on the device (copied in by torch kernels)
        self.pat_cache = [torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(2,) + self.g.tensor_shape(),
                                                        dtype=np.int16)).cuda().view(torch.bfloat16)
                          for _ in range(iters)]
        self.pat_rows = [torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(2, self.T, HEADS, HD),
                                                       dtype=np.int16)).cuda().view(torch.bfloat16)
                         for _ in range(iters)]
        self.got_stage = [torch.empty_like(self.stage) for _ in range(iters)]
        self.got_src = [torch.empty((2,) + self.g.tensor_shape(), dtype=torch.bfloat16, device="cuda")
                        for _ in range(iters)]
        self.got_dst = [torch.empty((2,) + self.g.tensor_shape(), dtype=torch.bfloat16, device="cuda")
                        for _ in range(iters)]

    def iteration(self, i: int):
        for k in range(2):
            self.src[k].copy_(self.pat_cache[i][k])
        K.kv_pack_blocks(self.scache, self.x, self.n, self.stage)
        self.got_stage[i].copy_(self.stage)
        for k in range(2):
            self.dst[k].fill_(1.0)  # bf16 0x3f80 everywhere: unpack must replace the listed blocks
        self.stage.zero_()
        K.kv_unpack_blocks(self.dcache, self.stage, self.x, self.n, BS)
        for k in range(2):
            self.got_dst[i][k].copy_(self.dst[k])
            self.rows[k].copy_(self.pat_rows[i][k])
        K.kv_slot_mapping(self.table, self.req, self.pos, BS, self.slot)
        K.kv_reshape_and_cache(self.scache, self.rows, self.slot)
        for k in range(2):
            self.got_src[i][k].copy_(self.src[k])

    def check(self, i: int):
        host = [self.pat_cache[i][k].view(torch.int16).cpu().numpy().view(np.uint16) for k in range(2)]
        want_stage = oracle.pack(H.ora_cache(self.g, [h.copy() for h in host]), self.off, self.ids)
        np.testing.assert_array_equal(self.got_stage[i].cpu().numpy(), want_stage, err_msg=f"iteration {i}: pack")
        # unpack ran after the fill and saw the zeroed staging buffer: every listed destination
        # block is zero, every other block still holds the fill
        runs = self.x.host()
        got_dst = self.got_dst[i].view(torch.int16).cpu().numpy()
        listed = np.zeros(NB, dtype=bool)
        for r in range(runs["count"]):
            b0, nb = int(runs["dst_block"][r]), int(runs["n_blocks"][r])
            listed[b0:b0 + nb] = True
        assert listed.sum() == self.n
        assert not got_dst[:, listed].any(), f"iteration {i}: unpack read the staging before the memset"
        assert (got_dst[:, ~listed] == 0x3f80).all(), f"iteration {i}: unpack wrote outside its blocks"
        slot, bad = oracle.slot_mapping(self.table.cpu().numpy(), self.req.cpu().numpy(), self.pos.cpu().numpy(), BS)
        assert bad == 0
        sc = H.ora_cache(self.g, [h.copy() for h in host])
        rows = [self.pat_rows[i][k].reshape(self.T, -1).view(torch.uint8).cpu().numpy() for k in range(2)]
        assert oracle.reshape_and_cache(sc, rows, slot) == 0
        for k in range(2):
            np.testing.assert_array_equal(self.got_src[i][k].view(torch.int16).cpu().numpy().view(np.uint16),
                                          sc.tensors[k], err_msg=f"iteration {i}: reshape tensor {k}")


def test_interleaved_with_torch_work_eager():
    c = Case(iters=24, seed=7)
    K.kv_get_last_error(clear=True)
    for i in range(24):
        c.iteration(i)
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    for i in range(24):
        c.check(i)


def test_interleaved_with_torch_work_graph():
    c = Case(iters=8, seed=8)
    c.iteration(0)  # eager first: per-device state is looked up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(8):
            c.iteration(i)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert K.kv_get_last_error() == 0
    for i in range(8):
        c.check(i)
