"""One pass of the paged KV-cache hot path over one batch, through the C ABI.

A step runs these calls (3 on a second stream, beside 1 and 2; 4 waits for all three):
  1. kv_slot_mapping        new tokens' slots from the shared block table (when the batch has new tokens)
  2. kv_reshape_and_cache   their K/V rows into every layer's paged tensor
  3. kv_build_xfer_list     the send side's per-request block lists -> contiguous runs
                            (optionally after kv_clip_block_lists, the sliding-window clip)
  4. kv_pack_blocks         those runs of every tensor -> the staging buffer
  5. kv_unpack_blocks       the staging buffer -> the receiver's cache (whole blocks, or
                            token-granular onto another block size / head slice)
This module only allocates the step's buffers and orders the calls; every step of the
data path runs in libpagedkv.so.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import pagedkv as K
from .workloads import Case, Workload


@dataclass
class StepBytes:
    """Algorithmic bytes of each call of one step (payload read + written, plus index arrays)."""

    slot_mapping: int
    reshape_and_cache: int
    build_xfer_list: int
    pack: int
    unpack: int

    @property
    def total(self) -> int:
        return self.slot_mapping + self.reshape_and_cache + self.build_xfer_list + self.pack + self.unpack


class TransferStep:
    def __init__(self, wl: Workload, case: Case, src_tensors, dst_tensors=None, new_kv=None,
                 max_run_blocks: Optional[int] = None, device="cuda", host_stage: bool = False,
                 sw_window: Optional[int] = None):
        self.wl, self.case = wl, case
        self.device = torch.device(device)
        self.src = K.PagedCache.from_tensors(src_tensors, wl.src.layout)
        self.dst = K.PagedCache.from_tensors(dst_tensors, wl.dst.layout) if dst_tensors is not None else None
        self.new_kv = list(new_kv) if new_kv is not None else []
        dev = self.device

        def t(a):
            return torch.from_numpy(a).to(dev)

        self.req_offsets = t(case.req_offsets)
        self.src_ids = t(case.src_ids)
        self.equal = wl.equal_geometry
        self.dst_req_offsets = t(case.dst_req_offsets)
        self.dst_ids = t(case.dst_ids)
        self.n_tokens = case.n_tokens
        if self.n_tokens:
            self.block_table = t(case.block_table)
            self.token_req = t(case.token_req)
            self.token_pos = t(case.token_pos)
            self.slot = torch.empty(self.n_tokens, dtype=torch.int64, device=dev)
        self.slice_off = wl.slice_off
        self.slice_bytes = wl.moved_slice
        stage_block = wl.src.n_planes * wl.src.block_size * self.slice_bytes
        self.max_run_blocks = K.default_max_run_blocks(stage_block) if max_run_blocks is None else max_run_blocks
        n = case.n_blocks
        self.sw_window = sw_window
        if sw_window:
            if not self.equal:
                raise ValueError("the sliding-window clip keeps source and destination lists aligned entry by entry;"
                                 " it needs equal geometry")
            self.req_tokens = t(case.req_tokens)
            self.clip_offsets = torch.empty_like(self.req_offsets)
            self.clip_src = torch.empty(max(1, n), dtype=torch.int32, device=dev)
            self.clip_dst = torch.empty(max(1, n), dtype=torch.int32, device=dev)
            n = self.kept_blocks(case, sw_window, wl.src.block_size)
        self.n_listed = n
        self.xfer = K.XferList(n, dev, self.max_run_blocks)
        self.workspace = torch.empty(K.kv_xfer_workspace_bytes(n), dtype=torch.uint8, device=dev)
        sd = K.stage_desc(n, len(self.src.tensors), wl.src.n_planes, wl.src.block_size, self.slice_bytes)
        # the staging buffer lives in HBM, or in pinned host memory (the receiver's spill target)
        if host_stage:
            self.stage = torch.empty(max(16, K.stage_nbytes(sd)), dtype=torch.uint8, pin_memory=True)
        else:
            self.stage = torch.empty(max(16, K.stage_nbytes(sd)), dtype=torch.uint8, device=dev)

    # -- the five calls ---------------------------------------------------------
    def write_tokens(self, stream=None):
        if not self.n_tokens:
            return
        K.kv_slot_mapping(self.block_table, self.token_req, self.token_pos, self.src.block_size, self.slot, stream)
        K.kv_reshape_and_cache(self.src, self.new_kv, self.slot, stream)

    def write_tokens_call(self, stream=None):
        """The same write as write_tokens through the one call kv_write_tokens, slots kept (the row
        copy looks the slots up and writes them to self.slot)."""
        if not self.n_tokens:
            return
        K.kv_write_tokens(self.src, self.new_kv, self.block_table, self.token_req, self.token_pos, self.slot,
                          stream)

    def write_tokens_fused(self, stream=None):
        """The same cache write through kv_write_tokens without slot_out: the slot lookup fused into
        the row copy (one launch); the slots are not kept."""
        if not self.n_tokens:
            return
        K.kv_write_tokens(self.src, self.new_kv, self.block_table, self.token_req, self.token_pos, None, stream)

    @staticmethod
    def kept_blocks(case: Case, window: int, block_size: int) -> int:
        """Entries the sliding-window clip keeps, from the host's copy of the per-request
        token counts and list lengths (sizes the staging buffer without a device read)."""
        kept = 0
        for r in range(case.n_reqs):
            n = int(case.req_tokens[r])
            length = int(case.req_offsets[r + 1] - case.req_offsets[r])
            end = min(-(-n // block_size), length)
            first = min((max(0, n - window) if window > 0 else 0) // block_size, end)
            kept += end - first
        return kept

    def build(self, stream=None):
        use_dst = self.equal and self.dst is not None
        offsets, src, dst = self.req_offsets, self.src_ids, self.dst_ids if use_dst else None
        if self.sw_window:
            bs = self.wl.src.block_size
            K.kv_clip_block_lists(self.req_offsets, self.src_ids, self.req_tokens, self.sw_window, bs,
                                  self.clip_offsets, self.clip_src, stream)
            if use_dst:
                K.kv_clip_block_lists(self.req_offsets, self.dst_ids, self.req_tokens, self.sw_window, bs,
                                      self.clip_offsets, self.clip_dst, stream)
            offsets, src = self.clip_offsets, self.clip_src[:self.n_listed]
            dst = self.clip_dst[:self.n_listed] if use_dst else None
        K.kv_build_xfer_list(offsets, src, dst, self.max_run_blocks, self.xfer, self.workspace, stream)

    def pack(self, stream=None):
        K.kv_pack_blocks(self.src, self.xfer, self.n_listed, self.stage, self.slice_off, self.slice_bytes, stream)

    def unpack(self, stream=None):
        if self.dst is None:
            return
        if self.equal:
            K.kv_unpack_blocks(self.dst, self.stage, self.xfer, self.n_listed, self.wl.src.block_size,
                               self.slice_bytes, self.wl.dst_slice_off, stream=stream)
        else:
            K.kv_unpack_blocks(self.dst, self.stage, self.xfer, self.n_listed, self.wl.src.block_size,
                               self.slice_bytes, self.wl.dst_slice_off, self.req_offsets, self.dst_req_offsets,
                               self.dst_ids, stream=stream)

    def side_stream(self) -> "torch.cuda.Stream":
        """The second stream the builder runs on (created on first use), at the highest priority:
        its few small CTAs are then placed before reshape_and_cache's as SMs free up."""
        if getattr(self, "_side", None) is None:
            lo, hi = torch.cuda.Stream.priority_range()
            self._side = torch.cuda.Stream(self.device, priority=min(lo, hi))
        return self._side

    def run(self, stream=None):
        """The five calls.  The block lists do not depend on the new tokens, so the builder (after
        the clip, when there is one) runs on a second stream beside slot_mapping and
        reshape_and_cache; pack waits for both.  The builder is issued first: its one CTA needs a
        nearly empty SM, which it would not get once reshape_and_cache's grid fills the GPU."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        side = self.side_stream()
        side.wait_stream(main)  # the step's inputs are ready
        self.build(side)
        self.write_tokens(main)
        main.wait_stream(side)
        self.pack(main)
        self.unpack(main)

    def capture(self, fn=None, stream=None) -> "torch.cuda.CUDAGraph":
        """Capture run() (or another method of this step, e.g. write_tokens) into a CUDA graph for
        replay - the way to issue launch-bound steps such as a decode write.

        Run the step once eagerly first: the first call of each entry point on a device looks up
        per-device state, which must not happen during a capture.  A replay repeats the same
        five calls on the same buffers; refresh the input tensors in place between replays."""
        g = torch.cuda.CUDAGraph()
        s = stream if stream is not None else torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.graph(g, stream=s):
            (fn or self.run)()
        torch.cuda.current_stream(self.device).wait_stream(s)
        return g

    @property
    def launches_per_step(self) -> int:
        """Kernels of libpagedkv one run() launches (one launch per 128 tensors for the copies)."""
        groups = -(-len(self.src.tensors) // 128)
        n = 1 + groups  # builder + pack
        if self.sw_window:
            n += 2 * (2 if (self.equal and self.dst is not None) else 1)  # clip: count + copy per list
        if self.n_tokens:
            n += 1 + groups
        if self.dst is not None:
            n += groups
        return n

    # -- algorithmic bytes ----------------------------------------------------
    def bytes(self) -> StepBytes:
        wl, case = self.wl, self.case
        nt = len(self.src.tensors)
        payload = nt * self.n_listed * wl.src.n_planes * wl.src.block_size * self.slice_bytes
        T = self.n_tokens
        slot_b = T * (4 + 4 + 4 + 8) if T else 0  # req, pos, table entry read; slot written
        reshape_b = (nt * wl.src.n_planes * T * wl.src.row_bytes * 2 + T * 8) if T else 0
        lists = 2 if (self.equal and self.dst is not None) else 1
        build_b = self.n_listed * 4 * lists
        if self.sw_window:  # the clip reads every entry and writes the kept ones, per list
            build_b += (case.n_blocks + self.n_listed) * 4 * lists
        return StepBytes(slot_b, reshape_b, build_b, 2 * payload, 2 * payload if self.dst is not None else 0)
