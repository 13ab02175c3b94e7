"""Brute-force restatement of the path, used only to check the C oracle on tiny inputs.

Test infrastructure.  It takes a different route from the C oracle on purpose:
instead of the slot formula it enumerates how the paged allocator fills blocks
(a request's k-th block holds its next block_size tokens; drawing "vllm v1 调度逻辑
和 distributed 分布式原理", "Paged kv cache" and "batch tensor 组装"), numbers the
physical slots with numpy's C-order flat index, and moves rows one token at a
time through strided numpy views.
"""
from __future__ import annotations

import numpy as np


def token_slots(table_row, n_tokens, num_blocks, block_size):
    """Flat physical slot of each of a request's first n_tokens tokens, by enumeration."""
    slots = []
    for block in table_row:
        for offset in range(block_size):
            if len(slots) == n_tokens:
                return slots
            slots.append(int(np.ravel_multi_index((int(block), offset), (num_blocks, block_size))))
    assert len(slots) == n_tokens, "table too short"
    return slots


def slot_mapping(block_table, token_req, token_pos, num_blocks, block_size):
    out = []
    for r, pos in zip(token_req, token_pos):
        out.append(token_slots(block_table[r], int(pos) + 1, num_blocks, block_size)[-1])
    return np.array(out, dtype=np.int64)


def rows_view(tensor: np.ndarray, num_blocks, n_planes, block_size, block_stride, plane_stride,
              token_stride, row_bytes):
    """A [num_blocks, n_planes, block_size, row_bytes] uint8 view of one cache tensor."""
    flat = tensor.reshape(-1).view(np.uint8)
    return np.lib.stride_tricks.as_strided(
        flat, shape=(num_blocks, n_planes, block_size, row_bytes),
        strides=(block_stride, plane_stride, token_stride, 1), writeable=True)


def reshape_and_cache(views, new_rows, slots, num_blocks, block_size):
    """views[t]: rows_view of tensor t; new_rows[t][p]: [T, row_bytes] uint8."""
    for i, s in enumerate(slots):
        if s < 0:
            continue
        block, offset = np.unravel_index(int(s), (num_blocks, block_size))
        for t, v in enumerate(views):
            for p in range(v.shape[1]):
                v[block, p, offset, :] = new_rows[t][p][i]


def pack(views, req_lists, block_size, slice_off, slice_bytes):
    """Staging bytes: tensor, request, block, plane, slot; each entry one row slice."""
    parts = []
    num_blocks = views[0].shape[0] if views else 0
    for v in views:
        for ids in req_lists:
            slots = token_slots(ids, len(ids) * block_size, num_blocks, block_size)
            # group the request's tokens by block, then emit every plane of the block
            for k in range(len(ids)):
                blk_slots = slots[k * block_size:(k + 1) * block_size]
                for p in range(v.shape[1]):
                    for s in blk_slots:
                        b, o = np.unravel_index(s, (num_blocks, block_size))
                        parts.append(v[b, p, o, slice_off:slice_off + slice_bytes].copy())
    return np.concatenate(parts) if parts else np.zeros(0, np.uint8)


def unpack(views, stage, src_counts, dst_lists, src_block_size, dst_block_size, n_planes, slice_bytes,
           dst_slice_off):
    """Scatter staging (pack's order, source geometry) into destination views, token by token."""
    pos = 0
    num_blocks = views[0].shape[0] if views else 0
    for v in views:
        for n_src, dst_ids in zip(src_counts, dst_lists):
            n_tok = n_src * src_block_size
            dslots = token_slots(dst_ids, n_tok, num_blocks, dst_block_size)
            for k in range(n_src):
                for p in range(n_planes):
                    for o in range(src_block_size):
                        b, off = np.unravel_index(dslots[k * src_block_size + o], (num_blocks, dst_block_size))
                        v[b, p, off, dst_slice_off:dst_slice_off + slice_bytes] = stage[pos:pos + slice_bytes]
                        pos += slice_bytes
    assert pos == stage.shape[0]


def xfer_runs(req_lists, dst_lists=None, max_run_blocks=0):
    """Runs by grouping: inside a run, id minus list position is constant (for src and dst)."""
    runs = []
    pos = 0
    for r, ids in enumerate(req_lists):
        dids = None if dst_lists is None else dst_lists[r]
        group = None
        for k, s in enumerate(ids):
            key = (int(s) - k, None if dids is None else int(dids[k]) - k)
            if group is not None and group[0] == key and (max_run_blocks == 0 or group[1][3] < max_run_blocks):
                group[1][3] += 1
            else:
                group = (key, [r, int(s), -1 if dids is None else int(dids[k]), 1, pos + k])
                runs.append(group[1])
        pos += len(ids)
    return runs
