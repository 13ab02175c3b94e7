"""CPU oracle for the paged KV-cache data path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path never does: it runs entirely in the
CUDA library and fails loudly when that library is missing.

The arithmetic lives in ``pagedkv_oracle.c`` (plain C, single-threaded); this
module builds it with gcc, loads it with ctypes and marshals numpy arrays.
``brute.py`` holds a second, independent pure-Python statement used to check
the C oracle on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

__all__ = ["build", "Cache", "slot_mapping", "reshape_and_cache", "build_xfer_list", "pack", "unpack",
           "clip_block_lists", "fnv1a64", "block_hashes"]


def build(force: bool = False, out: str = _LIB, defines=()) -> str:
    """Compile the oracle into a shared library (gcc, no SIMD intrinsics)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out, _SRC]
        cmd += [f"-D{d}" for d in defines]
        subprocess.run(cmd, check=True)
    return out


class _OraCache(ctypes.Structure):
    _fields_ = [
        ("n_tensors", ctypes.c_int32),
        ("base", ctypes.POINTER(ctypes.c_void_p)),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("n_planes", ctypes.c_int32),
        ("block_stride", ctypes.c_int64),
        ("plane_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("row_bytes", ctypes.c_int32),
    ]


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.ora_slot_mapping.argtypes = [P, i32, i32, i64, P, P, i64, i32, P]
    lib.ora_reshape_and_cache.argtypes = [ctypes.POINTER(_OraCache), P, i64, P, i64]
    lib.ora_build_xfer_list.argtypes = [P, i32, P, P, i64, i32, P, P, P, P, P, i64]
    lib.ora_pack.argtypes = [ctypes.POINTER(_OraCache), i32, i32, P, i32, P, i64, P]
    lib.ora_unpack.argtypes = [ctypes.POINTER(_OraCache), i32, i32, i32, i32, P, i32, i64, P, P, i64, P]
    lib.ora_clip_block_lists.argtypes = [P, i32, P, i64, P, i32, i32, P, P]
    lib.ora_fnv1a64.argtypes = [P, i64]
    lib.ora_fnv1a64.restype = ctypes.c_uint64
    lib.ora_block_hashes.argtypes = [P, i32, P, i64, i32, ctypes.c_uint64, P, P]
    for f in (lib.ora_slot_mapping, lib.ora_reshape_and_cache, lib.ora_build_xfer_list,
              lib.ora_pack, lib.ora_unpack, lib.ora_clip_block_lists, lib.ora_block_hashes):
        f.restype = i64
    return lib


def _get(lib=None):
    """The bound oracle library: the default build, a given path, or an already bound library."""
    global _lib
    if isinstance(lib, ctypes.CDLL):
        return lib
    if lib is not None:
        return _bind(lib)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


class Cache:
    """A host paged cache: C-contiguous numpy tensors plus the byte geometry of a block."""

    def __init__(self, tensors, num_blocks, block_size, n_planes, block_stride, plane_stride,
                 token_stride, row_bytes):
        self.tensors = [np.ascontiguousarray(t) for t in tensors]
        self.num_blocks, self.block_size, self.n_planes = int(num_blocks), int(block_size), int(n_planes)
        self.block_stride, self.plane_stride = int(block_stride), int(plane_stride)
        self.token_stride, self.row_bytes = int(token_stride), int(row_bytes)
        self._bases = (ctypes.c_void_p * max(1, len(self.tensors)))(*[t.ctypes.data for t in self.tensors])

    def c(self) -> _OraCache:
        return _OraCache(len(self.tensors), ctypes.cast(self._bases, ctypes.POINTER(ctypes.c_void_p)),
                         self.num_blocks, self.block_size, self.n_planes, self.block_stride,
                         self.plane_stride, self.token_stride, self.row_bytes)


def slot_mapping(block_table, token_req, token_pos, block_size, lib=None):
    """slot[i] = block_table[req_i, pos_i // bs] * bs + pos_i % bs; -1 for invalid tokens.

    Returns (slots int64 [T], number of invalid tokens)."""
    bt = _i32(block_table)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    req, pos = _i32(token_req), _i32(token_pos)
    out = np.empty(req.shape[0], dtype=np.int64)
    bad = _get(lib).ora_slot_mapping(_ptr(bt), bt.shape[0], bt.shape[1], bt.shape[1], _ptr(req), _ptr(pos),
                                     req.shape[0], int(block_size), _ptr(out))
    return out, int(bad)


def reshape_and_cache(cache: Cache, new_rows, slot, lib=None) -> int:
    """Write new token rows into the cache at their slots (in place).

    new_rows: n_tensors * n_planes C-contiguous arrays [T, row_bytes] (tensor-major,
    plane-minor).  Returns the number of out-of-range tokens, or -1 on duplicate slots."""
    rows = [np.ascontiguousarray(r) for r in new_rows]
    assert len(rows) == len(cache.tensors) * cache.n_planes
    slot = np.ascontiguousarray(slot, dtype=np.int64)
    stride = rows[0].strides[0] if rows and rows[0].ndim > 1 else cache.row_bytes
    ptrs = (ctypes.c_void_p * max(1, len(rows)))(*[r.ctypes.data for r in rows])
    c = cache.c()
    return int(_get(lib).ora_reshape_and_cache(ctypes.byref(c), ptrs, stride, _ptr(slot), slot.shape[0]))


def build_xfer_list(req_offsets, src_ids, dst_ids=None, max_run_blocks=0, lib=None) -> dict:
    """Maximal contiguous runs per request (capped at max_run_blocks; 0 = no cap)."""
    off, src = _i32(req_offsets), _i32(src_ids)
    dst = None if dst_ids is None else _i32(dst_ids)
    n = src.shape[0]
    cap = max(n, 1)
    req, rs, rd, rl = (np.zeros(cap, np.int32) for _ in range(4))
    stage = np.zeros(cap, np.int64)
    k = _get(lib).ora_build_xfer_list(_ptr(off), off.shape[0] - 1, _ptr(src),
                                      None if dst is None else _ptr(dst), n, int(max_run_blocks),
                                      _ptr(req), _ptr(rs), _ptr(rd), _ptr(rl), _ptr(stage), cap)
    if k < 0:
        raise ValueError(f"oracle xfer_list rejected its input ({k})")
    return dict(req=req[:k], src_block=rs[:k], dst_block=rd[:k], n_blocks=rl[:k], stage_block=stage[:k])


def stage_bytes(n_tensors, n_blocks, n_planes, block_size, slice_bytes) -> int:
    return int(n_tensors) * int(n_blocks) * int(n_planes) * int(block_size) * int(slice_bytes)


def pack(cache: Cache, req_offsets, src_ids, slice_off=0, slice_bytes=None, lib=None) -> np.ndarray:
    """Gather the listed blocks into a fresh staging buffer (uint8)."""
    off, src = _i32(req_offsets), _i32(src_ids)
    sb = cache.row_bytes if slice_bytes is None else int(slice_bytes)
    out = np.empty(stage_bytes(len(cache.tensors), src.shape[0], cache.n_planes, cache.block_size, sb),
                   dtype=np.uint8)
    c = cache.c()
    st = _get(lib).ora_pack(ctypes.byref(c), int(slice_off), sb, _ptr(off), off.shape[0] - 1, _ptr(src),
                            src.shape[0], _ptr(out))
    if st != 0:
        raise ValueError("oracle pack rejected its input")
    return out


def unpack(cache: Cache, stage, req_offsets, dst_req_offsets, dst_ids, src_block_size, slice_bytes,
           dst_slice_off=0, lib=None) -> int:
    """Scatter a staging buffer into the cache (in place). Returns 0, or -1 if rejected."""
    off, doff, dids = _i32(req_offsets), _i32(dst_req_offsets), _i32(dst_ids)
    stage = np.ascontiguousarray(stage).view(np.uint8)
    n = int(off[-1]) if off.shape[0] else 0
    c = cache.c()
    return int(_get(lib).ora_unpack(ctypes.byref(c), int(dst_slice_off), int(slice_bytes), int(src_block_size),
                                    cache.n_planes, _ptr(off), off.shape[0] - 1, n, _ptr(doff), _ptr(dids),
                                    dids.shape[0], _ptr(stage)))


def clip_block_lists(req_offsets, ids, n_tokens, window, block_size, lib=None):
    """Sliding-window clip of per-request block lists; returns (out_offsets, out_ids)."""
    off, ids_, nt = _i32(req_offsets), _i32(ids), _i32(n_tokens)
    out_off = np.zeros(off.shape[0], np.int32)
    out = np.zeros(max(1, ids_.shape[0]), np.int32)
    k = _get(lib).ora_clip_block_lists(_ptr(off), off.shape[0] - 1, _ptr(ids_), ids_.shape[0], _ptr(nt), int(window),
                                       int(block_size), _ptr(out_off), _ptr(out))
    if k < 0:
        raise ValueError("oracle clip_block_lists rejected its input")
    return out_off, out[:k]


def fnv1a64(data: bytes, lib=None) -> int:
    """FNV-1a 64 of a byte string (the hash of the prefix chain)."""
    buf = np.frombuffer(bytes(data) or b"\0", dtype=np.uint8).copy()
    return int(_get(lib).ora_fnv1a64(_ptr(buf), len(data)))


def block_hashes(tok_offsets, tokens, block_size, seed, lib=None):
    """Prefix hash chain of every request's full blocks; returns (out_offsets int32, hashes uint64)."""
    off, tok = _i32(tok_offsets), _i32(tokens)
    n_full = sum(int(off[r + 1] - off[r]) // int(block_size) for r in range(off.shape[0] - 1))
    out_off = np.zeros(off.shape[0], np.int32)
    out = np.zeros(max(1, n_full), np.uint64)
    k = _get(lib).ora_block_hashes(_ptr(off), off.shape[0] - 1, _ptr(tok), tok.shape[0], int(block_size),
                                   int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out_off), _ptr(out))
    if k < 0:
        raise ValueError("oracle block_hashes rejected its input")
    return out_off, out[:k]
