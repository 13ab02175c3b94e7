"""ctypes binding of libpagedkv.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch CUDA
tensors, passes their data pointers and the current CUDA stream, and raises
``KvError`` on a non-zero status.  No step of the data path runs in Python or on the
CPU: when the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("PAGEDKV_LIB") or os.path.join(_HERE, "libpagedkv.so")

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_ALIGN, KV_ERR_RANGE, KV_ERR_CUDA, KV_ERR_TIMEOUT, KV_ERR_UNSUPPORTED = range(7)
KV_DERR_TABLE, KV_DERR_SLOT, KV_DERR_BLOCK, KV_DERR_LIST = 0x01, 0x02, 0x04, 0x08
KV_DERR_CAPACITY, KV_DERR_STAGE, KV_DERR_DST_TABLE, KV_DERR_TIMEOUT = 0x10, 0x20, 0x40, 0x80

RUN_WORDS = 6  # a kv_xfer_run is 24 bytes: six int32 words (the last two hold the int64 stage_block)
EXPORTS = ("kv_version", "kv_status_string", "kv_last_cuda_error", "kv_slot_mapping", "kv_reshape_and_cache",
           "kv_xfer_workspace_bytes", "kv_build_xfer_list", "kv_pack_blocks", "kv_unpack_blocks",
           "kv_get_last_error", "kv_build_xfer_list_static", "kv_unpack_blocks_signal", "kv_wait_signal",
           "kv_clip_block_lists", "kv_block_hashes", "kv_block_hashes_workspace_bytes", "kv_write_tokens")


class KvError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {_status_name(status)}{(' ' + detail) if detail else ''}")


class KvCacheDesc(ctypes.Structure):
    _fields_ = [
        ("n_tensors", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("n_planes", ctypes.c_int32),
        ("row_bytes", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("block_stride", ctypes.c_int64),
        ("plane_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("base", ctypes.POINTER(ctypes.c_uint64)),
    ]


class KvStageDesc(ctypes.Structure):
    _fields_ = [
        ("n_blocks", ctypes.c_int64),
        ("n_tensors", ctypes.c_int32),
        ("n_planes", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("slice_bytes", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load and bind libpagedkv.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        D = ctypes.POINTER(KvCacheDesc)
        S = ctypes.POINTER(KvStageDesc)
        sig = {
            "kv_version": ([], ctypes.c_char_p),
            "kv_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "kv_last_cuda_error": ([], ctypes.c_int),
            "kv_slot_mapping": ([P, i32, i32, i64, P, P, i64, i32, P, P], ctypes.c_int),
            "kv_reshape_and_cache": ([D, P, i64, P, i64, P], ctypes.c_int),
            "kv_xfer_workspace_bytes": ([i64, ctypes.POINTER(i64)], ctypes.c_int),
            "kv_build_xfer_list": ([P, i32, P, P, i64, i32, P, i64, P, P, i64, P], ctypes.c_int),
            "kv_pack_blocks": ([D, i32, S, P, P, i64, i32, P, i64, P], ctypes.c_int),
            "kv_unpack_blocks": ([D, i32, S, P, P, i64, i32, P, i64, P, P, P, i32, P], ctypes.c_int),
            "kv_get_last_error": ([ctypes.POINTER(i32), i32, P], ctypes.c_int),
            "kv_build_xfer_list_static": ([P, i32, P, P, i64, i32, P, i64, P, P], ctypes.c_int),
            "kv_unpack_blocks_signal": ([D, i32, S, P, P, i64, i32, P, i64, P, P, P, i32, P, ctypes.c_uint64, P],
                                        ctypes.c_int),
            "kv_wait_signal": ([P, ctypes.c_uint64, ctypes.c_uint32, P, P], ctypes.c_int),
            "kv_clip_block_lists": ([P, i32, P, i64, P, i32, i32, P, P, i64, P], ctypes.c_int),
            "kv_block_hashes": ([P, i32, P, i64, i32, ctypes.c_uint64, P, P, i64, P, i64, P], ctypes.c_int),
            "kv_block_hashes_workspace_bytes": ([i64, i32, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
            "kv_write_tokens": ([D, P, i64, P, i32, i32, i64, P, P, i64, P, P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes, f.restype = args, res
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load().kv_status_string(status).decode()
    except Exception:  # the library may be what is missing
        return f"status {status}"


def _check(fn: str, status: int):
    if status != KV_OK:
        detail = f"(cuda error {load().kv_last_cuda_error()})" if status == KV_ERR_CUDA else ""
        raise KvError(fn, status, detail)


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[ctypes.c_void_p]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpagedkv takes CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stage_ptr(t: torch.Tensor) -> ctypes.c_void_p:
    """Staging may live in device memory or in pinned host memory (reached over the host link)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("the staging buffer must be a CUDA tensor or pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def _i32(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def version() -> str:
    return load().kv_version().decode()


# ---------------------------------------------------------------------------
# cache geometry
# ---------------------------------------------------------------------------
@dataclass
class PagedCache:
    """A paged cache: equal-shaped device tensors plus their byte geometry (kv_cache_desc)."""

    tensors: list
    num_blocks: int
    block_size: int
    n_planes: int
    row_bytes: int
    block_stride: int
    plane_stride: int
    token_stride: int

    @classmethod
    def from_tensors(cls, tensors: Sequence[torch.Tensor], layout: str) -> "PagedCache":
        """layout: "separate" / "mla" ([num_blocks, bs, ...row]), "blocks_first"
        ([num_blocks, 2, bs, ...row]) or "kv_first" ([2, num_blocks, bs, ...row])."""
        tensors = list(tensors)
        t = tensors[0]
        e = t.element_size()
        st = [s * e for s in t.stride()]
        if layout in ("separate", "mla"):
            nb, bs, planes = t.shape[0], t.shape[1], 1
            block, plane, token, rest = st[0], st[0], st[1], t.shape[2:]
        elif layout == "blocks_first":
            nb, bs, planes = t.shape[0], t.shape[2], 2
            block, plane, token, rest = st[0], st[1], st[2], t.shape[3:]
            assert t.shape[1] == 2
        elif layout == "kv_first":
            nb, bs, planes = t.shape[1], t.shape[2], 2
            block, plane, token, rest = st[1], st[0], st[2], t.shape[3:]
            assert t.shape[0] == 2
        else:
            raise ValueError(layout)
        row = e
        for d in rest:
            row *= d
        for x in tensors:
            if x.shape != t.shape or x.stride() != t.stride() or x.dtype != t.dtype or not x.is_cuda:
                raise ValueError("cache tensors must share shape, strides and dtype and live on the GPU")
        return cls(tensors, int(nb), int(bs), planes, int(row), int(block), int(plane), int(token))

    def desc(self) -> KvCacheDesc:
        """The kv_cache_desc of these tensors, built once and rebuilt only if a tensor moved."""
        ptrs = tuple(x.data_ptr() for x in self.tensors)
        if getattr(self, "_desc_ptrs", None) != ptrs:
            n = len(ptrs)
            self._bases = (ctypes.c_uint64 * max(1, n))(*ptrs)
            self._desc = KvCacheDesc(n, self.block_size, self.n_planes, self.row_bytes, self.num_blocks,
                                     self.block_stride, self.plane_stride, self.token_stride,
                                     ctypes.cast(self._bases, ctypes.POINTER(ctypes.c_uint64)))
            self._desc_ptrs = ptrs
        return self._desc


def stage_desc(n_blocks: int, n_tensors: int, n_planes: int, block_size: int, slice_bytes: int) -> KvStageDesc:
    return KvStageDesc(int(n_blocks), int(n_tensors), int(n_planes), int(block_size), int(slice_bytes))


def stage_nbytes(sd: KvStageDesc) -> int:
    return sd.n_blocks * sd.n_tensors * sd.n_planes * sd.block_size * sd.slice_bytes


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def kv_slot_mapping(block_table: torch.Tensor, token_req: torch.Tensor, token_pos: torch.Tensor, block_size: int,
                    slot_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _i32(token_req, "token_req"), _i32(token_pos, "token_pos")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be a row-major int32 [n_reqs, max_blocks] CUDA tensor")
    n = token_req.shape[0]
    if slot_out is None:
        slot_out = torch.empty(n, dtype=torch.int64, device=token_req.device)
    _check("kv_slot_mapping", load().kv_slot_mapping(
        _ptr(block_table), block_table.shape[0], block_table.shape[1], block_table.stride(0), _ptr(token_req),
        _ptr(token_pos), n, int(block_size), _ptr(slot_out), _stream(stream)))
    return slot_out


def kv_reshape_and_cache(cache: PagedCache, new_kv: Sequence[torch.Tensor], slot: torch.Tensor, stream=None):
    """new_kv: n_tensors * n_planes tensors [T, ...row] (tensor-major, plane-minor), equal strides."""
    if slot.dtype != torch.int64:
        raise ValueError("slot must be int64")
    new_kv = list(new_kv)
    stride = new_kv[0].stride(0) * new_kv[0].element_size() if new_kv else cache.row_bytes
    ptrs = (ctypes.c_uint64 * max(1, len(new_kv)))(*[x.data_ptr() for x in new_kv])
    d = cache.desc()
    _check("kv_reshape_and_cache", load().kv_reshape_and_cache(
        ctypes.byref(d), ctypes.cast(ptrs, ctypes.c_void_p), stride, _ptr(slot), slot.shape[0], _stream(stream)))


def kv_write_tokens(cache: PagedCache, new_kv: Sequence[torch.Tensor], block_table: torch.Tensor,
                    token_req: torch.Tensor, token_pos: torch.Tensor, slot_out: Optional[torch.Tensor] = None,
                    stream=None):
    """kv_slot_mapping + kv_reshape_and_cache in one call: the row copy looks each token's slot up in
    the block table (one launch per 128 tensors); slot_out (int64 [T]) optionally gets the slots."""
    _i32(token_req, "token_req"), _i32(token_pos, "token_pos")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be a row-major int32 [n_reqs, max_blocks] CUDA tensor")
    new_kv = list(new_kv)
    stride = new_kv[0].stride(0) * new_kv[0].element_size() if new_kv else cache.row_bytes
    ptrs = (ctypes.c_uint64 * max(1, len(new_kv)))(*[x.data_ptr() for x in new_kv])
    _check("kv_write_tokens", load().kv_write_tokens(
        ctypes.byref(cache.desc()), ctypes.cast(ptrs, ctypes.c_void_p), stride, _ptr(block_table),
        block_table.shape[0], block_table.shape[1], block_table.stride(0), _ptr(token_req), _ptr(token_pos),
        token_req.shape[0], _ptr(slot_out), _stream(stream)))


def kv_xfer_workspace_bytes(n_blocks: int) -> int:
    out = ctypes.c_int64(0)
    _check("kv_xfer_workspace_bytes", load().kv_xfer_workspace_bytes(int(n_blocks), ctypes.byref(out)))
    return out.value


class XferList:
    """Device output of kv_build_xfer_list: run records [capacity, 6] int32 and the run count."""

    def __init__(self, capacity: int, device, max_run_blocks: int):
        self.capacity = int(capacity)
        self.max_run_blocks = int(max_run_blocks)
        self.runs = torch.empty((max(1, self.capacity), RUN_WORDS), dtype=torch.int32, device=device)
        self.n_runs = torch.zeros(1, dtype=torch.int32, device=device)
        self._ws = None
        self._ws_blocks = -1

    def workspace(self, n_blocks: int) -> torch.Tensor:
        """A builder workspace for lists of n_blocks entries, kept with this list for reuse."""
        if self._ws is None or self._ws_blocks < n_blocks:
            self._ws = torch.empty(kv_xfer_workspace_bytes(n_blocks), dtype=torch.uint8, device=self.runs.device)
            self._ws_blocks = n_blocks
        return self._ws

    def host(self) -> dict:
        """Copy the runs to the host as numpy columns (synchronises)."""
        n = min(int(self.n_runs.item()), self.capacity)
        r = self.runs[:n].cpu()
        return dict(req=r[:, 0].numpy(), src_block=r[:, 1].numpy(), dst_block=r[:, 2].numpy(),
                    n_blocks=r[:, 3].numpy(), stage_block=r[:, 4:6].contiguous().view(torch.int64)[:, 0].numpy(),
                    count=int(self.n_runs.item()))


def kv_build_xfer_list(req_offsets: torch.Tensor, src_ids: torch.Tensor, dst_ids: Optional[torch.Tensor] = None,
                       max_run_blocks: int = 0, out: Optional[XferList] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> XferList:
    _i32(req_offsets, "req_offsets"), _i32(src_ids, "src_ids")
    if dst_ids is not None:
        _i32(dst_ids, "dst_ids")
    n = src_ids.shape[0]
    if out is None:
        out = XferList(n, src_ids.device, max_run_blocks)
    if workspace is None:
        workspace = out.workspace(n)
    _check("kv_build_xfer_list", load().kv_build_xfer_list(
        _ptr(req_offsets), req_offsets.shape[0] - 1, _ptr(src_ids), _ptr(dst_ids), n, int(max_run_blocks),
        _ptr(out.runs), out.capacity, _ptr(out.n_runs), _ptr(workspace), workspace.numel(), _stream(stream)))
    out.max_run_blocks = int(max_run_blocks)
    return out


def kv_clip_block_lists(req_offsets: torch.Tensor, ids: torch.Tensor, n_tokens: torch.Tensor, window: int,
                        block_size: int, out_offsets: Optional[torch.Tensor] = None,
                        out_ids: Optional[torch.Tensor] = None, stream=None):
    """Sliding-window clip of per-request block lists; returns device (out_offsets, out_ids)
    where out_ids has room for every input entry and out_offsets[-1] is the kept count."""
    _i32(req_offsets, "req_offsets"), _i32(ids, "ids"), _i32(n_tokens, "n_tokens")
    if out_offsets is None:
        out_offsets = torch.empty_like(req_offsets)
    if out_ids is None:
        out_ids = torch.empty(max(1, ids.shape[0]), dtype=torch.int32, device=ids.device)
    _check("kv_clip_block_lists", load().kv_clip_block_lists(
        _ptr(req_offsets), req_offsets.shape[0] - 1, _ptr(ids), ids.shape[0], _ptr(n_tokens), int(window),
        int(block_size), _ptr(out_offsets), _ptr(out_ids), out_ids.shape[0], _stream(stream)))
    return out_offsets, out_ids


def kv_block_hashes_workspace_bytes(n_tokens: int, block_size: int) -> int:
    out = ctypes.c_int64(0)
    _check("kv_block_hashes_workspace_bytes", load().kv_block_hashes_workspace_bytes(int(n_tokens), int(block_size),
                                                                                     ctypes.byref(out)))
    return out.value


def kv_block_hashes(tok_offsets: torch.Tensor, tokens: torch.Tensor, block_size: int, seed: int,
                    out_offsets: Optional[torch.Tensor] = None, out_hashes: Optional[torch.Tensor] = None,
                    workspace="auto", stream=None):
    """Prefix hash chain of every request's full token blocks; returns device (out_offsets int32,
    out_hashes int64 holding the uint64 bit patterns).  workspace: "auto" (a uint8 device tensor
    of kv_block_hashes_workspace_bytes is allocated here, for the table path), None (the plain
    per-request chain) or a caller's uint8 tensor."""
    _i32(tok_offsets, "tok_offsets"), _i32(tokens, "tokens")
    cap = max(1, tokens.shape[0] // int(block_size))
    if out_offsets is None:
        out_offsets = torch.empty_like(tok_offsets)
    if out_hashes is None:
        out_hashes = torch.empty(cap, dtype=torch.int64, device=tokens.device)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError(f"workspace must be 'auto', None or a tensor, not {workspace!r}")
        need = kv_block_hashes_workspace_bytes(tokens.shape[0], block_size)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=tokens.device)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("kv_block_hashes", load().kv_block_hashes(
        _ptr(tok_offsets), tok_offsets.shape[0] - 1, _ptr(tokens), tokens.shape[0], int(block_size),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out_offsets), _ptr(out_hashes), out_hashes.shape[0], ws_ptr, ws_bytes,
        _stream(stream)))
    return out_offsets, out_hashes


KV_XFER_STATIC_MAX_BLOCKS = 4177920


def kv_build_xfer_list_static(req_offsets: torch.Tensor, src_ids: torch.Tensor,
                              dst_ids: Optional[torch.Tensor] = None, max_run_blocks: int = 0,
                              out: Optional[XferList] = None, stream=None) -> XferList:
    """kv_build_xfer_list without a workspace: the library's own fixed scratch array is used,
    so the call itself allocates nothing (the outputs are still the caller's)."""
    _i32(req_offsets, "req_offsets"), _i32(src_ids, "src_ids")
    if dst_ids is not None:
        _i32(dst_ids, "dst_ids")
    n = src_ids.shape[0]
    if out is None:
        out = XferList(n, src_ids.device, max_run_blocks)
    _check("kv_build_xfer_list_static", load().kv_build_xfer_list_static(
        _ptr(req_offsets), req_offsets.shape[0] - 1, _ptr(src_ids), _ptr(dst_ids), n, int(max_run_blocks),
        _ptr(out.runs), out.capacity, _ptr(out.n_runs), _stream(stream)))
    out.max_run_blocks = int(max_run_blocks)
    return out


def kv_pack_blocks(cache: PagedCache, xfer: XferList, n_blocks: int, stage: Optional[torch.Tensor] = None,
                   slice_off: int = 0, slice_bytes: Optional[int] = None, stream=None) -> torch.Tensor:
    sb = cache.row_bytes if slice_bytes is None else int(slice_bytes)
    sd = stage_desc(n_blocks, len(cache.tensors), cache.n_planes, cache.block_size, sb)
    if stage is None:
        stage = torch.empty(stage_nbytes(sd), dtype=torch.uint8, device=xfer.runs.device)
    d = cache.desc()
    _check("kv_pack_blocks", load().kv_pack_blocks(
        ctypes.byref(d), int(slice_off), ctypes.byref(sd), _ptr(xfer.runs), _ptr(xfer.n_runs), xfer.capacity,
        xfer.max_run_blocks, _stage_ptr(stage), stage.numel() * stage.element_size(), _stream(stream)))
    return stage


def kv_unpack_blocks(cache: PagedCache, stage: torch.Tensor, xfer: XferList, n_blocks: int, src_block_size: int,
                     slice_bytes: Optional[int] = None, dst_slice_off: int = 0,
                     src_req_offsets: Optional[torch.Tensor] = None, dst_req_offsets: Optional[torch.Tensor] = None,
                     dst_ids: Optional[torch.Tensor] = None, stream=None, signal: Optional[torch.Tensor] = None,
                     signal_add: int = 1):
    """Whole-block mode when dst_ids is None (runs carry destination ids), remap mode otherwise.
    With `signal` (see new_signal) the call is kv_unpack_blocks_signal: signal value += signal_add
    once every row has landed."""
    sb = cache.row_bytes if slice_bytes is None else int(slice_bytes)
    sd = stage_desc(n_blocks, len(cache.tensors), cache.n_planes, src_block_size, sb)
    n_reqs = 0 if dst_req_offsets is None else dst_req_offsets.shape[0] - 1
    d = cache.desc()
    args = [ctypes.byref(d), int(dst_slice_off), ctypes.byref(sd), _ptr(xfer.runs), _ptr(xfer.n_runs), xfer.capacity,
            xfer.max_run_blocks, _stage_ptr(stage), stage.numel() * stage.element_size(), _ptr(src_req_offsets),
            _ptr(dst_req_offsets), _ptr(dst_ids), n_reqs]
    if signal is None:
        _check("kv_unpack_blocks", load().kv_unpack_blocks(*args, _stream(stream)))
    else:
        _check("kv_unpack_blocks_signal", load().kv_unpack_blocks_signal(*args, _ptr(signal), int(signal_add),
                                                                         _stream(stream)))


def new_signal(device="cuda") -> torch.Tensor:
    """A zeroed kv_signal (16 bytes: value int64, arrived + reserved) in device memory."""
    return torch.zeros(2, dtype=torch.int64, device=device)


def signal_value(signal: torch.Tensor) -> int:
    return int(signal[0].item())


def kv_wait_signal(signal: torch.Tensor, expected: int, timeout_us: int, status: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """Queue a bounded device-side wait until signal value >= expected; returns the device status word."""
    if status is None:
        status = torch.full((1,), -1, dtype=torch.int32, device=signal.device)
    _check("kv_wait_signal", load().kv_wait_signal(_ptr(signal), int(expected), int(timeout_us), _ptr(status),
                                                   _stream(stream)))
    return status


def kv_get_last_error(clear: bool = True, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("kv_get_last_error", load().kv_get_last_error(ctypes.byref(out), 1 if clear else 0, _stream(stream)))
    return out.value


def default_max_run_blocks(stage_block_bytes: int, target_bytes: int = 16 * 1024) -> int:
    """A run cap that keeps one run at or under target_bytes per tensor (at least one block).

    16 KiB is the piece a copy kernel hands to one warp, so a capped run is never split."""
    return max(1, int(target_bytes) // max(1, int(stage_block_bytes)))
