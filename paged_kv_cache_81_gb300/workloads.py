"""Seeded synthetic inputs for the paged KV-cache data path.

This module holds the five workload presets and the generators of their inputs:
request lengths, fragmented free queues, block tables, token positions and cache
contents.  It computes nothing of the method itself (no slot arithmetic, no
gather, no scatter, no run detection): the CUDA path's tests, the benchmark and
the CPU oracle all take its arrays as plain inputs.

Sources for the shapes (vLLM PD-disaggregation pages):
  * "vllm v1 调度逻辑 和 distributed 分布式原理" drawing, "Paged kv cache": a block
    holds token slots 0..15 (block_size 16); the per-layer tensor panel: 48 layer
    tensors of 147456 blocks, 1.125 GB each, one block_table shared by every
    layer; "scheduler(step)": 8 prompts of "8k" take 576 x 8 blocks; the two
    layer shapes (num_blocks, 2, bs, H, D) and (2, num_blocks, bs, H, D).
  * The free_block_queue drawing (blocks B3, B7, B8, B9 returned with
    ref_count 0, new blocks taken with popleft) motivates the fragmented queue.
Every generator is seeded; the seed of preset k is 81 + k.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

LAYOUTS = ("separate", "blocks_first", "kv_first", "mla")


@dataclass(frozen=True)
class CacheGeom:
    """Shape of one paged cache.

    layout:
      "separate"     one K and one V tensor per layer, each [num_blocks, bs, H, D]
      "blocks_first" one tensor per layer, [num_blocks, 2, bs, H, D] (K plane, V plane)
      "kv_first"     one tensor per layer, [2, num_blocks, bs, H, D]
      "mla"          one latent tensor per layer, [num_blocks, bs, D] (H = 1)
    """

    layout: str
    num_blocks: int
    block_size: int
    heads: int
    head_dim: int
    elt_bytes: int = 2  # bf16

    def __post_init__(self):
        assert self.layout in LAYOUTS, self.layout

    @property
    def row_bytes(self) -> int:
        return self.heads * self.head_dim * self.elt_bytes

    @property
    def n_planes(self) -> int:
        return 2 if self.layout in ("blocks_first", "kv_first") else 1

    @property
    def tensors_per_layer(self) -> int:
        return 2 if self.layout == "separate" else 1

    @property
    def block_payload_bytes(self) -> int:
        """Bytes of one block of one tensor (all planes)."""
        return self.n_planes * self.block_size * self.row_bytes

    @property
    def tensor_bytes(self) -> int:
        return self.num_blocks * self.block_payload_bytes

    def tensor_shape(self) -> tuple:
        nb, bs, h, d = self.num_blocks, self.block_size, self.heads, self.head_dim
        return {
            "separate": (nb, bs, h, d),
            "blocks_first": (nb, 2, bs, h, d),
            "kv_first": (2, nb, bs, h, d),
            "mla": (nb, bs, h * d),
        }[self.layout]

    def byte_strides(self) -> dict:
        """Byte distance between consecutive blocks, planes and token slots."""
        row, bs, nb = self.row_bytes, self.block_size, self.num_blocks
        if self.layout == "blocks_first":
            return dict(block_stride=2 * bs * row, plane_stride=bs * row, token_stride=row)
        if self.layout == "kv_first":
            return dict(block_stride=bs * row, plane_stride=nb * bs * row, token_stride=row)
        # separate / mla: a single plane per tensor
        return dict(block_stride=bs * row, plane_stride=bs * row, token_stride=row)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int  # preset index; seed = 81 + index
    kind: str  # generator family: tiny | mid | page | mla | asym
    n_layers: int
    src: CacheGeom
    dst: CacheGeom
    slice_off: int = 0  # byte offset of the moved slice inside a source row
    slice_bytes: int = 0  # 0 = the whole row
    dst_slice_off: int = 0  # byte offset where the slice lands in a destination row
    spec: tuple = field(default=())  # family parameters as (key, value) pairs

    @property
    def seed(self) -> int:
        return 81 + self.index

    @property
    def n_tensors(self) -> int:
        return self.n_layers * self.src.tensors_per_layer

    @property
    def moved_slice(self) -> int:
        return self.slice_bytes or self.src.row_bytes

    @property
    def equal_geometry(self) -> bool:
        """True when a staged block maps onto exactly one destination block."""
        return (self.src.block_size == self.dst.block_size
                and self.moved_slice == self.dst.row_bytes
                and self.src.n_planes == self.dst.n_planes)

    def p(self, key, default=None):
        return dict(self.spec).get(key, default)

    def with_spec(self, **kw) -> "Workload":
        d = dict(self.spec)
        d.update(kw)
        return replace(self, spec=tuple(sorted(d.items())))


def _spec(**kw) -> tuple:
    return tuple(sorted(kw.items()))


# --- the five presets ------------------------------------------------------
TINY = Workload(
    "tiny", 0, "tiny", n_layers=2,
    src=CacheGeom("separate", 64, 16, 2, 64), dst=CacheGeom("separate", 64, 16, 2, 64),
    spec=_spec(n_reqs=3, len_lo=1, len_hi=100, new_tokens=8))

MID = Workload(
    "mid", 1, "mid", n_layers=32,
    src=CacheGeom("separate", 16384, 16, 8, 128), dst=CacheGeom("separate", 16384, 16, 8, 128),
    spec=_spec(n_reqs=16, blocks_per_req=128, max_piece=32, keep_prob=0.5))

PAGE = Workload(
    "page_shaped", 2, "page", n_layers=48,
    src=CacheGeom("blocks_first", 147456, 16, 1, 128),
    dst=CacheGeom("blocks_first", 147456, 16, 1, 128),
    spec=_spec(n_reqs=8, blocks_per_req=576))

MLA = Workload(
    "mla", 3, "mla", n_layers=61,
    src=CacheGeom("mla", 8192, 64, 1, 576), dst=CacheGeom("mla", 8192, 64, 1, 576),
    spec=_spec(decode_reqs=256, max_pos=32767, n_reqs=32, len_lo=1024, len_hi=32768,
               max_piece=8, table_blocks=512))

ASYM = Workload(
    "asym_remap", 4, "asym", n_layers=40,
    src=CacheGeom("separate", 32768, 16, 8, 128), dst=CacheGeom("separate", 8192, 64, 4, 128),
    slice_off=4 * 128 * 2, slice_bytes=4 * 128 * 2, dst_slice_off=0,
    spec=_spec(n_reqs=24, len_lo=512, len_hi=8192))

# The page-shaped cache in the other layer layout of the drawing, (2, num_blocks, bs, H, D)
# (FlashAttention's kv-first tensors); same seed, so the same block lists as PAGE.
PAGE_KV_FIRST = replace(PAGE, name="page_shaped_kv_first",
                        src=CacheGeom("kv_first", 147456, 16, 1, 128), dst=CacheGeom("kv_first", 147456, 16, 1, 128))

PRESETS = {w.name: w for w in (TINY, MID, PAGE, MLA, ASYM, PAGE_KV_FIRST)}


def small(wl: Workload) -> Workload:
    """A reduced copy of a preset: same structure, sizes the oracle finishes in seconds.

    The reduced cases still span many copy items and builder tiles and keep the
    ragged last blocks of the full preset.
    """
    if wl.kind == "tiny":
        return wl
    if wl.kind == "mid":
        g = replace(wl.src, num_blocks=2048)
        return replace(wl, name=wl.name + "_small", n_layers=2, src=g, dst=g).with_spec(n_reqs=5, blocks_per_req=96)
    if wl.kind == "page":
        g = replace(wl.src, num_blocks=4096)
        return replace(wl, name=wl.name + "_small", n_layers=3, src=g, dst=g).with_spec(n_reqs=3)
    if wl.kind == "mla":
        g = replace(wl.src, num_blocks=1024)
        return replace(wl, name=wl.name + "_small", n_layers=3, src=g, dst=g).with_spec(
            decode_reqs=64, n_reqs=4, len_lo=1024, len_hi=8192, max_pos=8191, table_blocks=128)
    if wl.kind == "asym":
        return replace(wl, name=wl.name + "_small", n_layers=2,
                       src=replace(wl.src, num_blocks=4096),
                       dst=replace(wl.dst, num_blocks=1024)).with_spec(n_reqs=5)
    raise ValueError(wl.kind)


# --- generated instances ---------------------------------------------------
@dataclass
class Case:
    """One generated instance of a workload (host numpy arrays)."""

    wl: Workload
    # transfer lists: CSR over requests
    req_offsets: np.ndarray  # int32 [R+1]
    src_ids: np.ndarray  # int32 [N]
    dst_req_offsets: np.ndarray  # int32 [R+1]
    dst_ids: np.ndarray  # int32 [Nd]
    # new-token write (slot_mapping + reshape_and_cache); T may be 0
    block_table: Optional[np.ndarray] = None  # int32 [Rw, M]
    token_req: Optional[np.ndarray] = None  # int32 [T]
    token_pos: Optional[np.ndarray] = None  # int32 [T]
    req_tokens: Optional[np.ndarray] = None  # int32 [R]: tokens each transferred request holds
    info: dict = field(default_factory=dict)

    @property
    def n_blocks(self) -> int:
        return int(self.src_ids.shape[0])

    @property
    def n_reqs(self) -> int:
        return int(self.req_offsets.shape[0] - 1)

    @property
    def n_tokens(self) -> int:
        return 0 if self.token_req is None else int(self.token_req.shape[0])


def csr(lists) -> tuple:
    """Concatenate per-request id lists into (offsets int32 [R+1], ids int32 [N])."""
    off = np.zeros(len(lists) + 1, dtype=np.int64)
    for i, l in enumerate(lists):
        off[i + 1] = off[i] + len(l)
    ids = np.concatenate([np.asarray(l, dtype=np.int64) for l in lists]) if lists else np.zeros(0, np.int64)
    return off.astype(np.int32), ids.astype(np.int32)


def fragmented_queue(rng: np.random.Generator, num_blocks: int, max_piece: int, keep_prob: float) -> np.ndarray:
    """A free-block queue whose order mixes kept contiguous pieces and scattered singletons.

    The ids 0..num_blocks-1 are cut, in order, into pieces of length U{1..max_piece}.
    Each piece stays an in-order unit with probability keep_prob; otherwise its ids
    become singleton units.  The units are shuffled and concatenated.
    """
    units = []
    start = 0
    while start < num_blocks:
        ln = int(rng.integers(1, max_piece + 1))
        piece = np.arange(start, min(start + ln, num_blocks), dtype=np.int64)
        start += ln
        if rng.random() < keep_prob:
            units.append(piece)
        else:
            units.extend(piece[i:i + 1] for i in range(piece.shape[0]))
    order = rng.permutation(len(units))
    return np.concatenate([units[i] for i in order]).astype(np.int32)


def pop_lists(queue: np.ndarray, counts, wrap: bool = False) -> list:
    """Pop consecutive id lists of the given lengths from the front of a queue."""
    out, pos = [], 0
    total = int(sum(counts))
    if wrap and total > queue.shape[0]:
        queue = np.tile(queue, -(-total // queue.shape[0]))
    assert total <= queue.shape[0], "queue too short"
    for c in counts:
        out.append(queue[pos:pos + c])
        pos += c
    return out


def blocks_for(tokens: int, block_size: int) -> int:
    """Blocks a request of `tokens` tokens occupies (the allocator's ceiling)."""
    return -(-int(tokens) // int(block_size))


def make_case(wl: Workload) -> Case:
    rng = np.random.default_rng(wl.seed)
    return {"tiny": _tiny, "mid": _mid, "page": _page, "mla": _mla, "asym": _asym}[wl.kind](wl, rng)


def _table(lists, width=None) -> np.ndarray:
    width = width or max(len(l) for l in lists)
    t = np.full((len(lists), width), -1, dtype=np.int32)
    for r, l in enumerate(lists):
        t[r, :len(l)] = l
    return t


def _tiny(wl, rng):
    nb, bs = wl.src.num_blocks, wl.src.block_size
    n, new = wl.p("n_reqs"), wl.p("new_tokens")
    lens = rng.integers(wl.p("len_lo"), wl.p("len_hi") + 1, size=n)
    perm = rng.permutation(nb)
    counts = [blocks_for(l + new, bs) for l in lens]
    src_lists = pop_lists(perm, counts)
    dst_lists = pop_lists(rng.permutation(wl.dst.num_blocks), counts)
    off, ids = csr(src_lists)
    doff, dids = csr(dst_lists)
    token_req = np.repeat(np.arange(n, dtype=np.int32), new)
    token_pos = np.concatenate([np.arange(l, l + new, dtype=np.int32) for l in lens])
    return Case(wl, off, ids, doff, dids, _table(src_lists), token_req, token_pos,
                req_tokens=(lens + new).astype(np.int32), info=dict(lens=lens.tolist()))


def _mid(wl, rng):
    nb = wl.src.num_blocks
    n, per = wl.p("n_reqs"), wl.p("blocks_per_req")
    q_src = fragmented_queue(rng, nb, wl.p("max_piece"), wl.p("keep_prob"))
    q_dst = fragmented_queue(rng, wl.dst.num_blocks, wl.p("max_piece"), wl.p("keep_prob"))
    off, ids = csr(pop_lists(q_src, [per] * n))
    doff, dids = csr(pop_lists(q_dst, [per] * n))
    return Case(wl, off, ids, doff, dids, req_tokens=np.full(n, per * wl.src.block_size, np.int32))


def _page(wl, rng):
    nb, bs = wl.src.num_blocks, wl.src.block_size
    n, per = wl.p("n_reqs"), wl.p("blocks_per_req")
    src = rng.choice(nb, size=n * per, replace=False).astype(np.int32)
    dst = rng.choice(wl.dst.num_blocks, size=n * per, replace=False).astype(np.int32)
    src_lists = [src[r * per:(r + 1) * per] for r in range(n)]
    off, ids = csr(src_lists)
    doff, dids = csr([dst[r * per:(r + 1) * per] for r in range(n)])
    # prefill of every prompt: positions 0 .. per*bs-1 (9216 tokens for 576 blocks)
    tok = per * bs
    token_req = np.repeat(np.arange(n, dtype=np.int32), tok)
    token_pos = np.tile(np.arange(tok, dtype=np.int32), n)
    return Case(wl, off, ids, doff, dids, _table(src_lists), token_req, token_pos,
                req_tokens=np.full(n, tok, np.int32))


def _mla(wl, rng):
    nb, bs = wl.src.num_blocks, wl.src.block_size
    # decode step: one new token per request; each request's current block is distinct
    dn, width = wl.p("decode_reqs"), wl.p("table_blocks")
    pos = rng.integers(0, wl.p("max_pos") + 1, size=dn).astype(np.int32)
    table = rng.integers(0, nb, size=(dn, width)).astype(np.int32)
    current = rng.choice(nb, size=dn, replace=False).astype(np.int32)
    table[np.arange(dn), pos // bs] = current  # place each request's current block
    # pack: long requests whose ids come from a queue fragmented into runs 1..max_piece
    n = wl.p("n_reqs")
    lens = rng.integers(wl.p("len_lo"), wl.p("len_hi") + 1, size=n)
    q = fragmented_queue(rng, nb, wl.p("max_piece"), 1.0)
    counts = [blocks_for(l, bs) for l in lens]
    off, ids = csr(pop_lists(q, counts, wrap=True))
    return Case(wl, off, ids, off.copy(), ids.copy(), table,
                np.arange(dn, dtype=np.int32), pos, req_tokens=lens.astype(np.int32), info=dict(lens=lens.tolist()))


def _asym(wl, rng):
    n = wl.p("n_reqs")
    lens = rng.integers(wl.p("len_lo"), wl.p("len_hi") + 1, size=n)
    sc = [blocks_for(l, wl.src.block_size) for l in lens]
    dc = [blocks_for(l, wl.dst.block_size) for l in lens]
    off, ids = csr(pop_lists(rng.permutation(wl.src.num_blocks).astype(np.int32), sc))
    doff, dids = csr(pop_lists(rng.permutation(wl.dst.num_blocks).astype(np.int32), dc))
    return Case(wl, off, ids, doff, dids, req_tokens=lens.astype(np.int32), info=dict(lens=lens.tolist()))


# --- cache and token contents ----------------------------------------------
SPECIAL_BF16 = np.array([0x7FC1, 0xFFFF, 0x7F80, 0xFF80, 0x8000, 0x0001, 0x8003, 0x007F],
                        dtype=np.uint16)  # NaNs, +-inf, -0, subnormals


def normal_bf16_bytes(rng: np.random.Generator, n_elems: int, specials: bool = True) -> np.ndarray:
    """Seeded N(0,1) values as bf16 bit patterns (uint16), with special patterns mixed in.

    bf16 is the upper half of an fp32 word; rounding is to nearest, ties to even.
    """
    f = rng.standard_normal(n_elems, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    if specials and n_elems >= 64:
        k = max(1, n_elems // 64)
        where = rng.choice(n_elems, size=k, replace=False)
        out[where] = SPECIAL_BF16[rng.integers(0, SPECIAL_BF16.shape[0], size=k)]
    return out


def host_cache_tensors(geom: CacheGeom, n_tensors: int, rng: np.random.Generator):
    """n_tensors host arrays (uint16 bf16 patterns) of geom's shape, seeded N(0,1) + specials."""
    shape = geom.tensor_shape()
    n = int(np.prod(shape))
    return [normal_bf16_bytes(rng, n).reshape(shape) for _ in range(n_tensors)]


def fill_random_(t, seed: int):
    """Fill a torch tensor (any device, byte size a multiple of 4) with seeded random bits."""
    import torch

    g = torch.Generator(device=t.device).manual_seed(int(seed))
    t.view(torch.int32).random_(-2 ** 31, 2 ** 31, generator=g)
    return t


# --- device tensors (torch; used by the GPU tests and the benchmark) ---------
def to_device_bf16(arrays, device):
    """Host uint16 bf16-pattern arrays -> torch bf16 tensors on `device` (bit-identical)."""
    import torch

    return [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device) for a in arrays]


def device_cache(geom: CacheGeom, n_tensors: int, device, seed: Optional[int] = None):
    """n_tensors bf16 device tensors of geom's shape, filled with seeded random bits (or left unset)."""
    import torch

    out = []
    for t in range(n_tensors):
        x = torch.empty(geom.tensor_shape(), dtype=torch.bfloat16, device=device)
        if seed is not None:
            fill_random_(x, seed * 1000003 + t)
        out.append(x)
    return out


def new_token_rows(geom: CacheGeom, n_tensors: int, n_tokens: int, device, seed: int):
    """New K/V rows for n_tokens tokens: n_tensors * n_planes views [T, H, D] of one bf16 buffer."""
    import torch

    h, d = (1, geom.heads * geom.head_dim) if geom.layout == "mla" else (geom.heads, geom.head_dim)
    buf = torch.empty((n_tensors * geom.n_planes, n_tokens, h, d), dtype=torch.bfloat16, device=device)
    if n_tokens:
        fill_random_(buf, seed)
    return [buf[k] for k in range(buf.shape[0])]
