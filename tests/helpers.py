"""Shared test helpers: golden-file parsing and oracle cache construction."""
from __future__ import annotations

import os

import numpy as np

import oracle
from paged_kv_cache_81_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_path(name):
    return os.path.join(GOLDEN, name)


def read_slot_golden():
    rows = []
    for line in open(golden_path("slot_mapping_examples.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        case, bs, table, pos, want = line.split()
        rows.append((case, int(bs), [int(x) for x in table.split(",")], int(pos), int(want)))
    return rows


def read_xfer_golden():
    cases, cur = [], None
    for line in open(golden_path("xfer_list_examples.txt"), encoding="utf-8"):
        line = line.rstrip("\n")
        s = line.strip()
        if s.startswith("#"):
            continue
        if s.startswith("case "):
            _, name, _, cap = s.split()
            cur = dict(name=name, cap=int(cap), src={}, dst={}, runs=[])
            cases.append(cur)
        elif s.startswith("src ") or s.startswith("dst "):
            kind, rest = s.split(" ", 1)
            r, ids = rest.split(":", 1)
            cur[kind][int(r)] = [int(x) for x in ids.split()]
        elif s.startswith("run "):
            cur["runs"].append([int(x) for x in s.split()[1:]])
    for c in cases:
        n = max(c["src"]) + 1
        c["src_lists"] = [c["src"].get(r, []) for r in range(n)]
        c["dst_lists"] = [c["dst"][r] for r in range(n)] if c["dst"] else None
    return cases


def ora_cache(geom: W.CacheGeom, tensors) -> oracle.Cache:
    st = geom.byte_strides()
    return oracle.Cache(tensors, geom.num_blocks, geom.block_size, geom.n_planes, st["block_stride"],
                        st["plane_stride"], st["token_stride"], geom.row_bytes)


def rows_view(geom: W.CacheGeom, tensor):
    from oracle import brute
    st = geom.byte_strides()
    return brute.rows_view(tensor, geom.num_blocks, geom.n_planes, geom.block_size, st["block_stride"],
                           st["plane_stride"], st["token_stride"], geom.row_bytes)


def req_lists(offsets, ids):
    return [np.asarray(ids[offsets[r]:offsets[r + 1]]) for r in range(len(offsets) - 1)]


def random_cache(geom, n_tensors, seed):
    rng = np.random.default_rng(seed)
    return W.host_cache_tensors(geom, n_tensors, rng)


def random_rows(n_rows, row_bytes, count, seed):
    rng = np.random.default_rng(seed)
    return [rng.integers(0, 256, size=(n_rows, row_bytes), dtype=np.uint8) for _ in range(count)]


def read_clip_golden():
    rows = []
    for line in open(golden_path("sw_clip_examples.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        left, right = line.split(";")
        a = [int(x) for x in left.split()]
        rows.append(dict(bs=a[0], window=a[1], n=a[2], ids=a[3:], want=[int(x) for x in right.split()]))
    return rows


def read_fnv_golden():
    rows = []
    for line in open(golden_path("fnv1a64_vectors.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        data, want = [x.strip() for x in line.split(";")]
        rows.append((b"" if data == "-" else bytes.fromhex(data), int(want, 16)))
    return rows
