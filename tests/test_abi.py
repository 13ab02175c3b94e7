"""The C ABI on the CPU: the library loads, exports every declared entry point, and
rejects bad host-visible arguments before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from paged_kv_cache_81_gb300 import build
from paged_kv_cache_81_gb300 import pagedkv as K

HEADER = os.path.join(build.INCLUDE, "pagedkv.h")


def declared():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"^KV_API\s+[\w\s\*]+?\b(kv_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return K.load()


def test_header_declares_the_path(lib):
    names = declared()
    for n in ("kv_slot_mapping", "kv_reshape_and_cache", "kv_build_xfer_list", "kv_pack_blocks",
              "kv_unpack_blocks", "kv_get_last_error"):
        assert n in names
    assert set(names) == set(K.EXPORTS)


def test_every_declared_symbol_exported(lib):
    for n in declared():
        assert hasattr(lib, n), n
    assert lib.kv_version().decode().startswith("pagedkv")
    assert lib.kv_status_string(K.KV_ERR_ALIGN).decode() == "KV_ERR_ALIGN"


def test_struct_sizes_match_header(lib):
    assert ctypes.sizeof(K.KvCacheDesc) == 56
    assert ctypes.sizeof(K.KvStageDesc) == 24
    assert K.RUN_WORDS * 4 == 24


def _desc(bases, **kw):
    arr = (ctypes.c_uint64 * len(bases))(*bases)
    d = dict(n_tensors=len(bases), block_size=16, n_planes=2, row_bytes=256, num_blocks=100,
             block_stride=8192, plane_stride=4096, token_stride=256)
    d.update(kw)
    desc = K.KvCacheDesc(d["n_tensors"], d["block_size"], d["n_planes"], d["row_bytes"], d["num_blocks"],
                         d["block_stride"], d["plane_stride"], d["token_stride"],
                         ctypes.cast(arr, ctypes.POINTER(ctypes.c_uint64)))
    desc._keep = arr
    return desc


def _pack(lib, desc, sd, slice_off=0, stage=0x10000, stage_bytes=1 << 40, runs=0x20000, n_runs=0x30000):
    return lib.kv_pack_blocks(ctypes.byref(desc), slice_off, ctypes.byref(sd), ctypes.c_void_p(runs),
                              ctypes.c_void_p(n_runs), 10, 0, ctypes.c_void_p(stage), stage_bytes, None)


def test_host_validation_without_gpu(lib):
    """Each of these returns before any CUDA call, so it runs on a machine without a GPU."""
    sd = K.stage_desc(4, 1, 2, 16, 256)
    assert _pack(lib, _desc([0x1008]), sd) == K.KV_ERR_ALIGN  # base not 16-byte aligned
    assert _pack(lib, _desc([0]), sd) == K.KV_ERR_INVALID_ARG  # null base
    assert _pack(lib, _desc([0x1000], token_stride=200), sd) == K.KV_ERR_ALIGN
    assert _pack(lib, _desc([0x1000], n_planes=3), sd) == K.KV_ERR_INVALID_ARG
    assert _pack(lib, _desc([0x1000]), sd, slice_off=16) == K.KV_ERR_RANGE  # 16 + 256 > row
    assert _pack(lib, _desc([0x1000]), sd, stage_bytes=100) == K.KV_ERR_RANGE  # staging too small
    assert _pack(lib, _desc([0x1000]), sd, stage=0x10008) == K.KV_ERR_ALIGN
    assert _pack(lib, _desc([0x1000]), K.stage_desc(4, 2, 2, 16, 256)) == K.KV_ERR_INVALID_ARG  # tensor count
    assert _pack(lib, _desc([0x1000]), K.stage_desc(4, 1, 2, 8, 256)) == K.KV_ERR_INVALID_ARG  # block size
    assert _pack(lib, _desc([0x1000]), K.stage_desc(4, 1, 2, 16, 24)) == K.KV_ERR_ALIGN  # slice size
    # zero work is a no-op that needs no device
    assert _pack(lib, _desc([0x1000]), K.stage_desc(0, 1, 2, 16, 256)) == K.KV_OK
    # byte counts that do not fit in int64 are refused, not wrapped past the size checks
    assert _pack(lib, _desc([0x1000]), K.stage_desc(1 << 60, 1, 2, 16, 256), stage_bytes=(1 << 63) - 1) == \
        K.KV_ERR_RANGE
    assert _pack(lib, _desc([0x1000], num_blocks=1 << 60), sd) == K.KV_ERR_RANGE
    # unpack: whole-block mode needs equal block sizes; remap mode needs both CSRs
    d = _desc([0x1000])
    bad_bs = K.stage_desc(4, 1, 2, 8, 256)
    assert lib.kv_unpack_blocks(ctypes.byref(d), 0, ctypes.byref(bad_bs), ctypes.c_void_p(0x2000),
                                ctypes.c_void_p(0x3000), 10, 0, ctypes.c_void_p(0x10000), 1 << 40, None, None,
                                None, 0, None) == K.KV_ERR_INVALID_ARG
    assert lib.kv_unpack_blocks(ctypes.byref(d), 0, ctypes.byref(sd), ctypes.c_void_p(0x2000),
                                ctypes.c_void_p(0x3000), 10, 0, ctypes.c_void_p(0x10000), 1 << 40, None, None,
                                ctypes.c_void_p(0x4000), 2, None) == K.KV_ERR_INVALID_ARG
    # slot mapping / builder argument checks
    assert lib.kv_slot_mapping(None, 1, 1, 1, None, None, 0, 16, None, None) == K.KV_OK  # nothing to do
    assert lib.kv_slot_mapping(None, 1, 1, 1, None, None, 5, 0, None, None) == K.KV_ERR_INVALID_ARG
    assert lib.kv_build_xfer_list(None, 1, None, None, 5, 0, None, 5, None, None, 0, None) == K.KV_ERR_INVALID_ARG
    ws = ctypes.c_int64(0)
    assert lib.kv_xfer_workspace_bytes(5000, ctypes.byref(ws)) == K.KV_OK and ws.value == 256 + 3 * 32
    assert lib.kv_reshape_and_cache(ctypes.byref(_desc([0x1000])), None, 256, None, 0, None) == K.KV_OK


def test_fastdiv_exhaustive_small_and_random():
    """The multiply-shift division used by the kernels, compiled for the host."""
    import subprocess
    import tempfile
    src = r'''
#include <cstdio>
#include <cstdint>
#include <random>
#define __host__
#define __device__
#define __forceinline__ inline
struct uint4 { unsigned x, y, z, w; };
#include "kv_common_host_probe.h"
int main() {
    std::mt19937_64 g(1);
    for (uint32_t d = 1; d < 5000; d++) {
        pkv::FastDiv f = pkv::make_fastdiv(d);
        for (uint32_t n = 0; n < 20000; n++) if (pkv::fdiv(n, f) != n / d) { printf("bad %u %u\n", n, d); return 1; }
        for (int k = 0; k < 2000; k++) { uint32_t n = (uint32_t)g(); if (pkv::fdiv(n, f) != n / d) { printf("bad %u %u\n", n, d); return 1; } }
    }
    for (int k = 0; k < 200000; k++) {
        uint32_t d = (uint32_t)(g() % 0x7fffffffu) + 1, n = (uint32_t)g();
        pkv::FastDiv f = pkv::make_fastdiv(d);
        if (pkv::fdiv(n, f) != n / d) { printf("bad %u %u\n", n, d); return 1; }
        if (pkv::fdiv(0xffffffffu, f) != 0xffffffffu / d) { printf("bad max %u\n", d); return 1; }
    }
    puts("ok");
    return 0;
}
'''
    # extract the FastDiv section of the kernel header so the test checks the shipped code
    text = open(os.path.join(build.CSRC, "kv_common.cuh"), encoding="utf-8").read()
    a = text.index("struct FastDiv {")
    b = text.index("// ---", a)
    probe = "#pragma once\nnamespace pkv {\n" + text[a:b] + "}\n"
    with tempfile.TemporaryDirectory() as d:
        open(os.path.join(d, "kv_common_host_probe.h"), "w").write(probe)
        open(os.path.join(d, "t.cpp"), "w").write(src)
        subprocess.run(["g++", "-O2", "-std=c++17", "-I", d, "-o", os.path.join(d, "t"), os.path.join(d, "t.cpp")],
                       check=True)
        r = subprocess.run([os.path.join(d, "t")], capture_output=True, text=True)
        assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout


def test_hash_workspace_size(lib):
    out = ctypes.c_int64(-1)
    assert lib.kv_block_hashes_workspace_bytes(73728, 16, ctypes.byref(out)) == K.KV_OK
    assert out.value == 4608 * (256 * 8 + 4)  # per slot: a 256-entry table of 8-byte sums and a flag
    assert lib.kv_block_hashes_workspace_bytes(48, 16, ctypes.byref(out)) == K.KV_OK
    assert out.value == 3 * 2052 + 4  # rounded up to a multiple of 16
    assert lib.kv_block_hashes_workspace_bytes(15, 16, ctypes.byref(out)) == K.KV_OK and out.value == 0
    assert lib.kv_block_hashes_workspace_bytes(16, 0, ctypes.byref(out)) == K.KV_ERR_INVALID_ARG
    assert lib.kv_block_hashes_workspace_bytes(-1, 16, ctypes.byref(out)) == K.KV_ERR_INVALID_ARG
    assert lib.kv_block_hashes_workspace_bytes(16, 16, None) == K.KV_ERR_INVALID_ARG


def test_header_and_c_example_compile_as_c11():
    """pagedkv.h is a C header: the plain C11 caller (tests/c/abi_example.c) compiles against it with
    every warning an error.  The CUDA runtime header comes from the toolkit next to nvcc."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cuda_include = os.path.join(os.path.dirname(os.path.dirname(build.nvcc())), "include")
    if not os.path.exists(os.path.join(cuda_include, "cuda_runtime.h")):
        pytest.skip("no CUDA runtime header")
    example = os.path.join(os.path.dirname(__file__), "c", "abi_example.c")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I" + build.INCLUDE,
                        "-I" + cuda_include, example], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
