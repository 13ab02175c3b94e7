"""The C ABI driven from a plain C11 program (no Python, no torch): compile it against
include/pagedkv.h, link libpagedkv.so, run it on the GPU."""
from __future__ import annotations

import os
import subprocess

import pytest
import torch

from paged_kv_cache_81_gb300 import build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_c_program_drives_the_path(tmp_path):
    lib = build.build()
    cuda = os.path.dirname(os.path.dirname(build.nvcc()))
    exe = tmp_path / "abi_example"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-O1", "-I", build.INCLUDE, "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "c", "abi_example.c"), "-o", str(exe), "-L", libdir, "-l:libpagedkv.so",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}",
           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.startswith("c abi ok")
