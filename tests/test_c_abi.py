"""The C ABI used from plain C: tests/c_abi_check.c includes only
include/pagedkv.h, links libpagedkv.so and runs its host-side calls (the
block allocator, the split-size queries, the argument checks).  No device is
needed."""

import os
import shutil
import subprocess

import pytest

from paged_kv_cache_247_gb300 import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_caller(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(_build.LIB)
    exe = str(tmp_path / "c_abi_check")
    cmd = [cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c_abi_check.c"), "-L", libdir, "-lpagedkv",
           f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "c abi ok"
