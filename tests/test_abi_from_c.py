"""The C ABI from C: a C99 program that includes include/ce_rows.h (compiled
as C, not C++) and links the library runs its host-side checks. CPU only."""
import os
import subprocess

import pytest

import row_wise_softmax_ce_gb300 as ce
from row_wise_softmax_ce_gb300 import build as cuda_build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_links_and_runs(tmp_path):
    cuda_build.build()
    exe = os.path.join(tmp_path, "abi_from_c")
    lib_dir = os.path.dirname(ce.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c", "abi_from_c.c"), "-o", exe, "-L", lib_dir, "-lcerows",
           f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi from C: ok" in r.stdout
