"""The decode kernels' CTA split, on the host: the kernel's per-CTA walk and
the plan's one-pass walk both equal a brute-force cut of the stated cost rule
(lucebox PR #555, Summary: the context is split across the GPU by occupancy),
and every CTA range holds a tile.  Compiles tests/cut_check.cu with nvcc
against the in-tree library; no GPU needed."""
import os
import shutil
import subprocess

import pytest

from paged_kv_gqa_11_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_weighted_cut_matches_brute_force(tmp_path):
    nvcc = shutil.which("nvcc")
    if nvcc is None:
        pytest.skip("nvcc not on PATH")
    lib = _build.build()
    exe = str(tmp_path / "cut_check")
    cmd = [nvcc, *_build.ARCH, "-std=c++17", "-O2", "-I", _build.INCLUDE, "-I", _build.CSRC,
           os.path.join(HERE, "cut_check.cu"), "-o", exe, "-L", os.path.dirname(lib), "-lpa",
           "-Xlinker", "-rpath", "-Xlinker", os.path.dirname(lib)]
    subprocess.run(cmd, check=True, capture_output=True)
    out = subprocess.run([exe, "1500"], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout, out.stdout
