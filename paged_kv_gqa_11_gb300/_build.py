"""Build libpa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Translation units compile in parallel; the CUDA runtime is linked shared so
that the library and PyTorch use one runtime (one current device, one set of
streams) in the same process.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
TYPES = {"f16": 1, "q4_0": 2, "q8_0": 8}  # pa_type numbers
# (source, object name, extra defines): the split-decode kernels are one
# source compiled once per (K, V) format pair.
UNITS = [("pa_pool.cpp", "pa_pool", []), ("pa_append.cu", "pa_append", []), ("pa_decode.cu", "pa_decode", [])]
UNITS += [("pa_decode_kern.cu", f"pa_decode_kern_{k}_{v}", [f"-DPA_KT={TYPES[k]}", f"-DPA_VT={TYPES[v]}"])
          for k in TYPES for v in TYPES]


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pa.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    procs = []
    objs = []
    for src, name, defs in UNITS:
        path = os.path.join(CSRC, src)
        obj = os.path.join(obj_dir, name + ".o")
        objs.append(obj)
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, *defs, "-c", path, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
        else:
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-I", INCLUDE, "-I", os.path.join(cuda, "include"),
                   "-c", path, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out.decode(errors="replace"))
        if p.returncode:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("libpa build failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-Xcompiler", "-fPIC",
            "-Xlinker", "-rpath", "-Xlinker", os.path.join(cuda, "lib64"), *objs, "-o", tmp]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
