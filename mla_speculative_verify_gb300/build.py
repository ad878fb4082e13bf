"""Build the sm_103a library libmla_verify_sm103.so in-tree (nvcc + g++, no cmake).

The CUDA translation unit and the host-only sources compile in parallel; the
result lands in ``mla_speculative_verify_gb300/_lib/`` (git-ignored).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libmla_verify_sm103.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

CUDA_SOURCES = ["kernel_sm103.cu", "kernel_pair_sm103.cu", "static_workspace.cu"]
HOST_SOURCES = ["plan.cpp", "status.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the sm_103a library cannot be built")


def _sources_newer_than(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return any(os.path.getmtime(f) > t for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source changed; return its path."""
    if not force and not _sources_newer_than(LIB_PATH):
        return LIB_PATH
    nvcc = _nvcc()
    cuda_home = os.path.dirname(os.path.dirname(nvcc))
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, f"obj{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda_home, "include")]
    procs, objs = [], []
    for src in CUDA_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v", *inc, "-c",
               os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    for src in HOST_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", *inc, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose and out:
            sys.stderr.write(out)
        if pr.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("building the sm_103a library failed:\n" + msg)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("linking the sm_103a library failed:\n" + r.stdout)
    os.replace(tmp, LIB_PATH)
    shutil.rmtree(obj_dir, ignore_errors=True)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
