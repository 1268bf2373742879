"""Builds libcsmkv.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libcsmkv.so")
OBJ_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]
_lock = threading.Lock()


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsmkv.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "csmkv.h"), os.path.abspath(__file__)]


def is_stale() -> bool:
    if not os.path.exists(OUT):
        return True
    t = os.path.getmtime(OUT)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel and link the shared library."""
    with _lock:
        if not force and not is_stale():
            return OUT
        nvcc = _nvcc()
        os.makedirs(OBJ_DIR, exist_ok=True)
        procs, objs = [], []
        for src in _sources():
            obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
            objs.append(obj)
            cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        errors = []
        for cmd, pr in procs:
            out, _ = pr.communicate()
            if pr.returncode != 0:
                errors.append(" ".join(cmd) + "\n" + out.decode(errors="replace"))
            elif verbose and out:
                print(out.decode(errors="replace"))
        if errors:
            raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
        libdir = os.path.realpath(os.path.join(os.path.dirname(nvcc), "..", "lib64"))
        tmp = OUT + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-Xlinker", f"-rpath,{libdir}"]
        res = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + res.stdout.decode(errors="replace"))
        os.replace(tmp, OUT)
        return OUT
