"""Builds libdfattn.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process, in parallel, into
``_build/``; the shared library lands next to this file.  ``checked=True``
builds libdfattn_checked.so instead (into ``_build/checked/``): the same
sources compiled with DF_CHECKED, whose tensor-core kernels range-check the
indices of their shared-memory gathers and window copies and report a
failure as DF_ERR_DEVICE_CHECK in the workspace error word.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdfattn.so")
LIB_CHECKED = os.path.join(HERE, "libdfattn_checked.so")
SOURCES = ["df_host.cu", "df_aux.cu", "df_fp32.cu", "df_fwd.cu", "df_bwd.cu", "df_bwd_dq.cu", "df_bwd_dkv.cu", "df_bias.cu", "df_rel.cu", "df_noalloc.cu", "df_pack.cu", "df_proj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return p


def _deps_mtime() -> float:
    m = 0.0
    for d in (CSRC, os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            m = max(m, os.path.getmtime(os.path.join(d, f)))
    return m


def build(force: bool = False, verbose: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compile every CUDA source and link libdfattn.so (libdfattn_checked.so
    with checked=True); returns its path."""
    lib = LIB_CHECKED if checked else LIB
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    extra = list(extra_flags or []) + (["-DDF_CHECKED"] if checked else [])

    def one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcublasLt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
