"""Compile libciera (the sm_103a kernels and the C ABI) in-tree with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libciera.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libciera_checked.so")
SOURCES = ["ciera_kernels.cu", "ciera_rans.cu", "ciera_api.cpp", "ciera_noalloc.cu"]
HEADERS = [os.path.join(ROOT, "include", "ciera.h"), os.path.join(CSRC, "ciera_internal.h"),
           os.path.join(CSRC, "ciera_device.cuh"), os.path.join(CSRC, "ciera_rans.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libciera cannot be built")


def library_path(checked: bool = False) -> str:
    """The plain library, or the checked build (-DCIERA_CHECKED: global
    accesses at computed offsets tested against their buffers)."""
    return LIB_CHECKED if checked else LIB


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Build ``_build/libciera.so`` (or, with ``checked``,
    ``_build/libciera_checked.so``) if missing or out of date; returns its
    path."""
    lib = library_path(checked)
    if not force and not _stale(lib):
        return lib
    tag = "checked" if checked else "plain"
    obj_dir = os.path.join(OUT_DIR, tag)
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    common = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra_flags]
    if checked:
        common.append("-DCIERA_CHECKED")
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(obj_dir, src.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        procs.append(subprocess.Popen([cc, *common, "-c", os.path.join(CSRC, src), "-o", obj]))
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("nvcc failed while compiling libciera")
    tmp = lib + ".%d.tmp" % os.getpid()
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib
