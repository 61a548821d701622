"""Build the in-tree CUDA library ``lib/libmrr_v2.so`` for GB300 (sm_103a) with nvcc.

Usage: ``python -m moe_expert_token_gb300.build``.  The library links the CUDA runtime
statically, so it needs only the driver at run time.
"""
from __future__ import annotations

import os
import platform
import shutil
import struct
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("gating_f16.cu", "gating_bf16.cu", "gating_f32.cu", "mrr_v2.cu",
                                            "mrr_v2_noalloc.cu", "mrr_push.cu", "gating.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "gating_kernel.cuh"),
                  os.path.join(CSRC, "ws_layout.h"), os.path.join(CSRC, "mrr_shape.h"),
                  os.path.join(INCLUDE, "mrr_v2.h"), os.path.join(INCLUDE, "mrr_gating.h")]
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libmrr_v2.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]
LINK_FLAGS = ["-shared"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libmrr_v2.so")


_ELF_MACHINE = {"x86_64": 62, "aarch64": 183}


def built_for_this_host(path: str) -> bool:
    """True when the ELF file at ``path`` targets this machine (x86_64 here, aarch64 on Grace)."""
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    want = _ELF_MACHINE.get(platform.machine())
    return want is None or struct.unpack_from("<H", head, 18)[0] == want


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH) or not built_for_this_host(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path.

    Each source compiles to an object in its own nvcc process (in parallel), then one nvcc call
    links the shared library.
    """
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    nvcc = nvcc_path()
    objs, procs = [], []
    try:
        for src in SOURCES:
            obj = os.path.join(LIB_DIR, os.path.splitext(os.path.basename(src))[0] + tag + ".o")
            cmd = [nvcc, *ARCH_FLAGS, *COMPILE_FLAGS, "-I", INCLUDE, "-c", "-o", obj, src]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
                print(" ".join(cmd), file=sys.stderr)
            objs.append(obj)
            procs.append((cmd, subprocess.Popen(cmd)))
        failed = [cmd for cmd, proc in procs if proc.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB_PATH + tag
        subprocess.run([nvcc, *ARCH_FLAGS, *LINK_FLAGS, "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for _, proc in procs:
            if proc.poll() is None:
                proc.kill()
                proc.wait()
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
