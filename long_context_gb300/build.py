"""Build step for the native library ``libcpattn.so`` (sm_103a).

Compiles the CUDA/C++ sources under ``csrc/`` in parallel with nvcc and links
them into ``long_context_gb300/libcpattn.so``.  The CUDA runtime is linked
statically and the driver is reached through the runtime's entry-point query,
so the library loads on a machine without a GPU (the host-only planner can run
there) and needs only the NVIDIA driver on a GPU machine.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcpattn.so")

SOURCES = ["plan.cpp", "api.cu", "schedule.cu", "merge.cu", "attn_fwd.cu", "attn_bwd.cu",
           "dcp.cu", "decode.cu", "noalloc.cu", "ulysses.cu"]
HEADERS = ["kernels.h", "ptx.cuh", "work.cuh", "debug.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required")
    return nvcc


def _flags(verbose_ptxas=False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "cpattn.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def _build_variant(name, define, force):
    lib = os.path.join(PKG, "lib%s.so" % name)
    build()
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(LIB):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags() + ["-D%s=1" % define]

    def compile_one(src):
        obj = os.path.join(BUILD, name + "_" + src + ".o")
        r = subprocess.run([nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stderr)
    os.replace(tmp, lib)
    return lib


def build_fault_injection(force=False):
    """Test-only variant ``libcpattn_fault.so`` built with
    ``-DCPATTN_FAULT_INJECT_DROP_P``: the attention kernel's first CTA skips
    one hand-off so that a bounded device wait runs out.  Used by the failure
    detection test; never loaded by the package."""
    return _build_variant("cpattn_fault", "CPATTN_FAULT_INJECT_DROP_P", force)


def build_debug(force=False):
    """Debug variant ``libcpattn_debug.so`` built with ``-DCPATTN_DEBUG``: the
    attention kernels (forward, backward, schedule) check every global index
    and TMA coordinate they derive and report a violation as
    CPATTN_ERR_DEVICE_BOUNDS in the workspace error word (never a trap).
    Same C ABI as libcpattn.so."""
    return _build_variant("cpattn_debug", "CPATTN_DEBUG", force)


def build(force=False, verbose_ptxas=False, quiet=True):
    """Compile and link ``libcpattn.so`` unless it is up to date."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags(verbose_ptxas)

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if not quiet or verbose_ptxas:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False)
    print(LIB)
