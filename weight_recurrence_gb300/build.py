"""Builds liblinattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu translation unit compiles in parallel to an object under
``weight_recurrence_gb300/_build/``; one nvcc link makes
``weight_recurrence_gb300/lib/liblinattn.so`` with the CUDA runtime linked
statically, so the library depends on nothing but the driver.  The checked
variant (``--checked``) compiles the same sources with ``-DLA_CHECKED`` into
``_build_checked/`` and ``lib/liblinattn_checked.so``.

    python -m weight_recurrence_gb300.build [--force] [--verbose] [--checked]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
# release: the product library; checked: the same sources with -DLA_CHECKED,
# whose kernels test their computed indices against the buffers' extents and
# record LA_ERR_BOUNDS instead of making an access out of range
VARIANTS = {
    "release": ("_build", "liblinattn.so", []),
    "checked": ("_build_checked", "liblinattn_checked.so", ["-DLA_CHECKED"]),
}
BUILD = os.path.join(PKG, VARIANTS["release"][0])
LIB = os.path.join(LIBDIR, VARIANTS["release"][1])
LIB_CHECKED = os.path.join(LIBDIR, VARIANTS["checked"][1])


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblinattn.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    inc = os.path.join(os.path.dirname(PKG), "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_variants(variants=("release",), force: bool = False, verbose: bool = False, extra_flags=()):
    """Compile (incrementally) every translation unit of the given variants at
    once, in parallel, then link each library; returns the library paths."""
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    hdrs = headers()
    plan, procs = [], []
    for name in variants:
        bdir, libname, vflags = VARIANTS[name]
        bdir = os.path.join(PKG, bdir)
        os.makedirs(bdir, exist_ok=True)
        objs, started = [], 0
        for src in sources():
            obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            if force or _stale(obj, [src] + hdrs):
                cmd = [cc, *ARCH, *NVCC_FLAGS, *vflags, *extra_flags, "-c", src, "-o", obj]
                if verbose:
                    print(" ".join(cmd), flush=True)
                procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
                started += 1
        plan.append((os.path.join(LIBDIR, libname), objs, started))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0 or verbose:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    for lib, objs, started in plan:
        if force or started or _stale(lib, objs):
            tmp = lib + ".tmp%d" % os.getpid()
            cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.check_call(cmd)
            os.replace(tmp, lib)
    return [lib for lib, _, _ in plan]


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile (incrementally) and link one variant; returns the library path."""
    return build_variants(("checked" if checked else "release",), force, verbose, extra_flags)[0]


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true", help="also build liblinattn_checked.so")
    a = ap.parse_args()
    names = ("release", "checked") if a.checked else ("release",)
    for path in build_variants(names, force=a.force, verbose=a.verbose):
        print(path)
