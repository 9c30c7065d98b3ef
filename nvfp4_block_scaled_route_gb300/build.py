"""Build libnvfp4moe.so (and its debug-bounds variant) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel, then linked into
one shared library next to this file.  Objects go to csrc/_build/.  A source
newer than the library (or a changed flag set) triggers a rebuild.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(CSRC, "_build")
LIB = os.path.join(PKG, "libnvfp4moe.so")
SOURCES = ["api.cu", "quantize.cu", "route.cu", "reduce.cu", "gemm.cu", "router.cu", "peak.cu",
           "ep.cu"]
HEADERS = ["internal.h", "ptx.cuh", "quant.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stamp() -> str:
    h = hashlib.sha256()
    h.update(repr((ARCH, FLAGS)).encode())
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(ROOT, "include", "nvfp4moe.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def _variant(debug_bounds: bool):
    """(library path, object directory, extra flags) of a build variant: the
    normal library, or libnvfp4moe_debug.so with the in-kernel index checks
    of NVMOE_DEBUG_BOUNDS (a failed check records NVMOE_ERR_DEVICE_BOUNDS in
    the status word and skips the access)."""
    if debug_bounds:
        return (os.path.join(PKG, "libnvfp4moe_debug.so"), os.path.join(CSRC, "_build_debug"),
                ["-DNVMOE_DEBUG_BOUNDS"])
    return LIB, BUILD, []


def build(force: bool = False, verbose: bool = False, extra_flags=(),
          debug_bounds: bool = False, both: bool = False) -> str:
    """Compile (if needed) and return the path of libnvfp4moe.so (or of the
    debug-bounds library).  both: build the two variants, their translation
    units compiled concurrently; returns the normal library's path."""
    variants = [False, True] if both else [debug_bounds]
    jobs = []          # (variant, lib, build dir, stamp, objs, procs)
    cc = None
    for dbg in variants:
        lib, bdir, vflags = _variant(dbg)
        os.makedirs(bdir, exist_ok=True)
        flags = [*vflags, *extra_flags]
        stamp = _stamp() + repr(tuple(flags))
        stamp_file = os.path.join(bdir, "stamp")
        if not force and os.path.exists(lib) and os.path.exists(stamp_file):
            with open(stamp_file) as f:
                if f.read() == stamp:
                    continue
        cc = cc or nvcc()
        objs, procs = [], []
        for name in SOURCES:
            obj = os.path.join(bdir, name.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [cc, *ARCH, *FLAGS, *flags, "-c", os.path.join(CSRC, name), "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((name, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT)))
        jobs.append((lib, stamp_file, stamp, objs, procs))
    for lib, stamp_file, stamp, objs, procs in jobs:
        failed = []
        for name, p in procs:
            out, _ = p.communicate()
            if verbose or p.returncode != 0:
                sys.stderr.write(out.decode(errors="replace"))
            if p.returncode != 0:
                failed.append(name)
        if failed:
            raise RuntimeError(f"nvcc failed for {failed} ({os.path.basename(lib)})")
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            sys.stderr.write(r.stdout.decode(errors="replace"))
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
        with open(stamp_file, "w") as f:
            f.write(stamp)
    return _variant(debug_bounds and not both)[0]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
