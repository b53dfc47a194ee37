"""Build libls_sampler.so in-tree with nvcc for sm_103a.

    python -m logits_sampling_gb300.build [--force]

Compiles logits_sampling_gb300/csrc/*.cu into logits_sampling_gb300/libls_sampler.so
(-gencode arch=compute_103a,code=sm_103a, -O3, -lineinfo, no fast-math).  The
build is skipped when the library is newer than every source and header.

VARIANTS holds test-only builds of the same sources with other compile-time
constants (never loaded by the package itself): ``reselect`` puts the top-p
candidate bound above every cut, so every top-p row takes the re-select over
all of its entries -- the path that otherwise runs only when rounding beats
the bound's slack.
"""
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libls_sampler.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
VARIANTS = {"reselect": ["-DLS_TOPP_SLACK=-64.0f"]}


def variant_path(name):
    return os.path.join(PKG, f"libls_sampler_{name}.so")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libls_sampler.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + sorted(
        glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force=False, verbose=False, variant=None):
    """Compile the shared library (or a test-only variant of VARIANTS);
    returns its path.  Each translation unit (one per kernel mode and cluster
    size, plus the C ABI) compiles in its own nvcc process, in parallel; the
    objects are then linked."""
    lib = LIB if variant is None else variant_path(variant)
    extra = [] if variant is None else VARIANTS[variant]
    if not force and up_to_date(lib):
        return lib
    tag = f".{variant or 'main'}.tmp{os.getpid()}"
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(PKG, os.path.basename(src)[:-3] + tag + ".o")
        cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", *extra,
               "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd))
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    failed = [p.args[-3] for p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, "nvcc", f"compiling {failed} failed")
        tmp = lib + tag
        subprocess.run([_nvcc(), *ARCH_FLAGS, "-shared", *objs, "-o", tmp, "-lcudart"], check=True)
        os.replace(tmp, lib)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return lib



if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
    if "--variants" in sys.argv:
        for name in VARIANTS:
            print(build(force="--force" in sys.argv, variant=name))
