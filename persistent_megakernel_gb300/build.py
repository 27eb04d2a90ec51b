"""Build ``libdec.so`` in-tree: the megakernel (nvcc, sm_103a) plus the host runtime and packer.

Three translation units compiled in parallel, then linked with nvcc. No CMake. Rebuilds
only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libdec.so")
BUILD_DIR = os.path.join(HERE, "_build")
# "trace": the self-timing variant (-DDEC_TRACE), a separate library next to the default one
VARIANTS = {"": [], "trace": ["-DDEC_TRACE"]}


def lib_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(HERE, f"libdec_{variant}.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdec.so")
    return cand


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(INCLUDE, "dec.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def sources_sha256() -> str:
    """sha256 over every source and header the library is built from, in a fixed order."""
    sha = hashlib.sha256()
    for p in sorted(sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))) + [
            os.path.join(INCLUDE, "dec.h")]:
        sha.update(os.path.basename(p).encode())
        sha.update(open(p, "rb").read())
    return sha.hexdigest()


def _log(msg: str) -> None:
    # stderr: a bench prints its one result line on stdout
    sys.stderr.write(f"[libdec build] {msg}\n")
    sys.stderr.flush()


def build(force: bool = False, verbose: bool = False, extra_nvcc=(), variant: str = "", defines=()) -> str:
    """Build libdec.so (or libdec_<variant>.so with the variant's -D flags plus `defines`).
    Prints one line saying whether it compiled from source or found the library up to date,
    with the sha256 of the sources."""
    lib = lib_path(variant)
    if not force and not _stale(lib):
        _log(f"{os.path.basename(lib)} up to date (sources sha256 {sources_sha256()[:16]}), not recompiled")
        return lib
    defs = VARIANTS.get(variant, []) + list(defines)
    nvcc = _nvcc()
    cuda = _cuda_home(nvcc)
    bdir = os.path.join(BUILD_DIR, variant or "default")
    os.makedirs(bdir, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, *defs,
                   "-Xptxas", "-v" if verbose else "-O3", *extra_nvcc, "-c", src, "-o", obj]
        else:
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-fopenmp", "-I", INCLUDE, "-I", os.path.join(cuda, "include"), *defs,
                   "-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("building libdec.so failed:\n" + msg)
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart", "-lgomp"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("linking libdec.so failed:\n" + r.stdout)
    os.replace(tmp, lib)
    _log(f"{os.path.basename(lib)} compiled from source: {len(objs)} translation units, sources sha256 "
         f"{sources_sha256()[:16]}, nvcc {' '.join(ARCH)} -O3 {' '.join(defs)}".rstrip())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="trace" if "--trace" in sys.argv else ""))
