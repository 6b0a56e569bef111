"""Build libqsa.so (the C ABI plus its sm_103a kernels) in-tree with nvcc.

Each translation unit is compiled in parallel for exactly one target,
sm_103a, then linked into a shared library next to this file.  The CUDA
runtime is linked statically, so the library needs only the driver at run
time.  Usage:  python -m sparse_selected_attention_gb300.build [-v] [--all]

Besides the release library there are test variants of the same sources,
built by build_all():
  libqsa_wait0.so  every bounded pipeline wait gives up at once
                   (QSA_WAIT_LIMIT=0), so a test can watch the time-out path
                   set its error bit and stop cleanly;
  libqsa_check.so  device-side index checks (QSA_CHECK=1): an index outside
                   its buffer sets a device word (read by qsa_check_word)
                   and the access is skipped.
and libqsa_l2probe.so, the benchmark's L2 gather-rate probe.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqsa.so")
# variant -> (extra defines, library file)
VARIANTS = {
    "release": ([], "libqsa.so"),
    "wait0": (["-DQSA_WAIT_LIMIT=0"], "libqsa_wait0.so"),
    "check": (["-DQSA_CHECK=1"], "libqsa_check.so"),
}
SOURCES = ["api.cpp", "prep.cu", "score.cu", "select.cu", "attn.cu", "ids.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def lib_path(variant: str = "release") -> str:
    return os.path.join(PKG, VARIANTS[variant][1])


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False, variant: str = "release") -> str:
    """Compile and link one variant; returns the library path.  Rebuilds only
    stale parts."""
    defines, libname = VARIANTS[variant]
    bdir = BUILD if variant == "release" else os.path.join(BUILD, variant)
    lib = os.path.join(PKG, libname)
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(INCLUDE, "qsa.h")] + [
        os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            extra = ["-Xptxas", "-v"] if (ptxas_info and src.endswith(".cu")) else []
            jobs.append([cc, *ARCH, *FLAGS, *defines, *extra, "-c", s, "-o", o])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda c: _run(c, verbose), jobs))
    if ptxas_info:
        for r in results:
            sys.stdout.write(r.stderr)
    if force or jobs or _stale(lib, objs):
        tmp = lib + ".tmp"
        _run([cc, *ARCH, "-shared", "-o", tmp, *objs], verbose)
        os.replace(tmp, lib)
    return lib


def build_host_sanitized(verbose: bool = False) -> str:
    """libqsa_asan.so: the release kernels with the host side (api.cpp, the
    argument validation) compiled by g++ under AddressSanitizer and
    UndefinedBehaviorSanitizer.  For the CPU tests only; load it with the
    sanitizer runtimes preloaded (tests/test_sanitizers_cpu.py)."""
    build(verbose=verbose)
    bdir = os.path.join(BUILD, "asan")
    os.makedirs(bdir, exist_ok=True)
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    gxx = shutil.which("g++")
    if not gxx:
        raise RuntimeError("g++ not found")
    san = ["-fsanitize=address,undefined", "-fno-omit-frame-pointer", "-fno-sanitize-recover=undefined"]
    api_o = os.path.join(bdir, "api.cpp.o")
    _run([gxx, "-O1", "-g", "-std=c++17", "-fPIC", *san, "-I", INCLUDE, "-I", CSRC,
          "-I", os.path.join(cuda_home, "include"), "-c", os.path.join(CSRC, "api.cpp"), "-o", api_o], verbose)
    objs = [os.path.join(BUILD, src + ".o") for src in SOURCES if src != "api.cpp"]
    lib = os.path.join(PKG, "libqsa_asan.so")
    _run([gxx, "-shared", *san, "-o", lib, api_o, *objs, "-L", os.path.join(cuda_home, "lib64"),
          "-lcudart_static", "-ldl", "-lrt", "-lpthread"], verbose)
    return lib


PROBE_LIB = os.path.join(PKG, "libqsa_l2probe.so")


def build_probe(verbose: bool = False, force: bool = False) -> str:
    """libqsa_l2probe.so: the L2 gather-rate probe that the benchmark uses as
    the attention's L2 roofline (not part of the attention path)."""
    src = os.path.join(CSRC, "l2probe.cu")
    if force or _stale(PROBE_LIB, [src]):
        tmp = PROBE_LIB + ".tmp"
        _run([nvcc(), *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", src, "-o", tmp], verbose)
        os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


def build_all(verbose: bool = False, force: bool = False) -> list:
    """Every variant (release first), the variants and the probe in parallel."""
    out = [build(verbose=verbose, force=force)]
    rest = [v for v in VARIANTS if v != "release"]
    with ThreadPoolExecutor(max_workers=len(rest) + 1) as ex:
        futs = [ex.submit(build, verbose=verbose, force=force, variant=v) for v in rest]
        probe = ex.submit(build_probe, verbose=verbose, force=force)
        out += [f.result() for f in futs] + [probe.result()]
    return out


if __name__ == "__main__":
    v = "-v" in sys.argv
    if "--all" in sys.argv:
        print("\n".join(build_all(verbose=v, force="--force" in sys.argv)))
    else:
        print(build(verbose=v, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv))
