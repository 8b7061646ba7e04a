"""Build libdiffattn.so in-tree for sm_103a with nvcc (one process per translation unit).

    python -m differential_attention_gb300.builder [--force] [--verbose] [--ptxas-info] [--debug]

The shared library lands next to this file; objects go to `_build/`. Both are git-ignored.
`--debug` builds libdiffattn_debug.so (objects in `_build_debug/`) with -DDIFFATTN_DEBUG: every
kernel then checks its tile coordinates and gathered or stored rows against their tensors'
extents and reports a failure through diffattn_device_status (a sanitizer substitute; slower).
"""
from __future__ import annotations

import argparse
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
LIB = os.path.join(PKG, "libdiffattn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libdiffattn_debug.so")
SOURCES = ["api.cu", "simt.cu", "decode.cu", "decode_v2_tc.cu", "backward.cu", "host_pipeline.cu", "tmap.cu", "prefill_tc.cu", "prefill_exact.cu", "prefill_v2.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdiffattn.so")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files + [os.path.abspath(__file__)]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
                  debug: bool = False) -> str:
    """Compile every .cu source for sm_103a and link libdiffattn.so (or, with `debug`, the
    bounds-checking libdiffattn_debug.so). Returns the library path."""
    lib_path, build_dir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    deps = _deps()
    if not force and not ptxas_info and not _stale(lib_path, deps):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
                     "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr"]
    if debug:
        common += ["-DDIFFATTN_DEBUG"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if ptxas_info:
        for _, log in results:
            sys.stdout.write(log)
    objs = [o for o, _ in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    ap.add_argument("--debug", action="store_true")
    a = ap.parse_args()
    print(build_library(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info, debug=a.debug))
