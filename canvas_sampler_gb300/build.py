"""Builds the sampler's shared library in-tree with nvcc for sm_103a.

    python -m canvas_sampler_gb300.build [--verbose]

Translation units compile in parallel; the library links the CUDA runtime statically so the
only run-time dependency is the driver.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libds_sampler.so"
SOURCES = ["ds_api.cu", "ds_rows.cu", "ds_simt.cu", "ds_tc.cu", "ds_tc_logits.cu",
           "ds_tc_selfcond.cu", "ds_tc_fused.cu", "ds_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"command failed ({p.returncode}): {' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return p.stdout + p.stderr


def build(verbose: bool = False, ptxas_verbose: bool = False, extra_flags=None) -> str:
    """Compile every translation unit and link the library; extra_flags (e.g. -D tuning
    definitions) are passed to every nvcc compile."""
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    flags = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
             "-I", os.path.join(ROOT, "include"), "-I", CSRC] + ARCH
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    flags += list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        out = _run([nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + flags, verbose)
        return obj, out

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if ptxas_verbose:
        for _, out in results:
            sys.stdout.write(out)
    objs = [o for o, _ in results]
    tmp = lib_path() + ".tmp"
    _run([nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"], verbose)
    os.replace(tmp, lib_path())
    return lib_path()


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print register / shared-memory usage")
    a = ap.parse_args()
    print(build(verbose=a.verbose, ptxas_verbose=a.ptxas))
