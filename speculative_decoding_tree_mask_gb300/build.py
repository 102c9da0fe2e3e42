"""Builds the CUDA library in-tree with nvcc for sm_103a.

``python -m speculative_decoding_tree_mask_gb300.build`` or ``build()`` compiles every
translation unit under ``csrc/`` in parallel and links ``libspecverify.so`` next to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libspecverify.so")
# The debug flavour: the same kernels with their consistency checks compiled in (SPEC_DEBUG).
DEBUG_OBJDIR = os.path.join(HERE, "_build_debug")
DEBUG_LIBRARY = os.path.join(HERE, "libspecverify_debug.so")
SOURCES = ["api.cu", "row_stats.cu", "tree_mask.cu", "walk_greedy.cu", "walk_sample_point.cu",
           "walk_sample_dense.cu", "walk_sample_logits_bf16.cu", "walk_sample_logits_f32.cu",
           "lazy_greedy.cu", "kv_commit.cu", "noalloc.cu", "budget.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(INCLUDE, "spec_verify.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          nvtx: bool = False, debug: bool = False) -> str:
    """Compile and link the library; returns its path. Rebuilds only when a source changed.
    `nvtx` compiles an NVTX range around every ABI entry point (for timeline profilers);
    `debug` builds the checked flavour (SPEC_DEBUG) as libspecverify_debug.so instead."""
    library = DEBUG_LIBRARY if debug else LIBRARY
    objdir = DEBUG_OBJDIR if debug else OBJDIR
    if not force and os.path.exists(library) and os.path.getmtime(library) >= _newest_input():
        return library
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    extra = list(extra or []) + (["-DSPEC_NVTX"] if nvtx else []) + \
        (["-DSPEC_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = library + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, library)
    return library


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv or "--nvtx" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None,
                nvtx="--nvtx" in sys.argv, debug="--debug" in sys.argv))
