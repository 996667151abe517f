"""Builds the CUDA library libfocus_gb300.so in-tree for sm_103a.

Every translation unit under csrc/ is compiled by nvcc in parallel and linked
into one shared library with the CUDA runtime linked statically, so the
library needs only the NVIDIA driver at run time.  Run as
``python -m learned_group_sparse_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libfocus_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Translation units whose arithmetic is exp2 / log2 / reciprocal-heavy use
# the fast hardware approximations; the assignment keeps IEEE fp32.
FAST_MATH = {"focus_attn_group.cu", "focus_attn_window.cu", "focus_gated_bwd_tc.cu",
             "focus_gated_tc.cu", "focus_merge.cu"}


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(os.path.dirname(HERE), "include", "focus.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose_ptxas: bool) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, src[:-3] + ".o")
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-c", os.path.join(CSRC, src), "-o", obj]
    if src in FAST_MATH:
        cmd.append("--use_fast_math")
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    """Compiles (if stale) and returns the path of libfocus_gb300.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and not verbose_ptxas and os.path.exists(LIB) and \
            os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    if verbose_ptxas:
        for (_, log), s in zip(results, srcs):
            sys.stderr.write(f"== {s}\n{log}")
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp,
           *[o for o, _ in results], "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
