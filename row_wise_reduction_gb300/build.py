"""Build librowops.so in-tree with nvcc for sm_103a.

Compiles each translation unit under ``csrc/`` in parallel into ``_build/``
and links them (static CUDA runtime) into ``librowops.so`` next to this file;
with gcc, also the binding's small CPython call module ``_rowops_call``.
Run ``python -m row_wise_reduction_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import sysconfig
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "librowops.so")

SOURCES = [
    "rowops_api.cu",
    "softmax_f32.cu",
    "softmax_bf16.cu",
    "ln_gelu_f32.cu",
    "ln_gelu_bf16.cu",
    "online_softmax.cu",
    "online_softmax_noalloc.cu",
    "tma_softmax_f32.cu",
    "tma_softmax_bf16.cu",
    "tma_ln_gelu_f32.cu",
    "tma_ln_gelu_bf16.cu",
    "rms_f32.cu",
    "rms_bf16.cu",
    "tma_rms_f32_plain.cu",
    "tma_rms_f32_residual.cu",
    "tma_rms_bf16_plain.cu",
    "tma_rms_bf16_residual.cu",
    "reduce_f32.cu",
    "reduce_bf16.cu",
    "ln_gelu_erf_f32.cu",
    "ln_gelu_erf_bf16.cu",
    "tma_ln_gelu_erf_f32.cu",
    "tma_ln_gelu_erf_bf16.cu",
    "gelu.cu",
    "ln_gelu_bwd.cu",
    "ln_gelu_flat.cu",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the rowops CUDA library needs the CUDA 13 toolkit")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "rowops.h")]
    return [d for d in deps if os.path.isfile(d)]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _inputs() + [os.path.abspath(__file__)])


PYCALL_SRC = os.path.join(CSRC, "pycall.c")
PYCALL = os.path.join(PKG, "_rowops_call" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_pycall(force: bool = False) -> Optional[str]:
    """Compile the binding's CPython call module (gcc, Python headers); None
    where either is missing, in which case the binding calls the library
    through ctypes alone."""
    if not force and os.path.exists(PYCALL) and os.path.getmtime(PYCALL) >= os.path.getmtime(PYCALL_SRC):
        return PYCALL
    inc = sysconfig.get_paths().get("include")
    gcc = shutil.which("gcc") or shutil.which("cc")
    if not gcc or not inc or not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    tmp = PYCALL + f".tmp{os.getpid()}"
    r = subprocess.run([gcc, "-O2", "-shared", "-fPIC", "-I", inc, PYCALL_SRC, "-o", tmp], capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed on pycall.c:\n{r.stderr[-4000:]}")
    os.replace(tmp, PYCALL)
    return PYCALL


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if sources changed) and return the path of librowops.so."""
    build_pycall(force)
    if not (force or ptxas_info or _stale()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, _, r in results:
        log.append(f"== {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-6000:]}")
    with open(os.path.join(BUILD, "nvcc.log"), "w") as f:
        f.write("\n".join(log))
    if verbose:
        print("\n".join(log))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for _, o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
