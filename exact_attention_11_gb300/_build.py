"""Builds libfattn.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into
``exact_attention_11_gb300/libfattn.so`` (CUDA runtime linked statically; the
driver API is reached through cudaGetDriverEntryPointByVersion, so no libcuda
link is needed).  ``python -m exact_attention_11_gb300._build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfattn.so")
SOURCES = ["api.cu", "fwd_f32.cu", "fwd_bf16.cu", "decode.cu", "decode_noalloc.cu",
           "bwd_bf16.cu", "bwd_bf16_d128.cu", "bwd_bf16_d64.cu", "decode_gqa.cu", "fp8_quant.cu",
           "fwd_d256.cu", "mask_tiles.cu", "decode_gqa_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: libfattn needs the CUDA toolkit to build")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "fattn.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


# Kernels that rebalance registers with setmaxnreg: ptxas must give them
# exactly this many registers per thread at launch, or the warpgroups that
# raise their count could wait forever for registers that do not exist.
SETMAXNREG_KERNELS = {"fwd_bf16.cu": ("fwd_bf16_tc_kernel", 168),
                      "bwd_bf16_d64.cu": ("bwd_pipe64_kernel", 168),
                      "bwd_bf16_d128.cu": ("bwd_pipe_kernel", 168)}


def _check_registers(src: str, ptxas_log: str) -> None:
    if src not in SETMAXNREG_KERNELS:
        return
    name, want = SETMAXNREG_KERNELS[src]
    found = []
    current = None
    for line in ptxas_log.splitlines():
        if "Compiling entry function" in line:
            current = line
        elif "Used" in line and "registers" in line and current and name in current:
            found.append(int(line.split("Used")[1].split("registers")[0]))
    if not found or any(r != want for r in found):
        raise RuntimeError(f"{src}: {name} must be built with exactly {want} registers per "
                           f"thread for its setmaxnreg split; ptxas reported {found}")


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        flags = list(extra_flags)
        if src in SETMAXNREG_KERNELS and "-Xptxas" not in flags:
            flags += ["-Xptxas", "-v"]
        cmd = [cc, *ARCH, *FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        _check_registers(src, r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force=True, verbose=v, extra_flags=(["-Xptxas", "-v"] if v else [])))
