"""In-tree build of the two CUDA libraries (sm_103a only).

    libkda_h0.so  fp32 state pool   (-DKDA_STATE16=0)
    libkda_h1.so  fp16 state pool   (-DKDA_STATE16=1)

Both come from the same two source files; the pool dtype is a compile-time
constant, as the _h0/_h1 kernel names of ROCm/ATOM pull request 2945 (Changes)
make it.  The libraries link the shared CUDA runtime, so they share the
runtime instance (and the streams) of the PyTorch process that loads them.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
LIB_DIR = os.path.join(PKG_DIR, "lib")
SOURCES = [os.path.join(CSRC, f) for f in ("kda_api.cu", "kda_common.cuh", "kda_decode_tma.cuh",
                                          "kda_verify_tma.cuh", "kda_conv.cuh", "kda_ckpt.cuh",
                                          "kda_prefill_chunk.cuh", "kda_stage.cuh")] + [os.path.join(INCLUDE, "kda.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def lib_path(state16: bool) -> str:
    return os.path.join(LIB_DIR, f"libkda_h{int(bool(state16))}.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the KDA CUDA libraries cannot be built")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def nvcc_command(state16: bool, out: str, extra: list[str] | None = None) -> list[str]:
    return [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
            f"-I{INCLUDE}", f"-DKDA_STATE16={int(bool(state16))}",
            *(extra or []), os.path.join(CSRC, "kda_api.cu"), "-o", out]


def _build_one(state16: bool, force: bool) -> str:
    out = lib_path(state16)
    if force or _stale(out):
        os.makedirs(LIB_DIR, exist_ok=True)
        tmp = f"{out}.tmp{os.getpid()}"
        proc = subprocess.run(nvcc_command(state16, tmp), capture_output=True, text=True)
        if proc.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(out)}:\n{proc.stderr}")
        os.replace(tmp, out)
    return out


def build(force: bool = False) -> list[str]:
    """Compile both libraries (in parallel) if any source is newer than them."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda s: _build_one(s, force), (False, True)))


if __name__ == "__main__":
    for p in build(force=True):
        print(p)
