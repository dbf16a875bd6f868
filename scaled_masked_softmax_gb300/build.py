"""Builds libsms.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

Translation units are compiled in parallel into ``_build/`` at the repository
root and linked into ``scaled_masked_softmax_gb300/libsms.so``.  A rebuild is
skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsms.so")

SOURCES = ["sms_abi.cu", "sms_warp.cu", "sms_warp_bool.cu", "sms_stream.cu", "sms_ring.cu", "sms_ring_fwd_f32.cu",
           "sms_ring_fwd_f16.cu", "sms_ring_fwd_bf16.cu", "sms_ring_bwd.cu", "sms_tile_fwd.cu", "sms_tile_bwd.cu",
           "sms_online.cu", "sms_attn_abi.cu", "sms_attn_fwd.cu", "sms_attn_bwd.cu",
           "sms_attn_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsms")


def _inputs(csrc=CSRC):
    files = [os.path.join(csrc, f) for f in os.listdir(csrc)]
    files.append(os.path.join(INCLUDE, "sms.h"))
    return files


def up_to_date(lib=LIB, csrc=CSRC) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs(csrc))


def build_library(force: bool = False, verbose: bool = False, extra_flags=None, csrc: str = CSRC, out: str = LIB,
                  build_dir: str = BUILD) -> str:
    """Compile the sources in ``csrc`` into the shared library ``out``."""
    if not force and up_to_date(out, csrc):
        return out
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = NVCC_FLAGS + ["-I", csrc] + (list(extra_flags) if extra_flags else [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + ARCH + flags + ["-c", os.path.join(csrc, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(out)} failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys

    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
