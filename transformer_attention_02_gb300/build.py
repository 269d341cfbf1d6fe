"""Build the CUDA library ``libattn.so`` in-tree with nvcc for sm_103a.

Nine translation units (the host ABI, the host-buffer pipeline, the attention
block's GEMM and LayerNorm, and six families of attention-kernel variants),
compiled in parallel to objects under ``_build/`` and linked into one shared
library; one -gencode, no cmake. The results sit next to this file and are
git-ignored.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIBRARY = os.path.join(HERE, "libattn.so")
OBJDIR = os.path.join(HERE, "_build")
SOURCES = [os.path.join(CSRC, f) for f in
           ("attn_api.cu", "attn_host.cu", "block_kernels.cu", "fwd_bf16.cu", "fwd_f16.cu", "fwd_rope_bf16.cu",
            "fwd_rope_f16.cu", "fwd_pack_bf16.cu", "fwd_pack_f16.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in
                     ("attn_kernel.cuh", "ptx.cuh", "attn_launch.h", "attn_fwd_inst.cuh", "block_params.h",
                      "gemm_kernel.cuh")] + [
    os.path.join(ROOT, "include", "attn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = [*ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def up_to_date(output: str = LIBRARY) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(d) <= t for d in DEPENDS)


def build(force: bool = False, output: str = LIBRARY, verbose: bool = False) -> str:
    if not force and up_to_date(output):
        return output
    nvcc = nvcc_path()
    os.makedirs(OBJDIR, exist_ok=True)
    include = ["-I", os.path.join(ROOT, "include")]

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJDIR, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [nvcc, *FLAGS, *include, "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 1)) as pool:
        objects = list(pool.map(compile_one, SOURCES))
    subprocess.run([nvcc, *ARCH, "-shared", "-o", output + ".tmp", *objects], check=True)
    os.replace(output + ".tmp", output)
    return output


if __name__ == "__main__":  # pragma: no cover
    print(build(force=True, verbose=True))
