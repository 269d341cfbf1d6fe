"""Build the CUDA library ``libattn.so`` in-tree with nvcc for sm_103a.

One translation unit (host ABI + every kernel instantiation), one -gencode,
no cmake. The result sits next to this file and is git-ignored.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIBRARY = os.path.join(HERE, "libattn.so")
SOURCES = [os.path.join(CSRC, "attn_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("attn_kernel.cuh", "ptx.cuh")] + [
    os.path.join(ROOT, "include", "attn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


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
    cmd = [nvcc_path(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", output + ".tmp", *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(output + ".tmp", output)
    return output


if __name__ == "__main__":  # pragma: no cover
    print(build(force=True, verbose=True))
