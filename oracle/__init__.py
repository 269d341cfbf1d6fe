"""FP64 CPU oracle for the fused attention forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product library never does.
It shares no code with the CUDA path. The arithmetic lives in
``attn_oracle.c`` (the plain definition, FP64, OpenMP over query rows); this
module only compiles that file with gcc and marshals numpy arrays through ctypes.

Every function of the oracle is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle.py`` (brute force, a library special case, closed forms,
invariants and planted-mistake checks); none is left unpinned.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

MASK_NONE, MASK_CAUSAL, MASK_ADDITIVE, MASK_CAUSAL_ADDITIVE = 0, 1, 2, 3
DTYPES = {"bf16": 0, "f16": 1}


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags=()) -> str:
    """Compile the oracle's C source into a shared library (gcc, OpenMP).

    No -ffast-math: the oracle keeps IEEE double semantics and evaluation order.
    """
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           *extra_flags, "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True)
    return output


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, library: str = LIBRARY):
        stale = library == LIBRARY and os.path.exists(library) and \
            os.path.getmtime(library) < os.path.getmtime(SOURCE)
        if not os.path.exists(library) or stale:
            build(output=library)
        self.path = library
        self._lib = ctypes.CDLL(library)
        P = ctypes.c_void_p
        I = ctypes.c_int
        f = self._lib.oracle_attn_fwd_rope
        f.argtypes = [P, P, P, I, P, I, I, I, I, I, I, I, ctypes.c_double,
                      I, P, P, I, I, P, P, P, I, ctypes.c_double, ctypes.c_longlong, ctypes.c_longlong, I]
        f.restype = I
        self._lib.oracle_num_threads.restype = I
        r = self._lib.oracle_rope_rotate
        r.argtypes = [P, I, I, I, I, I, ctypes.c_double, ctypes.c_longlong, I, P]
        r.restype = I

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def attention(self, q, k, v, *, mask_kind: int, mask=None, scale=None,
                  dtype: str = "bf16", slices=None, rows=None, n_threads: int = 0,
                  want_psum: bool = False, rope_base: float = 0.0, q_pos0: int = 0, k_pos0: int = 0,
                  rope_round: bool = False):
        """FP64 attention on 16-bit inputs.

        q: (B,Sq,Hq,D), k/v: (B,Sk,Hkv,D) as uint16/int16 bit patterns (numpy)
        of bf16 or fp16 values; mask: (B,Sq,Sk) float32 for the additive kinds.
        slices: list of (b, h) pairs (default: every slice in (b, h) order);
        rows: (begin, end) query-row range (default: all rows).
        rope_base > 0 rotates q and k (rotary position embedding, interleaved
        pairs, angle pos * rope_base^(-2i/D)) with query row i at position
        q_pos0 + i and key j at k_pos0 + j; rope_round rounds each rotated
        element to the nearest value of `dtype` (ties to even), the reading in
        which the rotated q and k are held in the input's 16-bit type.

        Returns (o, lse[, psum]) with o of shape (n_slices, rows, D) and lse of
        shape (n_slices, rows), both float64. With the default slices and rows,
        reshape with ``to_bshd`` / ``to_bhs`` for the full tensors.
        """
        q = np.ascontiguousarray(np.asarray(q).view(np.uint16))
        k = np.ascontiguousarray(np.asarray(k).view(np.uint16))
        v = np.ascontiguousarray(np.asarray(v).view(np.uint16))
        B, Sq, Hq, D = q.shape
        Bk, Sk, Hkv, Dk = k.shape
        if (Bk, Dk) != (B, D) or v.shape != k.shape:
            raise ValueError("q/k/v shapes disagree")
        additive = mask_kind in (MASK_ADDITIVE, MASK_CAUSAL_ADDITIVE)
        if additive:
            mask = np.ascontiguousarray(np.asarray(mask, dtype=np.float32))
            if mask.shape != (B, Sq, Sk):
                raise ValueError("mask must be (B, Sq, Sk) float32")
        if slices is None:
            slices = [(b, h) for b in range(B) for h in range(Hq)]
        sb = np.ascontiguousarray([s[0] for s in slices], dtype=np.int32)
        sh = np.ascontiguousarray([s[1] for s in slices], dtype=np.int32)
        r0, r1 = (0, Sq) if rows is None else rows
        n = len(slices)
        o = np.zeros((n, r1 - r0, D), dtype=np.float64)
        lse = np.zeros((n, r1 - r0), dtype=np.float64)
        psum = np.zeros((n, r1 - r0), dtype=np.float64) if want_psum else None
        sc = float("nan") if scale is None else float(scale)
        rc = self._lib.oracle_attn_fwd_rope(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, DTYPES[dtype],
            mask.ctypes.data if additive else None, int(mask_kind),
            B, Hq, Hkv, Sq, Sk, D, sc,
            n, sb.ctypes.data, sh.ctypes.data, r0, r1,
            o.ctypes.data, lse.ctypes.data,
            psum.ctypes.data if want_psum else None, int(n_threads),
            float(rope_base), int(q_pos0), int(k_pos0), int(bool(rope_round)))
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments (rc={rc})")
        return (o, lse, psum) if want_psum else (o, lse)

    def rotate(self, x, *, base: float, pos0: int = 0, dtype: str = "bf16", rope_round: bool = True):
        """Rotary embedding alone: x (B, S, H, D) 16-bit bit patterns, row s at
        position pos0 + s; returns the rotated values as float64, same shape
        (rounded to `dtype` when rope_round)."""
        x = np.ascontiguousarray(np.asarray(x).view(np.uint16))
        B, S, H, D = x.shape
        y = np.zeros(x.shape, dtype=np.float64)
        rc = self._lib.oracle_rope_rotate(x.ctypes.data, DTYPES[dtype], B, S, H, D, float(base), int(pos0),
                                          int(bool(rope_round)), y.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments (rc={rc})")
        return y


def to_bshd(o_slices: np.ndarray, B: int, Hq: int) -> np.ndarray:
    """(B*Hq, S, D) slices in (b, h) order -> (B, S, Hq, D)."""
    n, S, D = o_slices.shape
    return o_slices.reshape(B, Hq, S, D).transpose(0, 2, 1, 3)


def to_bhs(lse_slices: np.ndarray, B: int, Hq: int) -> np.ndarray:
    """(B*Hq, S) slices in (b, h) order -> (B, Hq, S)."""
    return lse_slices.reshape(B, Hq, -1)


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def attention(*args, **kwargs):
    """Module-level shortcut for ``default().attention``."""
    return default().attention(*args, **kwargs)


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build())
    sys.exit(0)
