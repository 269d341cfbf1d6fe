"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the FP64 oracle on the same seeded inputs, and compare.

Tolerances (fixed for the measured path): O max-abs error <= 2e-2 and
mean-abs error <= 2e-3 against FP64; for heavy-tailed (Student-t) values the
error is taken relative to max(1, |o_ref|). LSE: |lse - lse_ref| <= 1e-3 *
max(1, |lse_ref|). No NaN/Inf anywhere; rows with no visible key must be
exactly o = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from transformer_attention_02_gb300 import attention
from transformer_attention_02_gb300 import inputs as I

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def run_gpu(q, k, v, mask, causal, scale=None, device="cuda"):
    dev = torch.device(device)
    m = None if mask is None else mask.to(dev)
    o, lse = attention(q.to(dev), k.to(dev), v.to(dev), causal=causal, mask=m, scale=scale)
    torch.cuda.synchronize()
    return o, lse


def check(o_gpu, lse_gpu, q, k, v, mask, mask_kind, *, scale=None, slices=None, rows=None,
          heavy_tail=False, label="", rope=None):
    """Compare GPU outputs with the oracle on the given (b, h) slices and rows.

    rope: None, or dict(base=, q_pos0=, k_pos0=) for the rotary variant (the
    oracle then rotates q and k and holds them in the input's 16-bit type).
    """
    rope_kw = {} if rope is None else dict(rope_base=rope["base"], q_pos0=rope["q_pos0"],
                                           k_pos0=rope["k_pos0"], rope_round=True)
    B, Sq, Hq, D = q.shape
    if slices is None:
        slices = [(b, h) for b in range(B) for h in range(Hq)]
    r0, r1 = (0, Sq) if rows is None else rows
    ref_o, ref_l = oracle.default().attention(
        I.bits(q), I.bits(k), I.bits(v), mask_kind=mask_kind,
        mask=None if mask is None else mask.numpy(), scale=scale, slices=slices, rows=(r0, r1),
        dtype="f16" if q.dtype == torch.float16 else "bf16", **rope_kw)
    og = o_gpu.float().cpu()
    lg = lse_gpu.float().cpu()
    got_o = np.stack([og[b, r0:r1, h, :].numpy() for b, h in slices]).astype(np.float64)
    got_l = np.stack([lg[b, h, r0:r1].numpy() for b, h in slices]).astype(np.float64)

    assert np.isfinite(got_o).all(), f"{label}: non-finite O"
    empty = ~np.isfinite(ref_l)
    assert np.all(ref_l[empty] == -np.inf)
    assert np.all(got_l[empty] == -np.inf), f"{label}: rows with no visible key need lse = -inf"
    assert np.all(got_o[empty] == 0.0), f"{label}: rows with no visible key need o = 0"
    assert np.isfinite(got_l[~empty]).all(), f"{label}: non-finite LSE"

    diff = np.abs(got_o - ref_o)
    if heavy_tail:
        diff = diff / np.maximum(1.0, np.abs(ref_o))
    lse_err = np.abs(got_l[~empty] - ref_l[~empty]) / np.maximum(1.0, np.abs(ref_l[~empty]))
    stats = dict(o_max=float(diff.max()) if diff.size else 0.0,
                 o_mean=float(diff.mean()) if diff.size else 0.0,
                 lse_max=float(lse_err.max()) if lse_err.size else 0.0,
                 o_max_raw=float(np.abs(got_o - ref_o).max()) if diff.size else 0.0)
    assert stats["o_max"] <= O_MAX_ABS, f"{label}: O max err {stats}"
    assert stats["o_mean"] <= O_MEAN_ABS, f"{label}: O mean err {stats}"
    assert stats["lse_max"] <= LSE_REL, f"{label}: LSE err {stats}"
    return stats


def full_scan(o_gpu, lse_gpu, may_be_empty=False):
    """Every O element finite; every LSE finite (or -inf where rows may be empty)."""
    assert bool(torch.isfinite(o_gpu).all()), "non-finite O"
    if may_be_empty:
        assert not bool(torch.isnan(lse_gpu).any()) and not bool((lse_gpu == float("inf")).any())
    else:
        assert bool(torch.isfinite(lse_gpu).all()), "non-finite LSE"
