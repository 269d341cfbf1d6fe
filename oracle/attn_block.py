"""FP64 oracle of the fused attention block — TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this module; the product path never does.

The block ("ATB orchestration blog" (hwcomputing.csdn.net/6a15a709662f9a54cb774da1),
section 2, the graph-operator layer: its fused attention block example and the
atb.GraphOp listing that follows it): for x of shape (B, S, hidden),

    n    = LayerNorm(x)            per token over hidden, eps = 1e-5, gain gamma, bias beta
    qkv  = n W_qkv^T + b_qkv       one projection to (Hq + 2 Hkv) * D features: [q | k | v]
    a    = FlashAttention(q, k, v) causal, scale 1/sqrt(D), heads of D features
    y    = a W_o^T + b_o + x       output projection, then the residual (the block's input)

Readings (where the pages leave a step open):
- LayerNorm is the usual one: mean and biased variance over the hidden
  features, (x - mean) / sqrt(var + eps) * gamma + beta.
- "Linear" has a bias (x W^T + b, W of shape (out, in)).
- The projection's output features are ordered [q | k | v], each split into
  heads of D consecutive features; the listing's single head count means
  Hq = Hkv (MHA), and GQA (Hkv < Hq) is the same split with fewer K/V heads.
- The residual is the block's input x ("ResidualAdd(output, input)").
- With hold_in set to "bf16" or "f16", every intermediate tensor (n, q, k, v,
  a) is rounded to that 16-bit type, as the chain's operators hand 16-bit
  tensors to each other; each stage itself is computed exactly in FP64 from
  those values, and y is returned unrounded. With hold_in=None the whole
  chain is exact FP64.

Steps use library primitives where the definition is a plain one: numpy's
FP64 matrix product for the two projections, PyTorch's conversion for the
16-bit rounding, and the compiled FP64 attention oracle (oracle_attn_fwd) for
the attention step (it takes 16-bit inputs, so with hold_in=None the exact
attention below is used instead).
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-5


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Row-wise LayerNorm in FP64 over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None) -> np.ndarray:
    """x W^T + b in FP64 (W of shape (out, in))."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    return y if b is None else y + np.asarray(b, np.float64)


def hold(x: np.ndarray, dtype: str | None) -> np.ndarray:
    """Round to the 16-bit type (PyTorch's conversion), or keep exact."""
    if dtype is None:
        return np.asarray(x, np.float64)
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float16).double().numpy()


def _bits16(x: np.ndarray, dtype: str) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy()


def attention_exact(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool) -> np.ndarray:
    """Plain FP64 attention for (B, S, H, D) inputs (GQA by contiguous groups),
    scale 1/sqrt(D); used when the chain is exact."""
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Sq, Hq, D))
    for b in range(B):
        for h in range(Hq):
            s = (q[b, :, h, :] @ k[b, :, h // g, :].T) / math.sqrt(D)
            if causal:
                i = np.arange(Sq)[:, None]
                j = np.arange(Sk)[None, :]
                s = np.where(j <= i + (Sk - Sq), s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            out[b, :, h, :] = (p / p.sum(axis=1, keepdims=True)) @ v[b, :, h // g, :]
    return out


def block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, *, Hq: int, Hkv: int, D: int, causal: bool = True,
          eps: float = EPS, hold_in: str | None = "bf16", orc=None, want_parts: bool = False):
    """The attention block on x (B, S, hidden) (values, any float dtype).

    Returns y (B, S, hidden) FP64, or (y, parts) with the intermediate tensors
    (n, q, k, v, a) as held. The attention step runs for every token (it needs
    all keys of each batch entry)."""
    x = np.asarray(x, np.float64)
    B, S, hidden = x.shape
    if hidden != Hq * D or w_qkv.shape != ((Hq + 2 * Hkv) * D, hidden) or w_o.shape != (hidden, Hq * D):
        raise ValueError("inconsistent block sizes")
    n = hold(layer_norm(x, gamma, beta, eps), hold_in)
    qkv = hold(linear(n.reshape(B * S, hidden), w_qkv, b_qkv), hold_in).reshape(B, S, (Hq + 2 * Hkv) * D)
    q = qkv[..., : Hq * D].reshape(B, S, Hq, D)
    k = qkv[..., Hq * D: (Hq + Hkv) * D].reshape(B, S, Hkv, D)
    v = qkv[..., (Hq + Hkv) * D:].reshape(B, S, Hkv, D)
    if hold_in is None:
        a = attention_exact(q, k, v, causal)
    else:
        import oracle as _oracle
        orc = orc or _oracle.default()
        kind = _oracle.MASK_CAUSAL if causal else _oracle.MASK_NONE
        o, _ = orc.attention(_bits16(q, hold_in), _bits16(k, hold_in), _bits16(v, hold_in), mask_kind=kind,
                             dtype=hold_in, scale=1.0 / math.sqrt(D))
        a = _oracle.to_bshd(o, B, Hq)
    a = hold(a, hold_in)
    y = linear(a.reshape(B * S, Hq * D), w_o, b_o).reshape(B, S, hidden) + x
    if want_parts:
        return y, dict(n=n, q=q, k=k, v=v, a=a)
    return y
