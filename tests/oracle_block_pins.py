"""Pins of the attention-block oracle (oracle/attn_block.py) to things other
than itself: a pure-Python brute force of the whole chain (exact, and with the
16-bit holding done element by element by PyTorch's scalar conversion),
PyTorch's float64 layer_norm and linear (library special cases), and
invariants of the block (a zero output projection leaves the residual, causal
prefixes, head relabelling, the output bias). Each pin takes the oracle module
so that the planted-mistake tests can run them on a modified copy."""
import math

import numpy as np
import torch


def _params(B, S, Hq, Hkv, D, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    hidden = Hq * D
    r = lambda *shape, s=1.0: (torch.randn(shape, generator=g, dtype=torch.float64) * s).to(torch.bfloat16).double().numpy()
    x = r(B, S, hidden, s=scale)
    gamma = r(hidden, s=0.5) + 1.0
    beta = r(hidden, s=0.2)
    w_qkv = r((Hq + 2 * Hkv) * D, hidden, s=1.0 / math.sqrt(hidden))
    b_qkv = r((Hq + 2 * Hkv) * D, s=0.1)
    w_o = r(hidden, Hq * D, s=1.0 / math.sqrt(hidden))
    b_o = r(hidden, s=0.1)
    return x, gamma, beta, w_qkv, b_qkv, w_o, b_o


def _round16(v, dtype):
    if dtype is None:
        return v
    return float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16 if dtype == "bf16" else torch.float16))


def _brute(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq, Hkv, D, causal, eps, dtype):
    """The block with plain loops over Python floats (math.fsum sums)."""
    B, S, hidden = x.shape
    F = (Hq + 2 * Hkv) * D
    y = np.zeros((B, S, hidden))
    for b in range(B):
        n = []
        for t in range(S):
            row = [float(v) for v in x[b, t]]
            mean = math.fsum(row) / hidden
            var = math.fsum((v - mean) ** 2 for v in row) / hidden
            n.append([_round16((row[c] - mean) / math.sqrt(var + eps) * gamma[c] + beta[c], dtype)
                      for c in range(hidden)])
        qkv = [[_round16(math.fsum(n[t][c] * w_qkv[f, c] for c in range(hidden)) + b_qkv[f], dtype)
                for f in range(F)] for t in range(S)]
        a = [[0.0] * (Hq * D) for _ in range(S)]
        grp = Hq // Hkv
        for h in range(Hq):
            hk = h // grp
            for i in range(S):
                qi = qkv[i][h * D:(h + 1) * D]
                keys = [j for j in range(S) if (j <= i or not causal)]
                w = []
                for j in keys:
                    kj = qkv[j][(Hq + hk) * D:(Hq + hk + 1) * D]
                    w.append(math.exp(math.fsum(qi[d] * kj[d] for d in range(D)) / math.sqrt(D)))
                tot = math.fsum(w)
                for d in range(D):
                    val = math.fsum(w[idx] * qkv[j][(Hq + Hkv + hk) * D + d] for idx, j in enumerate(keys)) / tot
                    a[i][h * D + d] = _round16(val, dtype)
        for t in range(S):
            for c in range(hidden):
                y[b, t, c] = math.fsum(a[t][f] * w_o[c, f] for f in range(Hq * D)) + b_o[c] + x[b, t, c]
    return y


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, what
    err = np.abs(a - b) / np.maximum(1.0, np.abs(b))
    assert float(err.max()) <= tol, f"{what}: {float(err.max()):.3e}"


def pin_block_brute_force_exact(ob):
    for n, (B, S, Hq, Hkv, D, causal) in enumerate([(2, 5, 2, 1, 4, True), (1, 6, 2, 2, 4, False),
                                                    (1, 4, 4, 2, 2, True)]):
        p = _params(B, S, Hq, Hkv, D, 100 + n)
        y = ob.block(*p, Hq=Hq, Hkv=Hkv, D=D, causal=causal, hold_in=None)
        _close(y, _brute(*p, Hq, Hkv, D, causal, 1e-5, None), 1e-12, f"block exact {n}")


def pin_block_brute_force_held(ob):
    for n, (B, S, Hq, Hkv, D, causal, dt) in enumerate([(2, 5, 2, 1, 4, True, "bf16"),
                                                        (1, 4, 2, 2, 4, True, "f16")]):
        p = _params(B, S, Hq, Hkv, D, 200 + n)
        y = ob.block(*p, Hq=Hq, Hkv=Hkv, D=D, causal=causal, hold_in=dt)
        _close(y, _brute(*p, Hq, Hkv, D, causal, 1e-5, dt), 1e-11, f"block held {dt}")


def pin_layer_norm_library(ob):
    x, gamma, beta = _params(3, 7, 4, 4, 8, 300)[:3]
    want = torch.nn.functional.layer_norm(torch.from_numpy(x), (x.shape[-1],), torch.from_numpy(gamma),
                                          torch.from_numpy(beta), eps=1e-5).numpy()
    _close(ob.layer_norm(x, gamma, beta), want, 1e-12, "layer_norm")


def pin_linear_library(ob):
    x, _, _, w, b, _, _ = _params(2, 9, 4, 2, 8, 301)
    want = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    _close(ob.linear(x, w, b), want, 1e-12, "linear")


def pin_zero_output_projection_leaves_the_residual(ob):
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = _params(2, 6, 2, 1, 8, 302)
    for hold_in in (None, "bf16"):
        y = ob.block(x, gamma, beta, w_qkv, b_qkv, np.zeros_like(w_o), np.zeros_like(b_o), Hq=2, Hkv=1, D=8,
                     hold_in=hold_in)
        assert np.array_equal(y, x), hold_in


def pin_output_bias_shifts_the_output(ob):
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = _params(1, 5, 2, 2, 4, 303)
    y0 = ob.block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=2, Hkv=2, D=4, hold_in=None)
    y1 = ob.block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o + 0.75, Hq=2, Hkv=2, D=4, hold_in=None)
    _close(y1 - y0, np.full_like(y0, 0.75), 1e-12, "output bias")


def pin_causal_prefix(ob):
    """A token's output depends on itself and earlier tokens only."""
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = _params(1, 8, 2, 1, 4, 304)
    y0 = ob.block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=2, Hkv=1, D=4, hold_in=None)
    x2 = x.copy()
    x2[:, 5:, :] += 3.0
    y2 = ob.block(x2, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=2, Hkv=1, D=4, hold_in=None)
    assert np.array_equal(y0[:, :5], y2[:, :5])
    assert not np.allclose(y0[:, 5:], y2[:, 5:])


def pin_head_relabelling(ob):
    """Swapping two heads in every projection (q, k, v rows and the matching
    W_o columns) leaves y unchanged (MHA)."""
    Hq = Hkv = 2
    D = 4
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = _params(1, 6, Hq, Hkv, D, 305)
    perm = np.concatenate([np.r_[D:2 * D, 0:D] + blk * Hq * D for blk in range(3)])
    colp = np.r_[D:2 * D, 0:D]
    y0 = ob.block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=Hq, Hkv=Hkv, D=D, hold_in=None)
    y1 = ob.block(x, gamma, beta, w_qkv[perm], b_qkv[perm], w_o[:, colp], b_o, Hq=Hq, Hkv=Hkv, D=D, hold_in=None)
    _close(y1, y0, 1e-12, "head relabelling")


ALL_BLOCK_PINS = [
    pin_block_brute_force_exact, pin_block_brute_force_held, pin_layer_norm_library, pin_linear_library,
    pin_zero_output_projection_leaves_the_residual, pin_output_bias_shifts_the_output, pin_causal_prefix,
    pin_head_relabelling,
]
