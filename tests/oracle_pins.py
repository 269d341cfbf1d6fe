"""Checks that pin the FP64 oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with an independent statement of what attention computes:
a pure-Python brute force (math.fsum, no max subtraction) on tiny benign inputs,
PyTorch's float64 scaled_dot_product_attention and logsumexp (a library special
case), closed forms and invariants that the definition fixes. They are used
twice: ``test_oracle.py`` runs them on the real oracle, and
``test_oracle_mutations.py`` runs them on copies of the oracle with a planted
mistake and requires that at least one of them fails for every mistake.

The definition being pinned ("ATB engineering guide" §5.1 eager formula;
"CANN-ATB图优化-…融合算子" Pattern 2; "ops-transformer：…实战" §3.2):
  o = softmax(scale * Q K^T + mask) V, lse = logsumexp(scale * Q K^T + mask),
  causal keys visible iff j <= i + Sk - Sq, K/V head = h // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from transformer_attention_02_gb300 import inputs as I

NONE, CAUSAL, ADDITIVE, CAUSAL_ADDITIVE = 0, 1, 2, 3


# ----------------------------------------------------------------- helpers

def _rand16(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype)


def _finite_mask(B, Sq, Sk, seed, n_neg_inf=0):
    """FP32 additive mask with finite entries and n_neg_inf -inf keys per row."""
    g = torch.Generator().manual_seed(seed)
    m = torch.randn((B, Sq, Sk), generator=g) * 0.5
    if n_neg_inf:
        idx = torch.argsort(torch.rand((B, Sq, Sk), generator=g), dim=-1)[..., :n_neg_inf]
        m.scatter_(-1, idx, float("-inf"))
    return m


def _bits(t):
    return I.bits(t)


def _run(orc, q, k, v, kind, mask=None, scale=None, dtype="bf16", **kw):
    return orc.attention(_bits(q), _bits(k), _bits(v), mask_kind=kind,
                         mask=None if mask is None else mask.numpy(),
                         scale=scale, dtype=dtype, **kw)


def _brute(q, k, v, kind, mask, scale):
    """Pure-Python attention: exp without max subtraction, exact sums (fsum).

    Only for small benign inputs (|scores| of order 1). Returns o as
    (B*Hq, Sq, D) slices in (b, h) order and lse as (B*Hq, Sq), like the oracle.
    """
    qf, kf, vf = q.double().tolist(), k.double().tolist(), v.double().tolist()
    mf = None if mask is None else mask.double().tolist()
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    causal = kind in (CAUSAL, CAUSAL_ADDITIVE)
    additive = kind in (ADDITIVE, CAUSAL_ADDITIVE)
    o = np.zeros((B * Hq, Sq, D))
    lse = np.zeros((B * Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            g = h * Hkv // Hq
            for i in range(Sq):
                weights = []
                for j in range(Sk):
                    if causal and j > i + Sk - Sq:
                        continue
                    s = scale * math.fsum(qf[b][i][h][d] * kf[b][j][g][d] for d in range(D))
                    if additive:
                        s += mf[b][i][j]
                    if s == float("-inf"):
                        continue
                    weights.append((math.exp(s), j))
                z = math.fsum(w for w, _ in weights)
                if z == 0.0:
                    lse[b * Hq + h, i] = float("-inf")
                    continue
                for d in range(D):
                    o[b * Hq + h, i, d] = math.fsum(w * vf[b][j][g][d] for w, j in weights) / z
                lse[b * Hq + h, i] = math.log(z)
    return o, lse


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite values differ"
    err = np.abs(a[fin] - b[fin])
    lim = tol * np.maximum(1.0, np.abs(b[fin]))
    assert np.all(err <= lim), f"{what}: max err {err.max() if err.size else 0:.3e}"


# ------------------------------------------------------------------- pins

def pin_brute_force(orc):
    """Oracle == pure-Python brute force on tiny inputs, every mask kind."""
    cases = [
        # B, Hq, Hkv, Sq, Sk, D, kind, explicit scale
        (1, 2, 2, 5, 7, 8, NONE, 0.3),
        (2, 4, 2, 5, 9, 8, CAUSAL, None),        # GQA, Sq < Sk (bottom-right)
        (1, 2, 1, 9, 5, 8, CAUSAL, None),        # MQA, Sq > Sk: empty rows
        (2, 2, 2, 6, 6, 4, ADDITIVE, None),      # per-batch masks, shared by heads
        (2, 4, 1, 7, 7, 8, CAUSAL_ADDITIVE, 0.25),
    ]
    for n, (B, Hq, Hkv, Sq, Sk, D, kind, scale) in enumerate(cases):
        q = _rand16((B, Sq, Hq, D), 10 * n + 1)
        k = _rand16((B, Sk, Hkv, D), 10 * n + 2)
        v = _rand16((B, Sk, Hkv, D), 10 * n + 3)
        mask = _finite_mask(B, Sq, Sk, 10 * n + 4, n_neg_inf=2) if kind >= ADDITIVE else None
        o, lse = _run(orc, q, k, v, kind, mask, scale)
        eff = (1.0 / math.sqrt(D)) if scale is None else scale
        ob, lb = _brute(q, k, v, kind, mask, eff)
        _close(o, ob, what=f"brute case {n} O")
        _close(lse, lb, what=f"brute case {n} LSE")


def pin_brute_force_f16(orc):
    """The fp16 storage path agrees with brute force on torch-widened fp16 values."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 6, 6, 8
    q = _rand16((B, Sq, Hq, D), 71, torch.float16)
    k = _rand16((B, Sk, Hkv, D), 72, torch.float16)
    v = _rand16((B, Sk, Hkv, D), 73, torch.float16)
    o, lse = _run(orc, q, k, v, CAUSAL, dtype="f16")
    ob, lb = _brute(q, k, v, CAUSAL, None, 1.0 / math.sqrt(D))
    _close(o, ob, what="f16 O")
    _close(lse, lb, what="f16 LSE")


def pin_widening_exact(orc):
    """With one key, o = v exactly: checks the bf16 and fp16 widening bit-for-bit."""
    for dt, name in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
        fin = torch.finfo(dt)
        vals = torch.tensor([0.0, -0.0, 1.0, -1.5, fin.max, -fin.max, fin.tiny,
                             fin.tiny / 4, fin.eps, 3.140625, -1e-3, 65504.0 if name == "f16" else 1e30,
                             7.0, -2.0 ** -12, 0.1, -0.3], dtype=torch.float32).to(dt)
        D = vals.numel()
        v = vals.reshape(1, 1, 1, D)
        q = torch.zeros((1, 1, 1, D), dtype=dt)
        k = torch.zeros((1, 1, 1, D), dtype=dt)
        o, lse = _run(orc, q, k, v, NONE, dtype=name)
        want = vals.double().numpy()
        assert np.array_equal(o[0, 0], want), f"{name} widening: {o[0, 0]} vs {want}"
        assert lse[0, 0] == 0.0


def pin_sdpa_float64(orc):
    """Oracle == torch float64 scaled_dot_product_attention (O) and logsumexp (LSE)."""
    for (B, Hq, Hkv, Sq, Sk, D, kind) in [(2, 4, 2, 48, 48, 64, CAUSAL),
                                          (1, 4, 4, 33, 40, 32, ADDITIVE),
                                          (2, 8, 2, 20, 52, 16, CAUSAL_ADDITIVE)]:
        q = _rand16((B, Sq, Hq, D), 101)
        k = _rand16((B, Sk, Hkv, D), 102)
        v = _rand16((B, Sk, Hkv, D), 103)
        mask = _finite_mask(B, Sq, Sk, 104, n_neg_inf=3) if kind >= ADDITIVE else None
        o, lse = _run(orc, q, k, v, kind, mask)
        qd = q.double().permute(0, 2, 1, 3)
        kd = k.double().permute(0, 2, 1, 3)
        vd = v.double().permute(0, 2, 1, 3)
        bias = torch.zeros((B, 1, Sq, Sk), dtype=torch.float64)
        if kind >= ADDITIVE:
            bias = bias + mask.double()[:, None]
        if kind in (CAUSAL, CAUSAL_ADDITIVE):
            i = torch.arange(Sq)[:, None]
            j = torch.arange(Sk)[None, :]
            bias = bias.masked_fill(j > i + (Sk - Sq), float("-inf"))
        scale = 1.0 / math.sqrt(D)
        ref = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=bias, scale=scale,
                                             enable_gqa=True)
        kx = kd.repeat_interleave(Hq // Hkv, dim=1)
        ref_lse = torch.logsumexp(qd @ kx.transpose(-1, -2) * scale + bias, dim=-1)
        _close(o, ref.reshape(B * Hq, Sq, D).numpy(), tol=1e-11, what="sdpa O")
        _close(lse, ref_lse.reshape(B * Hq, Sq).numpy(), tol=1e-11, what="sdpa LSE")


def pin_rowsum_one(orc):
    """Normalised probabilities sum to 1 per row (0 for a row with no visible key)."""
    B, Hq, Sq, Sk, D = 1, 2, 12, 8, 16
    q = _rand16((B, Sq, Hq, D), 201, scale=3.0)
    k = _rand16((B, Sk, Hq, D), 202, scale=3.0)
    v = _rand16((B, Sk, Hq, D), 203)
    o, lse, ps = _run(orc, q, k, v, CAUSAL, want_psum=True)
    visible = (np.arange(Sq) + (Sk - Sq)) >= 0
    assert np.all(np.abs(ps[:, visible] - 1.0) <= 1e-12), ps
    assert np.all(ps[:, ~visible] == 0.0)


def pin_constant_v(orc):
    """V == c everywhere gives O == c for every row with a visible key."""
    B, Hq, Hkv, S, D = 2, 4, 2, 16, 8
    q = _rand16((B, S, Hq, D), 301, scale=2.0)
    k = _rand16((B, S, Hkv, D), 302, scale=2.0)
    v = torch.full((B, S, Hkv, D), 1.5, dtype=torch.bfloat16)
    o, _ = _run(orc, q, k, v, CAUSAL)
    assert np.all(np.abs(o - 1.5) <= 1e-12)


def pin_zero_q(orc):
    """Q = 0: O is the mean of V over the unmasked keys and LSE = ln(#unmasked)."""
    cfg = I.AttnConfig("zq", 2, 2, 2, 24, 64, 16, False, additive_mask=True,
                       values="zero_q", seed=5)
    q, k, v, mask = I.make_inputs(cfg)
    o, lse = _run(orc, q, k, v, ADDITIVE, mask)
    keep = torch.isfinite(mask)                                       # (B, Sq, Sk)
    n_keep = keep.sum(-1).double()                                    # (B, Sq)
    assert torch.all(n_keep == 64 - math.floor(0.3 * 64))
    vd = v.double()
    for b in range(2):
        for h in range(2):
            mean = (keep[b].double() @ vd[b, :, h, :]) / n_keep[b][:, None]
            _close(o[b * 2 + h], mean.numpy(), what="zero-q mean")
            _close(lse[b * 2 + h], torch.log(n_keep[b]).numpy(), what="zero-q lse")


def pin_causal_row0(orc):
    """Causal with Sq == Sk: row 0 sees only key 0, so O[0] = V[0], LSE[0] = s_00."""
    B, Hq, S, D = 1, 2, 10, 16
    q = _rand16((B, S, Hq, D), 401)
    k = _rand16((B, S, Hq, D), 402)
    v = _rand16((B, S, Hq, D), 403)
    o, lse = _run(orc, q, k, v, CAUSAL, scale=0.5)
    for h in range(Hq):
        assert np.array_equal(o[h, 0], v[0, 0, h].double().numpy())
        s00 = 0.5 * math.fsum(float(a) * float(b) for a, b in
                              zip(q[0, 0, h].double(), k[0, 0, h].double()))
        assert abs(lse[h, 0] - s00) <= 1e-12 * max(1.0, abs(s00))


def pin_shift_invariance(orc):
    """Adding c_i to every logit of row i (via the mask) keeps O and adds c_i to LSE."""
    B, Hq, Sq, Sk, D = 2, 2, 9, 11, 8
    q = _rand16((B, Sq, Hq, D), 501)
    k = _rand16((B, Sk, Hq, D), 502)
    v = _rand16((B, Sk, Hq, D), 503)
    zero = torch.zeros((B, Sq, Sk))
    c = torch.linspace(-3.0, 5.0, B * Sq).reshape(B, Sq, 1).expand(B, Sq, Sk).contiguous()
    o0, l0 = _run(orc, q, k, v, CAUSAL_ADDITIVE, zero)
    o1, l1 = _run(orc, q, k, v, CAUSAL_ADDITIVE, c)
    _close(o1, o0, tol=1e-12, what="shift O")
    cs = c[:, :, 0].double().numpy()                                   # (B, Sq)
    want = np.stack([l0[b * Hq + h] + cs[b] for b in range(B) for h in range(Hq)])
    _close(l1, want, tol=1e-12, what="shift LSE")


def pin_key_permutation(orc):
    """Without a causal mask, permuting keys (with V and mask columns) keeps O, LSE."""
    B, Hq, Sq, Sk, D = 1, 3, 7, 13, 8
    q = _rand16((B, Sq, Hq, D), 601)
    k = _rand16((B, Sk, Hq, D), 602)
    v = _rand16((B, Sk, Hq, D), 603)
    mask = _finite_mask(B, Sq, Sk, 604, n_neg_inf=2)
    perm = torch.randperm(Sk, generator=torch.Generator().manual_seed(605))
    o0, l0 = _run(orc, q, k, v, ADDITIVE, mask)
    o1, l1 = _run(orc, q, k[:, perm].contiguous(), v[:, perm].contiguous(), ADDITIVE,
                  mask[:, :, perm].contiguous())
    _close(o1, o0, what="perm O")
    _close(l1, l0, what="perm LSE")


def pin_gqa_equals_mha(orc):
    """GQA equals MHA with each K/V head repeated for its group of query heads."""
    B, Hq, Hkv, S, D = 2, 6, 2, 10, 8
    q = _rand16((B, S, Hq, D), 701)
    k = _rand16((B, S, Hkv, D), 702)
    v = _rand16((B, S, Hkv, D), 703)
    og, lg = _run(orc, q, k, v, CAUSAL)
    ke = k.repeat_interleave(Hq // Hkv, dim=2).contiguous()
    ve = v.repeat_interleave(Hq // Hkv, dim=2).contiguous()
    om, lm = _run(orc, q, ke, ve, CAUSAL)
    assert np.array_equal(og, om) and np.array_equal(lg, lm)


def pin_scale_half(orc):
    """Halving Q and doubling the scale changes nothing (both steps are exact)."""
    B, Hq, S, D = 1, 2, 9, 16
    q = _rand16((B, S, Hq, D), 801)
    k = _rand16((B, S, Hq, D), 802)
    v = _rand16((B, S, Hq, D), 803)
    o0, l0 = _run(orc, q, k, v, CAUSAL, scale=0.2)
    o1, l1 = _run(orc, q * 0.5, k, v, CAUSAL, scale=0.4)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def pin_default_scale(orc):
    """A missing, zero, negative or NaN scale means 1/sqrt(D)."""
    B, Hq, S, D = 1, 1, 5, 16
    q = _rand16((B, S, Hq, D), 901)
    k = _rand16((B, S, Hq, D), 902)
    v = _rand16((B, S, Hq, D), 903)
    ref = _run(orc, q, k, v, NONE, scale=0.25)
    for s in (None, 0.0, -1.0, float("nan"), float("inf")):
        got = _run(orc, q, k, v, NONE, scale=s)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def pin_two_key_closed_form(orc):
    """One query, two keys: o = v1 + (v0 - v1) * sigmoid(s0 - s1), lse in closed form."""
    qv = [1.0, 2.0]
    k0, k1 = [0.5, -1.0], [2.0, 0.25]
    v0, v1 = [3.0, -1.0], [-2.0, 4.0]
    scale = 0.75
    q = torch.tensor(qv).reshape(1, 1, 1, 2).to(torch.bfloat16)
    k = torch.tensor([k0, k1]).reshape(1, 2, 1, 2).to(torch.bfloat16)
    v = torch.tensor([v0, v1]).reshape(1, 2, 1, 2).to(torch.bfloat16)
    o, lse = _run(orc, q, k, v, NONE, scale=scale)
    s0 = scale * (qv[0] * k0[0] + qv[1] * k0[1])       # -1.125
    s1 = scale * (qv[0] * k1[0] + qv[1] * k1[1])       # 1.875
    sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    want = [v1[d] + (v0[d] - v1[d]) * sig for d in range(2)]
    assert np.allclose(o[0, 0], want, rtol=0, atol=1e-14), (o[0, 0], want)
    want_lse = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
    assert abs(lse[0, 0] - want_lse) <= 1e-14


def pin_fully_masked_row(orc):
    """A row whose keys are all -inf in the mask: O = 0, LSE = -inf, no NaN."""
    B, Hq, Sq, Sk, D = 1, 2, 4, 6, 8
    q = _rand16((B, Sq, Hq, D), 1001)
    k = _rand16((B, Sk, Hq, D), 1002)
    v = _rand16((B, Sk, Hq, D), 1003)
    mask = torch.zeros((B, Sq, Sk))
    mask[0, 2, :] = float("-inf")
    o, lse, ps = _run(orc, q, k, v, ADDITIVE, mask, want_psum=True)
    assert np.all(o[:, 2] == 0.0) and np.all(lse[:, 2] == -np.inf) and np.all(ps[:, 2] == 0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(np.delete(lse, 2, axis=1)))


def pin_subset_matches_full(orc):
    """A call on chosen slices and rows returns exactly those entries of the full call."""
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 20, 24, 16
    q = _rand16((B, Sq, Hq, D), 1101)
    k = _rand16((B, Sk, Hkv, D), 1102)
    v = _rand16((B, Sk, Hkv, D), 1103)
    of, lf = _run(orc, q, k, v, CAUSAL)
    sl = [(1, 3), (0, 1), (1, 0)]
    os_, ls = _run(orc, q, k, v, CAUSAL, slices=sl, rows=(5, 17))
    for n, (b, h) in enumerate(sl):
        assert np.array_equal(os_[n], of[b * Hq + h, 5:17])
        assert np.array_equal(ls[n], lf[b * Hq + h, 5:17])


def _rope_py(t, pos0, base):
    """Rotate a (B, S, H, D) tensor in pure Python: pair (2i, 2i+1) of the vector
    at sequence index s turns by (pos0 + s) * base ** (-2 i / D)."""
    x = t.double().tolist()
    B, S, H, D = t.shape
    for b in range(B):
        for si in range(S):
            ang0 = pos0 + si
            for h in range(H):
                v = x[b][si][h]
                for i in range(D // 2):
                    th = ang0 * base ** (-2.0 * i / D)
                    c, sn = math.cos(th), math.sin(th)
                    a, bb = v[2 * i], v[2 * i + 1]
                    v[2 * i], v[2 * i + 1] = a * c - bb * sn, bb * c + a * sn
    return torch.tensor(x, dtype=torch.float64)


def pin_rope_brute_force(orc):
    """With rotary embedding: oracle == rotate (pure Python) then brute-force attention."""
    for n, (B, Hq, Hkv, Sq, Sk, D, kind, qp, kp) in enumerate([
            (1, 2, 2, 5, 7, 8, NONE, 0, 0),
            (2, 4, 2, 4, 9, 8, CAUSAL, 5, 0),
            (1, 2, 1, 6, 6, 4, CAUSAL_ADDITIVE, 3, 3)]):
        q = _rand16((B, Sq, Hq, D), 1200 + n)
        k = _rand16((B, Sk, Hkv, D), 1210 + n)
        v = _rand16((B, Sk, Hkv, D), 1220 + n)
        mask = _finite_mask(B, Sq, Sk, 1230 + n, n_neg_inf=1) if kind >= ADDITIVE else None
        o, lse = _run(orc, q, k, v, kind, mask, rope_base=10000.0, q_pos0=qp, k_pos0=kp)
        ob, lb = _brute(_rope_py(q, qp, 10000.0), _rope_py(k, kp, 10000.0), v, kind, mask, 1.0 / math.sqrt(D))
        _close(o, ob, tol=1e-11, what=f"rope brute {n} O")
        _close(lse, lb, tol=1e-11, what=f"rope brute {n} LSE")


def pin_rope_two_dim_closed_form(orc):
    """D = 2 (one pair, frequency 1): q = (1, 0) at position p, k = (1, 0) at position p'
    gives the single logit scale * cos(p' - p), so lse = scale * cos(p' - p)."""
    q = torch.tensor([1.0, 0.0]).reshape(1, 1, 1, 2).to(torch.bfloat16)
    k = torch.tensor([1.0, 0.0]).reshape(1, 1, 1, 2).to(torch.bfloat16)
    v = torch.tensor([0.5, -2.0]).reshape(1, 1, 1, 2).to(torch.bfloat16)
    for qp, kp in ((3, 10), (10, 3), (0, 0)):
        o, lse = _run(orc, q, k, v, NONE, scale=0.5, rope_base=10000.0, q_pos0=qp, k_pos0=kp)
        assert abs(lse[0, 0] - 0.5 * math.cos(kp - qp)) <= 1e-14
        assert np.array_equal(o[0, 0], [0.5, -2.0])


def pin_rope_depends_on_relative_position(orc):
    """Shifting every query and key position by the same amount changes nothing."""
    B, Hq, Sq, Sk, D = 1, 2, 6, 9, 16
    q = _rand16((B, Sq, Hq, D), 1301)
    k = _rand16((B, Sk, Hq, D), 1302)
    v = _rand16((B, Sk, Hq, D), 1303)
    o0, l0 = _run(orc, q, k, v, CAUSAL, rope_base=10000.0, q_pos0=3, k_pos0=0)
    o1, l1 = _run(orc, q, k, v, CAUSAL, rope_base=10000.0, q_pos0=40, k_pos0=37)
    _close(o1, o0, tol=1e-10, what="rope shift O")
    _close(l1, l0, tol=1e-10, what="rope shift LSE")
    o2, _ = _run(orc, q, k, v, CAUSAL, rope_base=10000.0, q_pos0=4, k_pos0=0)
    assert not np.allclose(o2, o0, atol=1e-6)          # a different offset does change it


def pin_rope_position_zero_is_identity(orc):
    """A single query and key both at position 0: the rotation is the identity."""
    q = _rand16((1, 1, 2, 16), 1401)
    k = _rand16((1, 1, 2, 16), 1402)
    v = _rand16((1, 1, 2, 16), 1403)
    assert all(np.array_equal(a, b) for a, b in zip(_run(orc, q, k, v, NONE, rope_base=10000.0),
                                                    _run(orc, q, k, v, NONE)))


def _held_in(t64, dtype):
    """Round a float64 tensor to the 16-bit type with PyTorch's own conversion."""
    return t64.to(torch.bfloat16 if dtype == "bf16" else torch.float16).double()


def pin_rope_round_brute_force(orc):
    """rope_round: oracle == rotate (pure Python), round with PyTorch's 16-bit
    conversion, then brute-force attention; bf16 and fp16."""
    for n, (B, Hq, Hkv, Sq, Sk, D, kind, qp, kp, dt) in enumerate([
            (1, 2, 2, 5, 7, 8, NONE, 0, 0, "bf16"),
            (2, 4, 2, 4, 9, 8, CAUSAL, 5, 2, "bf16"),
            (1, 2, 1, 6, 6, 4, CAUSAL, 30, 27, "f16")]):
        tdt = torch.bfloat16 if dt == "bf16" else torch.float16
        q = _rand16((B, Sq, Hq, D), 1500 + n, dtype=tdt)
        k = _rand16((B, Sk, Hkv, D), 1510 + n, dtype=tdt)
        v = _rand16((B, Sk, Hkv, D), 1520 + n, dtype=tdt)
        o, lse = _run(orc, q, k, v, kind, None, dtype=dt, rope_base=10000.0, q_pos0=qp, k_pos0=kp,
                      rope_round=True)
        ob, lb = _brute(_held_in(_rope_py(q, qp, 10000.0), dt), _held_in(_rope_py(k, kp, 10000.0), dt), v,
                        kind, None, 1.0 / math.sqrt(D))
        _close(o, ob, tol=1e-11, what=f"rope round brute {n} O")
        _close(lse, lb, tol=1e-11, what=f"rope round brute {n} LSE")


def pin_rope_round_single_key_closed_form(orc):
    """D = 2, one key (1, 0) at position 0 (no rotation) and the query (1, 0) at
    position p: the only logit is scale * q_rot[0], and q_rot[0] is cos(p) held
    in the 16-bit type, so lse = scale * round16(cos p) and o = v."""
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        one = torch.tensor([1.0, 0.0]).reshape(1, 1, 1, 2).to(tdt)
        v = torch.tensor([0.25, -3.0]).reshape(1, 1, 1, 2).to(tdt)
        for p in (1, 2, 5, 7, 11, 20, 33, 100):
            o, lse = _run(orc, one, one, v, NONE, scale=1.0, dtype=dt, rope_base=10000.0, q_pos0=p,
                          k_pos0=0, rope_round=True)
            want = float(torch.tensor(math.cos(p), dtype=torch.float64).to(tdt).double())
            assert lse[0, 0] == want, (dt, p, lse[0, 0], want)
            assert np.array_equal(o[0, 0], [0.25, -3.0])


def pin_rope_rotate_alone(orc):
    """The rotation on its own equals the pure-Python rotation (exact), and
    PyTorch's 16-bit conversion of it (rope_round), for bf16 and fp16."""
    for n, (dt, tdt, pos0) in enumerate((("bf16", torch.bfloat16, 0), ("f16", torch.float16, 77))):
        x = _rand16((2, 5, 3, 8), 1600 + n, dtype=tdt)
        exact = _rope_py(x, pos0, 10000.0)
        _close(orc.rotate(_bits(x), base=10000.0, pos0=pos0, dtype=dt, rope_round=False), exact.numpy(),
               tol=1e-14, what=f"rotate exact {dt}")
        got = orc.rotate(_bits(x), base=10000.0, pos0=pos0, dtype=dt, rope_round=True)
        assert np.array_equal(got, _held_in(exact, dt).numpy()), f"rotate rounded {dt}"


ALL_PINS = [
    pin_brute_force, pin_brute_force_f16, pin_widening_exact, pin_sdpa_float64,
    pin_rowsum_one, pin_constant_v, pin_zero_q, pin_causal_row0, pin_shift_invariance,
    pin_key_permutation, pin_gqa_equals_mha, pin_scale_half, pin_default_scale,
    pin_two_key_closed_form, pin_fully_masked_row, pin_subset_matches_full,
    pin_rope_brute_force, pin_rope_two_dim_closed_form, pin_rope_depends_on_relative_position,
    pin_rope_position_zero_is_identity, pin_rope_round_brute_force, pin_rope_round_single_key_closed_form,
    pin_rope_rotate_alone,
]
