"""GPU parity of the rotary-embedding path against the FP64 oracle: the angle
table, the key rotation kernel, and attention with the queries rotated inside
the attention kernel at tile load ("ATB engineering guide" §4.1 fusion
pattern 5; interleaved pairs and base 10000 as in its §8.4). Covers GQA/MQA,
ragged lengths, query and key position offsets (chunked prefill, decode),
both head dimensions, fp16, the additive mask, split keys, the three ways of
supplying the keys (rotated here, rotated in place, already rotated) and a
Llama-2-7B-shaped prefill checked on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

BASE = 10000.0


def _table(max_pos, D):
    t = A.rope_table(max_pos, D, BASE)
    torch.cuda.synchronize()
    return t


def test_table_matches_double_precision_angles():
    for D in (64, 128):
        max_pos = 4099
        t = _table(max_pos, D).cpu().numpy().astype(np.float64)
        pos = np.arange(max_pos, dtype=np.float64)[:, None]
        i = np.arange(D // 2, dtype=np.float64)[None, :]
        theta = pos * BASE ** (-2.0 * i / D)
        # each entry is cos / sin of the double angle rounded to FP32: within
        # half an FP32 ulp of 1 plus a few double ulps of the trigonometry
        assert np.abs(t[..., 0] - np.cos(theta)).max() <= 6.0e-8
        assert np.abs(t[..., 1] - np.sin(theta)).max() <= 6.0e-8


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
def test_key_rotation_matches_oracle(dtype, D):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    g = torch.Generator().manual_seed(D + len(dtype))
    x = (torch.randn((2, 333, 4, D), generator=g) * 2.0).to(tdt)
    pos0 = 17
    table = _table(pos0 + 333, D)
    xd = x.cuda()
    y = A.rope_apply(xd, table, pos0=pos0)
    torch.cuda.synchronize()
    want = oracle.default().rotate(I.bits(x), base=BASE, pos0=pos0, dtype=dtype, rope_round=True)
    got = y.double().cpu().numpy()
    # The kernel rotates in FP32 and rounds once; the oracle rotates exactly and
    # rounds once. They agree except where the FP32 result and the exact one
    # straddle a rounding boundary (one unit in the last place), or where the
    # pair nearly cancels and the FP32 error of the products, a few 2^-24 of
    # the pair's magnitude, exceeds the 16-bit spacing of the tiny result.
    mag = np.maximum(np.abs(want), np.abs(got))
    ulp = np.spacing(mag.astype(np.float16 if dtype == "f16" else np.float32)).astype(np.float64)
    if dtype == "bf16":
        ulp = ulp * 65536.0                   # bf16 keeps 16 fewer fraction bits than FP32
    xin = np.abs(x.double().numpy()).reshape(*x.shape[:-1], D // 2, 2).max(axis=-1)
    fp32_err = 4.0 * 2.0 ** -24 * np.repeat(xin, 2, axis=-1)
    diff = np.abs(got - want)
    assert np.all(diff <= ulp + fp32_err), float((diff / (ulp + fp32_err)).max())
    assert np.count_nonzero(diff) <= max(4, diff.size // 1000)
    # in place gives the same bytes
    A.rope_apply(xd, table, pos0=pos0, out=xd)
    torch.cuda.synchronize()
    assert torch.equal(xd.view(torch.int16), y.view(torch.int16))


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, mask kind, q_pos0, k_pos0, num_splits, dtype
    (2, 8, 2, 300, 300, 128, 1, 0, 0, 1, "bf16"),        # GQA causal prefill, ragged tail
    (1, 4, 4, 200, 456, 128, 1, 256, 0, 1, "bf16"),      # chunked prefill: queries continue at 256
    (1, 4, 1, 1, 3000, 128, 1, 2999, 0, 0, "bf16"),      # MQA decode, automatic split
    (2, 4, 2, 130, 520, 64, 0, 5, 3, 1, "f16"),          # no mask, offsets, fp16, D = 64
    (1, 2, 2, 100, 260, 128, 3, 160, 0, 1, "bf16"),      # causal + additive mask
    (1, 2, 2, 600, 600, 128, 2, 0, 0, 1, "f16"),         # additive mask: both sub-tiles' O staged, ragged tail
    (1, 8, 8, 600, 600, 64, 1, 0, 0, 1, "bf16"),
    (2, 16, 4, 8, 2048, 128, 1, 2040, 0, 4, "f16"),      # short prefill over a cache, four ranges
    (1, 4, 2, 300, 400, 64, 2, 7, 3, 1, "bf16"),         # additive mask at D = 64, GQA, offsets
    (1, 2, 2, 161, 161, 128, 1, 0, 0, 1, "bf16"),        # upper sub-tile rows end inside the second rotating warp's rows
]


def _inputs(case):
    B, Hq, Hkv, Sq, Sk, D, kind, qp, kp, ns, dtype = case
    cfg = I.AttnConfig("rope", B, Hq, Hkv, Sq, Sk, D, causal=bool(kind & 1), additive_mask=bool(kind & 2),
                       seed=sum(case[:10]), dtype=dtype)
    return cfg, I.make_inputs(cfg)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_D{}_m{}_p{}-{}_s{}_{}".format(*c))
def test_rope_attention_matches_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, kind, qp, kp, ns, dtype = case
    cfg, (q, k, v, mask) = _inputs(case)
    table = _table(max(qp + Sq, kp + Sk), D)
    dev = torch.device("cuda")
    o, lse, _ = A.attention_rope(q.to(dev), k.to(dev), v.to(dev), table, q_pos0=qp, k_pos0=kp,
                                 causal=cfg.causal, mask=None if mask is None else mask.to(dev), num_splits=ns)
    torch.cuda.synchronize()
    check(o, lse, q, k, v, mask, cfg.mask_kind, label=f"rope {case}",
          rope=dict(base=BASE, q_pos0=qp, k_pos0=kp))


def test_key_supply_modes_agree_bitwise():
    case = (2, 8, 2, 333, 700, 128, 1, 100, 0, 1, "bf16")
    B, Hq, Hkv, Sq, Sk, D, kind, qp, kp, ns, dtype = case
    cfg, (q, k, v, _) = _inputs(case)
    table = _table(800, D)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1, krot = A.attention_rope(qd, kd, vd, table, q_pos0=qp, k_pos0=kp, causal=True)      # rotated here
    kpre = A.rope_apply(kd, table, pos0=kp)                                                    # a rotated cache
    o2, l2 = A.attention_rope(qd, kpre, vd, table, q_pos0=qp, k_rot=None, causal=True)
    kin = kd.clone()
    o3, l3, _ = A.attention_rope(qd, kin, vd, table, q_pos0=qp, k_pos0=kp, k_rot=kin, causal=True)  # in place
    torch.cuda.synchronize()
    assert torch.equal(krot, kpre) and torch.equal(kin, kpre)
    for o, l in ((o2, l2), (o3, l3)):
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(l, l1)
    # and rotating nothing (all positions 0 for a single query and key row) is plain attention
    q1, k1, v1 = qd[:, :1].contiguous(), kd[:, :1].contiguous(), vd[:, :1].contiguous()
    o4, l4, _ = A.attention_rope(q1, k1, v1, table, causal=True)
    o5, l5 = A.attention(q1, k1, v1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o4.view(torch.int16), o5.view(torch.int16)) and torch.equal(l4, l5)


def test_llama2_7b_shaped_prefill_sampled():
    """B=4, S=2048, 32 heads, D=128, causal, positions from 0: sampled slices
    and row windows (first tile, a middle tile boundary, the last rows)."""
    cfg = I.AttnConfig("l7b_rope", 4, 32, 32, 2048, 2048, 128, causal=True, seed=77)
    q, k, v, _ = I.make_inputs(cfg)
    table = _table(2048, 128)
    dev = torch.device("cuda")
    o, lse, _ = A.attention_rope(q.to(dev), k.to(dev), v.to(dev), table, causal=True)
    torch.cuda.synchronize()
    slices = [(0, 0), (1, 17), (3, 31)]
    for rows in ((0, 40), (1010, 1050), (2000, 2048)):
        check(o, lse, q, k, v, None, cfg.mask_kind, slices=slices, rows=rows, label=f"l7b rope {rows}",
              rope=dict(base=BASE, q_pos0=0, k_pos0=0))
