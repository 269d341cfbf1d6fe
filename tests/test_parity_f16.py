"""GPU parity of the fp16 entry point (attn_fwd_f16) against the FP64 oracle's
fp16 path: small shapes element by element (both head dimensions, every mask
kind, GQA/MQA, ragged tails, Sq != Sk) and the stress value sets at full size
on sampled slices."""
import pytest
import torch

from gpu_helpers import check, full_scan, run_gpu
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = [
    (1, 2, 2, 128, 128, 64, 1),
    (2, 8, 2, 300, 300, 128, 1),
    (1, 4, 1, 257, 513, 128, 0),
    (1, 4, 4, 300, 200, 64, 1),
    (2, 2, 2, 384, 384, 128, 2),
    (1, 4, 2, 300, 260, 64, 3),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B{}_H{}-{}_S{}-{}_D{}_m{}".format(*c))
def test_f16_small_shapes_match_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, kind = case
    cfg = I.AttnConfig("f16", B, Hq, Hkv, Sq, Sk, D, causal=bool(kind & 1), additive_mask=bool(kind & 2),
                       seed=sum(case), dtype="f16")
    q, k, v, mask = I.make_inputs(cfg)
    assert q.dtype == torch.float16
    o, lse = run_gpu(q, k, v, mask, cfg.causal)
    assert o.dtype == torch.float16
    check(o, lse, q, k, v, mask, cfg.mask_kind, label=f"f16 {case}")


@pytest.mark.parametrize("values", ["zero_q", "saturated", "student_t2"])
def test_f16_stress_sets_sampled(values):
    cfg = I.CONFIGS[f"stress_d128_{values}"].with_(dtype="f16")
    q, k, v, mask = I.make_inputs(cfg)
    o, lse = run_gpu(q, k, v, mask, cfg.causal)
    full_scan(o, lse)
    check(o, lse, q, k, v, mask, cfg.mask_kind, slices=[(0, 0), (1, 15)],
          heavy_tail=(values == "student_t2"), label=f"f16 {values}")


def test_f16_and_bf16_entry_points_are_distinct():
    """The same bits interpreted as fp16 and as bf16 must give the two different answers."""
    cfg = I.AttnConfig("x", 1, 2, 2, 128, 128, 64, causal=True, seed=4, dtype="f16")
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    o16, _ = A.attention(q.to(dev), k.to(dev), v.to(dev), causal=True)
    ob, _ = A.attention(q.view(torch.bfloat16).to(dev), k.view(torch.bfloat16).to(dev),
                        v.view(torch.bfloat16).to(dev), causal=True)
    assert not torch.equal(o16.view(torch.int16), ob.view(torch.int16))
