"""GPU parity of GQA head packing (decode and short prefills): the query heads
of a K/V head share each tile's rows when Hq/Hkv is a power of two and
Sq * Hq/Hkv <= 256. Cases cover group sizes 2 to 32 (MQA included), one and
both 128-row sub-tiles in use, the exact size limit, causal alignment with
several query rows, the additive mask, fp16, D = 64, and the single-pass and
split-key entry points, all against the FP64 oracle."""
import pytest
import torch

from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, Sq, Sk, D, mask kind, dtype, splits (None: single pass)
    (4, 32, 8, 1, 4096, 128, 1, "bf16", 0),      # decode, G = 4, automatic split
    (2, 32, 8, 1, 1000, 128, 1, "bf16", None),   # single pass, ragged keys
    (1, 8, 1, 1, 3000, 128, 1, "bf16", 0),       # MQA, G = 8
    (2, 32, 1, 3, 777, 64, 1, "bf16", 5),        # G = 32 (4 rows per sub-tile), D = 64
    (2, 16, 8, 60, 500, 128, 1, "bf16", None),   # G = 2, 60 rows: both sub-tiles (64 rows each)
    (1, 16, 4, 64, 900, 128, 1, "f16", 3),       # Sq * G = 256: the limit, both sub-tiles full
    (2, 8, 2, 20, 300, 128, 3, "bf16", None),    # causal + additive mask, G = 4
    (1, 4, 2, 7, 129, 64, 2, "f16", 2),          # additive mask only, G = 2
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_D{}_m{}_{}_s{}".format(*c))
def test_packed_heads_match_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, kind, dtype, ns = case
    assert (Hq // Hkv) & (Hq // Hkv - 1) == 0 and Sq * (Hq // Hkv) <= 256      # the packed regime
    cfg = I.AttnConfig("pack", B, Hq, Hkv, Sq, Sk, D, causal=bool(kind & 1), additive_mask=bool(kind & 2),
                       seed=sum(case[:7]), dtype=dtype)
    q, k, v, mask = I.make_inputs(cfg)
    dev = torch.device("cuda")
    m = None if mask is None else mask.to(dev)
    if ns is None:
        o, lse = A.attention(q.to(dev), k.to(dev), v.to(dev), causal=cfg.causal, mask=m)
    else:
        o, lse = A.attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=cfg.causal, mask=m, num_splits=ns)
    torch.cuda.synchronize()
    check(o, lse, q, k, v, mask, cfg.mask_kind, label=f"packed {case}")


def test_long_kv_cache_decode():
    """One query row against 262,144 cached keys (MQA, 8 query heads packed
    into one tile per sequence, automatic key ranges)."""
    cfg = I.AttnConfig("long_decode", 1, 8, 1, 1, 262144, 128, causal=True, seed=41)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    assert A.attn_splitkv_num_splits(1, 8, 1, 1, 262144, 0) > 1
    o, lse = A.attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=True, num_splits=0)
    torch.cuda.synchronize()
    check(o, lse, q, k, v, None, cfg.mask_kind, label="262k-key decode")


def test_host_pipeline_on_packed_decode():
    cfg = I.AttnConfig("host_decode", 4, 32, 8, 1, 2048, 128, causal=True, seed=43, dtype="f16")
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    ref_o, ref_l = A.attention(q.to(dev), k.to(dev), v.to(dev), causal=True)
    o, lse = A.attention_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_o.cpu().view(torch.int16)) and torch.equal(lse, ref_l.cpu())
    check(o, lse, q, k, v, None, cfg.mask_kind, label="host pipeline, packed decode")
