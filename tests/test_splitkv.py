"""GPU parity of the split-key entry points against the FP64 oracle: decode
and short-prefill shapes over long key sequences, ragged ranges, causal cuts
that leave whole ranges empty for some rows, the additive mask, fp16, and the
split result against the unsplit one."""
import pytest
import torch

from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, Sq, Sk, D, mask kind, num_splits
    (1, 16, 4, 1, 8192, 128, 1, 0),        # GQA decode, automatic split
    (2, 8, 8, 16, 8192, 64, 1, 0),
    (1, 8, 1, 1, 1000, 128, 0, 3),         # MQA, ragged ranges 3+3+2 blocks
    (1, 4, 2, 200, 1000, 128, 3, 4),       # causal + additive, some ranges empty for early rows
    (1, 2, 2, 400, 300, 64, 1, 2),         # Sq > Sk: rows with no key at all
    (4, 32, 8, 1, 4096, 128, 1, 2),        # batched GQA decode, two ranges
    (2, 4, 4, 64, 2100, 128, 2, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_D{}_m{}_s{}".format(*c))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_splitkv_matches_oracle(case, dtype):
    B, Hq, Hkv, Sq, Sk, D, kind, ns = case
    cfg = I.AttnConfig("split", B, Hq, Hkv, Sq, Sk, D, causal=bool(kind & 1), additive_mask=bool(kind & 2),
                       seed=sum(case), dtype=dtype)
    q, k, v, mask = I.make_inputs(cfg)
    dev = torch.device("cuda")
    o, lse = A.attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=cfg.causal,
                                 mask=None if mask is None else mask.to(dev), num_splits=ns)
    torch.cuda.synchronize()
    assert A.attn_splitkv_num_splits(B, Hq, Hkv, Sq, Sk, ns) > 1
    check(o, lse, q, k, v, mask, cfg.mask_kind, label=f"split {case} {dtype}")


def test_split_equals_unsplit_within_rounding():
    cfg = I.AttnConfig("s", 2, 8, 2, 512, 3000, 128, causal=True, seed=9)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = A.attention(qd, kd, vd, causal=True)
    o2, l2 = A.attention_splitkv(qd, kd, vd, causal=True, num_splits=5)
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2
    assert float(((l1 - l2).abs() / l1.abs().clamp(min=1)).max()) <= 1e-4


def test_splitkv_with_caller_workspace_allocates_nothing():
    cfg = I.AttnConfig("d", 4, 32, 8, 1, 4096, 128, causal=True, seed=2)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    need = A.attn_splitkv_workspace_bytes(4, 32, 8, 1, 4096, 128, 0)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((4, 32, 1), device=dev)
    A.attention_splitkv(qd, kd, vd, causal=True, workspace=ws, out=o, lse=lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(50):
        A.attention_splitkv(qd, kd, vd, causal=True, workspace=ws, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert A.attn_last_status(torch.cuda.current_stream().cuda_stream) == A.ATTN_OK


def test_splitkv_rejects_small_workspace_on_device():
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 4, 128), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 4096, 4, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(1024, dtype=torch.uint8, device=dev)
    with pytest.raises(A.AttnError) as e:
        A.attention_splitkv(q, k, k, num_splits=8, workspace=ws)
    assert e.value.code == A.ATTN_ERR_INVALID_ARG
