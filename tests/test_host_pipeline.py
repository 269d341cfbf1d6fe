"""GPU tests of the host-buffer entry points (attn_fwd_host / attn_fwd_host_f16):
Q, K, V, the mask, O and LSE in host memory, computed in a pipeline of
(batch entry, K/V-head group) units through device staging slots. Each unit is
an independent launch of the same fused kernel, so the results must equal the
all-on-device call bit for bit; one case is also checked against the oracle.
Covers several units per entry and several entries, GQA and MQA groups, fp16,
the additive mask (staged once per entry), an empty key sequence, pageable
host memory, and repeated calls on one workspace."""
import pytest
import torch

from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, Sq, Sk, D, mask kind, dtype
    (4, 8, 8, 300, 300, 128, 1, "bf16"),       # 2 groups per entry: 8 units, three slots reused
    (1, 16, 4, 200, 700, 64, 3, "f16"),        # one entry, 4 K/V-head units, causal + additive mask
    (3, 2, 1, 129, 129, 128, 2, "bf16"),       # MQA, one unit per entry, additive mask
    (2, 4, 2, 64, 0, 128, 1, "bf16"),          # no keys: o = 0, lse = -inf
]


def _bits(t):
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.float16) else t


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_D{}_m{}_{}".format(*c))
@pytest.mark.parametrize("pinned", [True, False])
def test_host_pipeline_equals_device_call(case, pinned):
    B, Hq, Hkv, Sq, Sk, D, kind, dtype = case
    cfg = I.AttnConfig("host", B, Hq, Hkv, Sq, Sk, D, causal=bool(kind & 1), additive_mask=bool(kind & 2),
                       seed=sum(case[:7]), dtype=dtype)
    q, k, v, mask = I.make_inputs(cfg)
    dev = torch.device("cuda")
    ref_o, ref_l = A.attention(q.to(dev), k.to(dev), v.to(dev), causal=cfg.causal,
                               mask=None if mask is None else mask.to(dev))
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
        mask = None if mask is None else mask.pin_memory()
    o, lse = A.attention_host(q, k, v, causal=cfg.causal, mask=mask)
    torch.cuda.synchronize()
    assert torch.equal(_bits(o), _bits(ref_o.cpu()))
    assert torch.equal(lse, ref_l.cpu())


def test_host_pipeline_matches_oracle_and_reuses_its_workspace():
    cfg = I.AttnConfig("host2", 2, 8, 2, 384, 512, 128, causal=True, seed=5)
    q, k, v, _ = I.make_inputs(cfg)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    need = A.attn_fwd_host_workspace_bytes(2, 8, 2, 384, 512, 128, cfg.mask_kind)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):                                       # back-to-back calls on one workspace
        outs.append(A.attention_host(q, k, v, causal=True, workspace=ws))
    torch.cuda.synchronize()
    for o, lse in outs[1:]:
        assert torch.equal(_bits(o), _bits(outs[0][0])) and torch.equal(lse, outs[0][1])
    check(outs[0][0], outs[0][1], q, k, v, None, cfg.mask_kind, label="host pipeline")
