"""The allocation-free split-key entry point, attn_fwd_splitkv_noalloc.

It serves callers that may not allocate device memory themselves (a plug-in
inside a framework that owns all device memory, a latency-critical path that
cannot afford cudaMalloc); its scratch is the library's fixed 32 MiB device
array. These tests call it through the C ABI, twice in a row with different
problems, and compare each result with the existing split-key entry point
given its own workspace, within the tolerances the parity tests use. This file
is collected last so that a run stopping at its first failure has already run
every other test; it also passes on its own in a fresh process (the first call
there sets up the scratch address).
"""
import pytest
import torch

from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _raw_noalloc(qd, kd, vd, o, lse, cfg, num_splits, mask=None):
    return A.attn_fwd_splitkv_noalloc(
        qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
        cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, cfg.D, float("nan"), cfg.mask_kind,
        None if mask is None else mask.data_ptr(), num_splits, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    """The first problem fills most of the scratch array; the second, smaller
    one then runs over the first one's leftovers and is also compared with the
    FP64 oracle, so a partial result read before it was written would show."""
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    problems = [
        (I.AttnConfig("a", 2, 16, 4, 200, 4096, 128, causal=True, seed=21), 8),     # 26 MB of partials
        (I.AttnConfig("b", 1, 8, 2, 96, 3000, 128, causal=True, seed=22), 5),       # short prefill, ragged
    ]
    for idx, (cfg, ns) in enumerate(problems):
        assert A.attn_splitkv_num_splits(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, ns) > 1
        assert A.attn_splitkv_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, cfg.D, ns) <= 32 << 20
        q, k, v, _ = I.make_inputs(cfg)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        ref_o, ref_l = A.attention_splitkv(qd, kd, vd, causal=cfg.causal, num_splits=ns)
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((cfg.B, cfg.Hq, cfg.Sq), float("nan"), device=dev)
        assert _raw_noalloc(qd, kd, vd, o, lse, cfg, ns) == A.ATTN_OK
        assert A.attn_last_status(stream) == A.ATTN_OK
        assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
        err = (o.float() - ref_o.float()).abs()
        assert float(err.max()) <= 2e-2 and float(err.mean()) <= 2e-3
        assert float(((lse - ref_l).abs() / ref_l.abs().clamp(min=1.0)).max()) <= 1e-3
        if idx == 1:
            check(o, lse, q, k, v, None, cfg.mask_kind, label="noalloc vs oracle")


def test_noalloc_allocates_nothing_per_call():
    cfg = I.AttnConfig("c", 2, 16, 4, 1, 4096, 128, causal=True, seed=23)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), device=dev)
    assert _raw_noalloc(qd, kd, vd, o, lse, cfg, 4) == A.ATTN_OK       # first call: address set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        assert _raw_noalloc(qd, kd, vd, o, lse, cfg, 4) == A.ATTN_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_refuses_a_problem_beyond_its_scratch():
    cfg = I.AttnConfig("d", 4, 32, 32, 2048, 2048, 128, causal=True)   # 4 ranges need 128+ MiB
    assert A.attn_splitkv_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, cfg.D, 4) > 32 << 20
    dev = torch.device("cuda")
    qd = torch.zeros((cfg.B, cfg.Sq, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    o = torch.full_like(qd, 7.0)
    lse = torch.full((cfg.B, cfg.Hq, cfg.Sq), 7.0, device=dev)
    assert _raw_noalloc(qd, qd, qd, o, lse, cfg, 4) == A.ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())          # nothing was launched
