"""GPU behaviour of the C ABI: invariants the definition fixes, checked on the
kernel's own outputs, plus determinism, complete writes, empty inputs,
argument checks with real device pointers, streams and allocation."""
import math

import pytest
import torch

from gpu_helpers import run_gpu
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(name="b", B=2, Hq=8, Hkv=2, Sq=384, Sk=384, D=128, causal=True, seed=11)
    base.update(kw)
    return I.AttnConfig(**base)


def test_gqa_equals_expanded_mha_bitwise():
    cfg = _cfg()
    q, k, v, _ = I.make_inputs(cfg)
    og, lg = run_gpu(q, k, v, None, True)
    g = cfg.Hq // cfg.Hkv
    om, lm = run_gpu(q, k.repeat_interleave(g, dim=2).contiguous(), v.repeat_interleave(g, dim=2).contiguous(),
                     None, True)
    assert torch.equal(og, om) and torch.equal(lg, lm)


def test_run_to_run_bitwise_deterministic():
    cfg = _cfg(D=64, Sq=777, Sk=777, causal=False)
    q, k, v, _ = I.make_inputs(cfg)
    o1, l1 = run_gpu(q, k, v, None, False)
    o2, l2 = run_gpu(q, k, v, None, False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_every_output_element_written():
    cfg = _cfg(Sq=300, Sk=300)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((cfg.B, cfg.Hq, cfg.Sq), float("nan"), device=dev)
    A.attention(q.to(dev), k.to(dev), v.to(dev), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(o).any()) and not bool(torch.isnan(lse).any())


def test_constant_v_gives_constant_o():
    cfg = _cfg()
    q, k, _, _ = I.make_inputs(cfg)
    v = torch.full((cfg.B, cfg.Sk, cfg.Hkv, cfg.D), 1.5, dtype=torch.bfloat16)
    o, _ = run_gpu(q, k, v, None, True)
    assert float((o.float() - 1.5).abs().max()) <= 2e-2


def test_causal_row_zero_is_v_zero():
    cfg = _cfg(Hkv=8)
    q, k, v, _ = I.make_inputs(cfg)
    o, lse = run_gpu(q, k, v, None, True, scale=0.1)
    assert torch.equal(o[:, 0].cpu(), v[:, 0])
    s00 = 0.1 * (q[:, 0].double() * k[:, 0].double()).sum(-1)          # (B, H)
    err = (lse[:, :, 0].double().cpu() - s00).abs() / s00.abs().clamp(min=1.0)
    assert float(err.max()) <= 1e-3


def test_row_shift_through_mask_keeps_o_and_moves_lse():
    cfg = _cfg(Sq=256, Sk=320, causal=False)
    q, k, v, _ = I.make_inputs(cfg)
    zero = torch.zeros((cfg.B, cfg.Sq, cfg.Sk))
    c = torch.linspace(-20.0, 20.0, cfg.B * cfg.Sq).reshape(cfg.B, cfg.Sq, 1).expand(-1, -1, cfg.Sk).contiguous()
    o0, l0 = run_gpu(q, k, v, zero, False)
    o1, l1 = run_gpu(q, k, v, c, False)
    assert float((o0.float() - o1.float()).abs().max()) <= 2e-2
    want = l0.cpu() + c[:, None, :, 0]
    assert float(((l1.cpu() - want).abs() / want.abs().clamp(min=1.0)).max()) <= 1e-3


def test_zero_length_keys_give_empty_rows():
    cfg = _cfg(Sk=0)
    q, k, v, _ = I.make_inputs(cfg)
    o, lse = run_gpu(q, k, v, None, False)
    assert bool((o == 0).all()) and bool((lse == float("-inf")).all())


def test_empty_batch_writes_nothing():
    dev = torch.device("cuda")
    q = torch.zeros((0, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    o, lse = A.attention(q, q, q)
    assert o.shape == q.shape and lse.shape == (0, 2, 16)


def test_misaligned_device_pointer_is_rejected():
    dev = torch.device("cuda")
    buf = torch.zeros(4 * 64 * 2 * 64 + 8, dtype=torch.bfloat16, device=dev)
    p = buf.data_ptr() + 2
    o = torch.empty((1, 64, 2, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 2, 64), device=dev)
    rc = A.attn_fwd(p, p, p, o.data_ptr(), lse.data_ptr(), 1, 2, 2, 64, 64, 64, 0.0, 0, None,
                    torch.cuda.current_stream().cuda_stream)
    assert rc == A.ATTN_ERR_INVALID_ARG


def test_side_stream_and_status():
    cfg = _cfg(D=64)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ref_o, ref_l = A.attention(qd, kd, vd, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, l = A.attention(qd, kd, vd, causal=True, stream=s)
    assert A.attn_last_status(s.cuda_stream) == A.ATTN_OK
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_library_allocates_no_device_memory():
    cfg = _cfg()
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), device=dev)
    A.attention(qd, kd, vd, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(100):
        A.attention(qd, kd, vd, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0


def test_default_scale_is_inverse_sqrt_d():
    cfg = _cfg(D=64, causal=False)
    q, k, v, _ = I.make_inputs(cfg)
    o1, l1 = run_gpu(q, k, v, None, False, scale=None)
    o2, l2 = run_gpu(q, k, v, None, False, scale=1.0 / math.sqrt(64))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_output_aligned_to_16_but_not_32_bytes():
    """O at an address that is 16-byte but not 32-byte aligned (the narrower store path)."""
    cfg = _cfg(Sq=200, Sk=200)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ref_o, ref_l = A.attention(qd, kd, vd, causal=True)
    buf = torch.zeros(qd.numel() + 16, dtype=torch.bfloat16, device=dev)
    off = 8 if (buf.data_ptr() % 32 == 0) else 0          # 8 bf16 = 16 bytes
    o = buf[off:off + qd.numel()].view(qd.shape)
    assert o.data_ptr() % 16 == 0 and o.data_ptr() % 32 != 0
    lse = torch.empty_like(ref_l)
    A.attention(qd, kd, vd, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
