"""GPU parity of the attention block and its parts against the FP64 oracle
(oracle/attn_block.py and the compiled attention oracle): the tensor-core
projection GEMM (bias, residual, ragged M, K tails, several tiles per CTA),
the LayerNorm, attention on a packed QKV tensor, and the whole block (MHA and
GQA, both head sizes, causal and not), including one Llama-2-7B-sized layer
(hidden 4096, 32 heads) on one 2048-token sequence."""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import check
from oracle import attn_block as OB
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _f64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("M,N,K,bias,res", [
    (300, 512, 384, True, True),        # ragged M, two N tiles
    (129, 96, 200, True, False),        # N below one tile, K not a multiple of 64
    (4096, 2560, 512, False, True),     # 320 tiles: several per CTA, both TMEM accumulators
    (1, 32, 8, False, False),
])
def test_linear_matches_fp64(M, N, K, bias, res):
    a, w = _rand((M, K), M + N), _rand((N, K), K, scale=K ** -0.5)
    b = _rand((N,), 7, 0.1) if bias else None
    r = _rand((M, N), 8) if res else None
    out = A.linear(a.to(DEV), w.to(DEV), None if b is None else b.to(DEV), None if r is None else r.to(DEV))
    torch.cuda.synchronize()
    exact = OB.linear(_f64(a), _f64(w), None if b is None else _f64(b)) + (0.0 if r is None else _f64(r))
    got = _f64(out)
    # One rounding to bf16 (at most one unit, 2^-7 |y|, counting the FP32 step),
    # plus the FP32 accumulation error, which scales with the sum of the
    # magnitudes of the terms rather than with their (possibly cancelling) sum.
    mag = np.abs(_f64(a)) @ np.abs(_f64(w)).T + (0.0 if r is None else np.abs(_f64(r)))
    bound = np.abs(exact) * 2.0 ** -7 + mag * 2.0 ** -20 + 1e-6
    assert np.all(np.abs(got - exact) <= bound), float(np.max(np.abs(got - exact) / bound))


# (6000, 512): more rows than the grid has warps (two blocks of eight warps
# per SM), so warps loop over several rows, with a ragged last pass. Rows of
# 1025-4096 values take the register-resident kernel (one block of eight warps
# per SM, the next row loaded ahead): (3000, 4096) gives each warp two or three
# rows; H = 1032 is 129 chunks of eight, one more than 32 lanes x 4.
@pytest.mark.parametrize("M,H", [(333, 256), (64, 1000), (257, 4096), (16, 8192), (6000, 512), (3000, 4096),
                                 (700, 1032)])
def test_layernorm_matches_fp64(M, H):
    x = _rand((M, H), H, 2.0)
    g = (_rand((H,), 1, 0.1).float() + 1.0).to(torch.bfloat16)
    b = _rand((H,), 2, 0.1)
    y = A.layernorm(x.to(DEV), g.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    exact = OB.layer_norm(_f64(x), _f64(g), _f64(b))
    got = _f64(y)
    ulp = np.abs(exact) * 2.0 ** -7 + 1e-5
    assert np.all(np.abs(got - exact) <= ulp), float(np.max(np.abs(got - exact) / ulp))


@pytest.mark.parametrize("B,S,Hq,Hkv,D,causal", [(2, 300, 4, 2, 128, True), (1, 200, 8, 8, 64, False),
                                                 (2, 32, 8, 2, 128, True)])    # S * 4 <= 256: heads packed
def test_packed_qkv_attention(B, S, Hq, Hkv, D, causal):
    qkv = _rand((B, S, (Hq + 2 * Hkv) * D), S + D)
    q = qkv[..., : Hq * D].reshape(B, S, Hq, D).contiguous()
    k = qkv[..., Hq * D: (Hq + Hkv) * D].reshape(B, S, Hkv, D).contiguous()
    v = qkv[..., (Hq + Hkv) * D:].reshape(B, S, Hkv, D).contiguous()
    o, lse = A.attention_qkvpacked(qkv.to(DEV), Hq, Hkv, D, causal=causal)
    o2, lse2 = A.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, lse2)
    check(o, lse, q, k, v, None, 1 if causal else 0, label="packed qkv")


def _block_case(cfg):
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = I.make_block_inputs(cfg)
    y = A.attention_block(*(t.to(DEV) for t in (x, gamma, beta, w_qkv, b_qkv, w_o, b_o)), Hq=cfg.Hq, Hkv=cfg.Hkv,
                          D=cfg.D, causal=cfg.causal)
    torch.cuda.synchronize()
    want = OB.block(*(_f64(t) for t in (x, gamma, beta, w_qkv, b_qkv, w_o, b_o)), Hq=cfg.Hq, Hkv=cfg.Hkv, D=cfg.D,
                    causal=cfg.causal, hold_in="bf16")
    got = _f64(y)
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    # y is rounded to bf16 (2^-9 |y|); the held intermediates may differ from the
    # oracle's by one bf16 unit where FP32 and FP64 straddle a rounding boundary.
    assert float(err.max()) <= 2e-2 and float(err.mean()) <= 2e-3, (float(err.max()), float(err.mean()))
    return err


@pytest.mark.parametrize("B,S,Hq,Hkv,D,causal", [
    (2, 200, 4, 4, 64, True),            # hidden 256
    (1, 300, 4, 2, 128, True),           # GQA, hidden 512, ragged tiles
    (2, 130, 8, 8, 64, False),           # non-causal
])
def test_block_matches_oracle(B, S, Hq, Hkv, D, causal):
    _block_case(I.BlockConfig("blk", B, S, Hq, Hkv, D, causal=causal, seed=B + S + D))


def test_llama2_7b_sized_block_one_sequence():
    _block_case(I.BlockConfig("l7b_block_1", 1, 2048, 32, 32, 128, seed=3))


def test_block_in_place():
    cfg = I.BlockConfig("inplace", 1, 128, 4, 4, 64, seed=11)
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = (t.to(DEV) for t in I.make_block_inputs(cfg))
    y = A.attention_block(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=4, Hkv=4, D=64)
    x2 = x.clone()
    A.attention_block(x2, gamma, beta, w_qkv, b_qkv, w_o, b_o, Hq=4, Hkv=4, D=64, out=x2)
    torch.cuda.synchronize()
    assert torch.equal(x2.view(torch.int16), y.view(torch.int16))
