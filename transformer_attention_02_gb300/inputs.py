"""Seeded synthetic inputs for the fused attention forward.

This module is the only code that both the CUDA path's tests/benchmark and the
FP64 oracle consume. It holds no attention arithmetic: it draws Q, K, V (and the
additive mask) on the CPU from a seeded ``torch.Generator`` and rounds them to
the 16-bit storage type once, so that both sides see the very same values.

Recipe (one generator per call, seeded with ``seed``):
  * Q, then K, then V, each drawn directly in (B, S, H, D) as float32 and
    rounded to bf16 (or fp16) with round-to-nearest-even.
  * value sets:
      normal      Q, K, V ~ N(0, 1)
      zero_q      Q = 0 (drawn, then zeroed), K, V ~ N(0, 1)
      saturated   Q, K = 30 * N(0, 1), V ~ N(0, 1)
      student_t2  Q, K, V ~ Student-t with 2 degrees of freedom, Z / sqrt(E)
                  with Z ~ N(0, 1) and E = -ln(U) ~ Exp(1), U ~ U[0, 1)
                  (U = 0 gives E = inf and t = 0), clipped to the largest
                  finite value of the storage type
  * the additive mask (a second generator seeded with seed + 1): FP32
    (B, Sq, Sk); per query row, floor(frac * Sk) keys picked by
    argsort(rand(Sk)) are -inf, all others 0.0. A row is never fully masked
    while frac < 1.

The stress value sets follow the advice in "ops-transformer：Transformer算子融合与
推理加速实战" §4.2 (all-zero input, large values driving softmax into
saturation, heavy-tailed values) rather than plain random numbers only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

VALUE_SETS = ("normal", "zero_q", "saturated", "student_t2")


@dataclass(frozen=True)
class AttnConfig:
    """One workload: shapes, mask kind and value set (all sizes runtime)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    additive_mask: bool = False
    values: str = "normal"
    mask_frac: float = 0.3
    seed: int = 0
    dtype: str = "bf16"

    @property
    def mask_kind(self) -> int:
        return (1 if self.causal else 0) + (2 if self.additive_mask else 0)

    @property
    def flops(self) -> float:
        """4*B*Hq*Sq*Sk*D, halved for a causal mask (square case)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "AttnConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return AttnConfig(**d)


def _cfg(name, B, Hq, Hkv, S, D, causal, **kw):
    return AttnConfig(name=name, B=B, Hq=Hq, Hkv=Hkv, Sq=S, Sk=S, D=D, causal=causal, **kw)


# The five workloads of the measured path (each a parity case; the second is
# the headline benchmark workload).
CONFIGS = {
    "tiny": _cfg("tiny", 1, 2, 2, 128, 64, True),
    "llama2_7b_prefill": _cfg("llama2_7b_prefill", 4, 32, 32, 2048, 128, True),
    "gqa_prefill": _cfg("gqa_prefill", 8, 32, 8, 4096, 128, True),
    "long_gqa_prefill": _cfg("long_gqa_prefill", 1, 64, 8, 16384, 128, True),
}
for _d in (64, 128):
    for _v in ("zero_q", "saturated", "student_t2"):
        _n = f"stress_d{_d}_{_v}"
        CONFIGS[_n] = _cfg(_n, 2, 16, 16, 2048, _d, False, additive_mask=True, values=_v)

# The three causal prefills at head dimension 64 (the pages' other supported
# size), for measurement.
for _n in ("llama2_7b_prefill", "gqa_prefill", "long_gqa_prefill"):
    CONFIGS[_n + "_d64"] = CONFIGS[_n].with_(name=_n + "_d64", D=64)

BENCH_CONFIG = "llama2_7b_prefill"

# Decode over a KV cache (one new query row per sequence; split-key path):
# Llama-3-8B-like GQA (32 query heads, 8 K/V heads of 128) and an MHA case.
DECODE_CONFIGS = {
    "gqa_decode": AttnConfig("gqa_decode", 16, 32, 8, 1, 8192, 128, causal=True),
    "gqa_decode_long": AttnConfig("gqa_decode_long", 4, 32, 8, 1, 32768, 128, causal=True),
    "mha_decode": AttnConfig("mha_decode", 16, 32, 32, 1, 4096, 128, causal=True),
}


def storage_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f16": torch.float16}[name]


def _draw(g: torch.Generator, shape, values: str, which: str, dt: torch.dtype) -> torch.Tensor:
    if values == "student_t2":
        z = torch.randn(shape, generator=g, dtype=torch.float32)
        u = torch.rand(shape, generator=g, dtype=torch.float32)
        e = -torch.log(u)
        x = z / torch.sqrt(e)
        big = torch.finfo(dt).max
        x = torch.nan_to_num(x, nan=0.0, posinf=big, neginf=-big).clamp_(-big, big)
    else:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if values == "saturated" and which in ("q", "k"):
            x = x * 30.0
        if values == "zero_q" and which == "q":
            x = torch.zeros_like(x)
    return x.to(dt)


def make_qkv(cfg: AttnConfig):
    """Q (B,Sq,Hq,D), K and V (B,Sk,Hkv,D) as CPU tensors of the storage type."""
    if cfg.values not in VALUE_SETS:
        raise ValueError(f"unknown value set {cfg.values!r}")
    dt = storage_dtype(cfg.dtype)
    g = torch.Generator(device="cpu")
    g.manual_seed(cfg.seed)
    q = _draw(g, (cfg.B, cfg.Sq, cfg.Hq, cfg.D), cfg.values, "q", dt)
    k = _draw(g, (cfg.B, cfg.Sk, cfg.Hkv, cfg.D), cfg.values, "k", dt)
    v = _draw(g, (cfg.B, cfg.Sk, cfg.Hkv, cfg.D), cfg.values, "v", dt)
    return q, k, v


def make_mask(cfg: AttnConfig) -> torch.Tensor:
    """FP32 (B, Sq, Sk) additive mask: floor(frac*Sk) random keys per row at -inf."""
    g = torch.Generator(device="cpu")
    g.manual_seed(cfg.seed + 1)
    n_masked = int(math.floor(cfg.mask_frac * cfg.Sk))
    if cfg.Sk > 0 and n_masked >= cfg.Sk:
        raise ValueError("mask_frac would mask whole rows")
    mask = torch.zeros((cfg.B, cfg.Sq, cfg.Sk), dtype=torch.float32)
    if n_masked == 0 or cfg.Sq == 0:
        return mask
    r = torch.rand((cfg.B, cfg.Sq, cfg.Sk), generator=g, dtype=torch.float32)
    idx = torch.argsort(r, dim=-1)[..., :n_masked]
    mask.scatter_(-1, idx, float("-inf"))
    return mask


def make_inputs(cfg: AttnConfig):
    """(q, k, v, mask_or_None) on the CPU for one workload."""
    q, k, v = make_qkv(cfg)
    mask = make_mask(cfg) if cfg.additive_mask else None
    return q, k, v, mask


def bits(t: torch.Tensor):
    """The raw 16-bit patterns of a bf16/fp16 CPU tensor, as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


# ------------------------------------------------------------ attention block

@dataclass(frozen=True)
class BlockConfig:
    """Sizes of one attention block: x (B, S, Hq*D) -> y (B, S, Hq*D)."""
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    causal: bool = True
    seed: int = 0

    @property
    def hidden(self) -> int:
        return self.Hq * self.D

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: the two projections (2 M N K each) plus the attention."""
        M, H, F = self.B * self.S, self.hidden, (self.Hq + 2 * self.Hkv) * self.D
        att = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return 2.0 * M * F * H + 2.0 * M * H * H + (att / 2 if self.causal else att)


BLOCK_CONFIGS = {
    "tiny_block": BlockConfig("tiny_block", 1, 128, 2, 2, 64),
    # one Llama-2-7B-sized layer's attention block on the prefill batch (hidden 4096, 32 heads of 128)
    "llama2_7b_block": BlockConfig("llama2_7b_block", 4, 2048, 32, 32, 128),
}


def make_block_inputs(cfg: BlockConfig):
    """x, ln_gamma, ln_beta, w_qkv, b_qkv, w_o, b_o as bf16 CPU tensors:
    x ~ N(0, 1); gamma ~ 1 + 0.1 N(0, 1); beta, the biases ~ 0.02 N(0, 1);
    weights ~ N(0, 1/hidden) (unit-variance projections)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(cfg.seed)
    H, F = cfg.hidden, (cfg.Hq + 2 * cfg.Hkv) * cfg.D

    def r(*shape, scale=1.0, shift=0.0):
        return (torch.randn(shape, generator=g) * scale + shift).to(torch.bfloat16)

    x = r(cfg.B, cfg.S, H)
    gamma = r(H, scale=0.1, shift=1.0)
    beta = r(H, scale=0.02)
    w_qkv = r(F, H, scale=H ** -0.5)
    b_qkv = r(F, scale=0.02)
    w_o = r(H, H, scale=H ** -0.5)
    b_o = r(H, scale=0.02)
    return x, gamma, beta, w_qkv, b_qkv, w_o, b_o
