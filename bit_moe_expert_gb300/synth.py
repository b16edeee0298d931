"""Seeded synthetic inputs for the 4-bit groupwise-affine MoE layer.

This module only *draws* inputs: it holds none of the layer's arithmetic
(no dequantisation, no routing, no matmul).  Both the CUDA path and the CPU
oracle consume exactly the bytes produced here.

Format (the checkpoint format described on "Perplexity's Lily Beats MLX-LM on
MacBook M5", section "Prefill: keep routing on the GPU, dequantize in flight",
and on "Perplexity builds a custom engine for Qwen on M5 Macs"): every group of
64 consecutive weights along K shares one bf16 scale and one bf16 bias, and a
weight is w = q * scale + bias with q an unsigned 4-bit code.

Layout used throughout (row-major, all integers little-endian):
  q      uint32 [E][N][K/8]   8 codes per word, code for k at bits 4*(k%8),
                              i.e. the low nibble holds the lowest k
  scale  uint16 [E][N][K/64]  bf16 bit patterns
  bias   uint16 [E][N][K/64]  bf16 bit patterns
gate and up are [E][I][d] (N=I, K=d); down is [E][d][I] (N=d, K=I).
Low-bit variants keep the layout with b = 3 or 2 bits per code: q is
[E][N][K*b/32], each row one bit stream with code k at bits b*k .. b*k+b-1
(a 3-bit code may straddle two words); codes uniform on 0..2^b-1, scale ~
U(0.004, 0.04) (b = 3) or U(0.008, 0.08) (b = 2), bias = -2^(b-1) * scale.

Value distributions (synthetic stand-ins for the pages' workloads):
  X ~ N(0,1) rounded to bf16 (round to nearest even); router logits ~ N(0,1)
  fp32; codes uniform on 0..15; scale ~ U(0.002, 0.02) rounded to bf16;
  bias = -8 * scale (exact in bf16, the factor is a power of two).
The skewed long-prefill workload adds 2*ln(1/rank_e) to expert e's logit,
rank being a seeded permutation of 1..E (Zipf-like expert popularity).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

GROUP = 64          # weights per (scale, bias) group along K


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int              # tokens per call
    d: int              # model dimension
    E: int              # routed experts
    k: int              # experts per token
    I: int              # routed expert intermediate size
    I_shared: int       # shared expert intermediate size (0 = no shared expert)
    layers: int         # distinct weight sets
    seed: int
    chunk: int = 0      # tokens per call when the prompt is processed in chunks (0 = T)
    zipf: bool = False  # skewed router logits
    bits: int = 4       # bits per expert weight code (4, 3 or 2)

    @property
    def tokens_per_call(self) -> int:
        return self.chunk if self.chunk else self.T


# The synthetic workloads: the five of the 4-bit layer, then low-bit variants.
CONFIGS = {
    "tiny": LayerConfig("tiny", T=16, d=256, E=16, k=2, I=128, I_shared=128, layers=1, seed=0),
    "decode": LayerConfig("decode", T=1, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=1),
    "prefill512": LayerConfig("prefill512", T=512, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=2),
    "prefill4096": LayerConfig("prefill4096", T=4096, d=2048, E=256, k=8, I=512, I_shared=512, layers=40,
                               seed=3, chunk=1024, zipf=True),
    "canvas": LayerConfig("canvas", T=256, d=2816, E=128, k=8, I=704, I_shared=0, layers=30, seed=4),
    # the decode layer with 3- and 2-bit expert codes (the low-bit experts of the "next" steps)
    "decode3b": LayerConfig("decode3b", T=1, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=7, bits=3),
    "decode2b": LayerConfig("decode2b", T=1, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=6, bits=2),
    # the 512-token prefill layer (every expert active, the tensor-core path bound by the weight stream)
    # with 3- and 2-bit expert codes
    "prefill512b3": LayerConfig("prefill512b3", T=512, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=8,
                                bits=3),
    "prefill512b2": LayerConfig("prefill512b2", T=512, d=2048, E=256, k=8, I=512, I_shared=512, layers=40, seed=9,
                                bits=2),
}


def expert_bytes(N: int, K: int, bits: int = 4) -> int:
    """Bytes of one packed matrix: K*bits/8 per row of codes plus 2+2 bytes per group."""
    return N * (K * bits // 8) + 2 * 2 * N * (K // GROUP)


def ffn_bytes(d: int, I: int, bits: int = 4) -> int:
    """Bytes of one expert (gate, up, down)."""
    return 2 * expert_bytes(I, d, bits) + expert_bytes(d, I, bits)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, layer: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, tag])))


# Scale range and bias factor per code width: bias = -half the code range
# times the scale (exact in bf16), so the weights are (q - 2^(bits-1)) * scale
# and the 2-bit weights span about the same range as the 4-bit ones.
SCALE_RANGE = {4: (0.002, 0.02), 3: (0.004, 0.04), 2: (0.008, 0.08)}


def draw_qmat(rng: np.random.Generator, E: int, N: int, K: int, bits: int = 4):
    """One stacked packed matrix: (q [E][N][K*bits/32] u32, scale, bias [E][N][K/64] u16)."""
    assert K % GROUP == 0 and bits in SCALE_RANGE
    q = rng.integers(0, 2**32, size=(E, N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
    s = f32_to_bf16_bits(rng.uniform(*SCALE_RANGE[bits], size=(E, N, K // GROUP)).astype(np.float32))
    b = f32_to_bf16_bits(bf16_bits_to_f32(s) * np.float32(-(1 << (bits - 1))))
    return q, s, b


@dataclasses.dataclass
class Layer:
    """Host copy of one synthetic layer's inputs and weights."""
    X: np.ndarray          # uint16 [T][d] bf16 bits
    logits: np.ndarray     # float32 [T][E]
    routed: dict           # {"gate": (q,s,b), "up": ..., "down": ...}
    shared: Optional[dict]  # same with E=1, or None


def draw_logits(cfg: LayerConfig, T: int, layer: int) -> np.ndarray:
    rng = _rng(cfg.seed, layer, 1)
    z = rng.standard_normal(size=(T, cfg.E))
    if cfg.zipf:
        rank = _rng(cfg.seed, 0, 99).permutation(cfg.E) + 1     # same ranks for every layer
        z = z + 2.0 * np.log(1.0 / rank)[None, :]
    return z.astype(np.float32)


def draw_x(cfg: LayerConfig, T: int, layer: int) -> np.ndarray:
    rng = _rng(cfg.seed, layer, 2)
    return f32_to_bf16_bits(rng.standard_normal(size=(T, cfg.d)).astype(np.float32))


def draw_router(cfg: LayerConfig, layer: int) -> np.ndarray:
    """Router weights Wr [E][d] as bf16 bit patterns, N(0, 1/d): with X ~ N(0, 1) the logits are about N(0, 1),
    the scale of the logits drawn directly for the other workloads."""
    rng = _rng(cfg.seed, layer, 3)
    return f32_to_bf16_bits((rng.standard_normal(size=(cfg.E, cfg.d)) / np.sqrt(cfg.d)).astype(np.float32))


def draw_experts(cfg: LayerConfig, layer: int, E: Optional[int] = None, I: Optional[int] = None,
                 tag: int = 10) -> dict:
    E = cfg.E if E is None else E
    I = cfg.I if I is None else I
    return {
        "gate": draw_qmat(_rng(cfg.seed, layer, tag + 0), E, I, cfg.d, cfg.bits),
        "up": draw_qmat(_rng(cfg.seed, layer, tag + 1), E, I, cfg.d, cfg.bits),
        "down": draw_qmat(_rng(cfg.seed, layer, tag + 2), E, cfg.d, I, cfg.bits),
    }


def draw_layer(cfg: LayerConfig, layer: int = 0, T: Optional[int] = None) -> Layer:
    """All inputs of one layer on the host (use for sizes that fit comfortably in RAM)."""
    T = cfg.T if T is None else T
    shared = draw_experts(cfg, layer, E=1, I=cfg.I_shared, tag=20) if cfg.I_shared else None
    return Layer(X=draw_x(cfg, T, layer), logits=draw_logits(cfg, T, layer),
                 routed=draw_experts(cfg, layer), shared=shared)


def small_config(**kw) -> LayerConfig:
    """An ad-hoc configuration for tests (defaults: the tiny workload)."""
    base = dataclasses.asdict(CONFIGS["tiny"])
    base.update(kw)
    base.setdefault("name", "custom")
    return LayerConfig(**base)


# ---------------------------------------------------------------------------
# Device-side drawing for the large workloads (torch's seeded generator).
# Same distributions as above; the bytes differ from the host generator, so a
# parity check copies the device bytes it needs back to the host.
# ---------------------------------------------------------------------------

def draw_qmat_torch(gen, E: int, N: int, K: int, device, bits: int = 4):
    import torch
    q = torch.randint(-2**31, 2**31, (E, N, K * bits // 32), generator=gen, device=device,
                      dtype=torch.int64).to(torch.int32)
    s = torch.empty((E, N, K // GROUP), device=device, dtype=torch.float32).uniform_(*SCALE_RANGE[bits],
                                                                                      generator=gen)
    s = s.to(torch.bfloat16)
    b = (s.float() * -float(1 << (bits - 1))).to(torch.bfloat16)
    return q, s.view(torch.int16), b.view(torch.int16)


def draw_experts_torch(cfg: LayerConfig, layer: int, device, E: Optional[int] = None,
                       I: Optional[int] = None, tag: int = 10) -> dict:
    import torch
    E = cfg.E if E is None else E
    I = cfg.I if I is None else I
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1_000_003 + layer * 1009 + tag)
    return {
        "gate": draw_qmat_torch(gen, E, I, cfg.d, device, cfg.bits),
        "up": draw_qmat_torch(gen, E, I, cfg.d, device, cfg.bits),
        "down": draw_qmat_torch(gen, E, cfg.d, I, device, cfg.bits),
    }


def config_summary(cfg: LayerConfig) -> dict:
    per_expert = ffn_bytes(cfg.d, cfg.I, cfg.bits)
    return {
        "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "I": cfg.I, "I_shared": cfg.I_shared,
        "layers": cfg.layers, "chunk": cfg.chunk, "zipf": cfg.zipf,
        "bytes_per_expert": per_expert,
        "bytes_per_layer_all_experts": cfg.E * per_expert + (ffn_bytes(cfg.d, cfg.I_shared, cfg.bits)
                                                              if cfg.I_shared else 0),
        "flops_per_token_per_expert": 6 * cfg.d * cfg.I,
        "log2_E": math.log2(cfg.E),
    }
