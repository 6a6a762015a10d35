"""Seeded synthetic inputs for the grouped expert MLP (shared by tests, bench and smoke).

This module only draws random numbers and rounds them to bfloat16; it holds none of the
layer's arithmetic (no routing, no GEMM, no activation, no quantisation), so that the CUDA
path and the fp64 oracle can be fed identical inputs without sharing any method code.

Recipe (one independent PCG64 stream per tensor, and per expert for the weights, so that
a subset of experts can be regenerated alone for sampled checks):

  logits  ~ N(0,1) fp32 [T, E]                       stream (seed, 0)
            (+ -s*ln(rank_e) for a Zipf(s) popularity, rank = permutation(E)+1,
             stream (seed, 5))
  x       ~ N(0,1) -> bf16 [T, H]                    stream (seed, 1)
  W1_e    ~ 0.02*N(0,1) -> bf16 [H, N1] logical      stream (seed, 2, e)
            N1 = 2F for gated activations, columns [0,F) gate, [F,2F) linear
            N1 = F for the non-gated squared ReLU
  W2_e    ~ 0.02*N(0,1) -> bf16 [F, H] logical       stream (seed, 3, e)
  dy      ~ N(0,1) -> bf16 [T, H]                    stream (seed, 4)
  rht signs (NVFP4) 16 fair bits -> uint16 mask        stream (seed, 8)

The workload shapes follow the Mixtral-8x7B, DeepSeek-V3 and GPT-OSS expert layers named on
the NVIDIA blog "Boosting MoE Training Throughput with Advanced Fusion Kernels" (section on
pretraining speedups) and the Transformer Engine MoE article (Mixtral results, Figure 5).
"""
from __future__ import annotations

import dataclasses
import numpy as np

GATED = ("swiglu", "clamped_swiglu", "geglu")


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    E: int
    k: int
    H: int
    F: int
    precision: str = "bf16"          # "bf16" | "mxfp8" | "nvfp4"
    activation: str = "swiglu"       # swiglu | clamped_swiglu | geglu | srelu
    seed: int = 0
    zipf_s: float = 0.0              # 0 = no popularity bias
    beta: float = 1.0
    gate_max: float = float("inf")
    lin_lo: float = float("-inf")
    lin_hi: float = float("inf")
    lin_offset: float = 0.0
    align: int = 32
    ilv: int = 64

    @property
    def gated(self) -> bool:
        return self.activation in GATED

    @property
    def N1(self) -> int:
        return 2 * self.F if self.gated else self.F

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def R_cap(self) -> int:
        return self.T * self.k + self.E * (self.align - 1)

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)

    def flops_fwd_bwd(self) -> float:
        # GEMM flops only: fwd 2*R*H*N1 + 2*R*F*H, bwd twice that.
        fwd = 2.0 * self.R * self.H * self.N1 + 2.0 * self.R * self.F * self.H
        return 3.0 * fwd


_CLAMP = dict(activation="clamped_swiglu", beta=1.702, gate_max=7.0, lin_lo=-7.0,
              lin_hi=7.0, lin_offset=1.0)

CONFIGS = {
    "tiny": LayerConfig("tiny", T=512, E=4, k=2, H=128, F=256, seed=0),
    "mixtral_bf16": LayerConfig("mixtral_bf16", T=8192, E=8, k=2, H=4096, F=14336, seed=1),
    "mixtral_mxfp8": LayerConfig("mixtral_mxfp8", T=16384, E=8, k=2, H=4096, F=14336,
                                 precision="mxfp8", seed=2, align=128),
    "dsv3_mxfp8": LayerConfig("dsv3_mxfp8", T=4096, E=256, k=8, H=7168, F=2048,
                              precision="mxfp8", seed=3, zipf_s=1.1, align=128),
    "gptoss_bf16": LayerConfig("gptoss_bf16", T=16384, E=128, k=4, H=2880, F=2880, seed=4,
                               **_CLAMP),
    "gptoss_mxfp8": LayerConfig("gptoss_mxfp8", T=16384, E=128, k=4, H=2880, F=2880, seed=4,
                                precision="mxfp8", align=128, **_CLAMP),
    # the GPT-OSS-shaped layer with the other activations of the sweep
    "gptoss_geglu_bf16": LayerConfig("gptoss_geglu_bf16", T=16384, E=128, k=4, H=2880, F=2880,
                                     seed=4, activation="geglu"),
    "gptoss_srelu_bf16": LayerConfig("gptoss_srelu_bf16", T=16384, E=128, k=4, H=2880, F=2880,
                                     seed=4, activation="srelu"),
    "gptoss_geglu_mxfp8": LayerConfig("gptoss_geglu_mxfp8", T=16384, E=128, k=4, H=2880,
                                      F=2880, seed=4, activation="geglu", precision="mxfp8",
                                      align=128),
    "gptoss_srelu_mxfp8": LayerConfig("gptoss_srelu_mxfp8", T=16384, E=128, k=4, H=2880,
                                      F=2880, seed=4, activation="srelu", precision="mxfp8",
                                      align=128),
    "mixtral_nvfp4": LayerConfig("mixtral_nvfp4", T=16384, E=8, k=2, H=4096, F=14336,
                                 precision="nvfp4", seed=5, align=128),
    "gptoss_nvfp4": LayerConfig("gptoss_nvfp4", T=16384, E=128, k=4, H=2880, F=2880, seed=4,
                                precision="nvfp4", align=128, **_CLAMP),
}


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng(list(key))


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def gen_logits(cfg: LayerConfig) -> np.ndarray:
    lg = _rng(cfg.seed, 0).standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if cfg.zipf_s:
        rank = _rng(cfg.seed, 5).permutation(cfg.E) + 1
        bias = (-cfg.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)
        lg = (lg + bias[None, :]).astype(np.float32)
    return lg


def gen_x(cfg: LayerConfig) -> np.ndarray:
    return round_to_bf16_bits(_rng(cfg.seed, 1).standard_normal((cfg.T, cfg.H), dtype=np.float32))


def gen_dy(cfg: LayerConfig) -> np.ndarray:
    return round_to_bf16_bits(_rng(cfg.seed, 4).standard_normal((cfg.T, cfg.H), dtype=np.float32))


def gen_w1_expert(cfg: LayerConfig, e: int) -> np.ndarray:
    """Logical W1 of expert e, [H, N1] bf16 bits; gated: columns [gate | linear]."""
    w = _rng(cfg.seed, 2, e).standard_normal((cfg.H, cfg.N1), dtype=np.float32)
    w *= np.float32(0.02)
    return round_to_bf16_bits(w)


def gen_w2_expert(cfg: LayerConfig, e: int) -> np.ndarray:
    """Logical W2 of expert e, [F, H] bf16 bits."""
    w = _rng(cfg.seed, 3, e).standard_normal((cfg.F, cfg.H), dtype=np.float32)
    w *= np.float32(0.02)
    return round_to_bf16_bits(w)


def gen_w1(cfg: LayerConfig) -> np.ndarray:
    return np.stack([gen_w1_expert(cfg, e) for e in range(cfg.E)])


def gen_w2(cfg: LayerConfig) -> np.ndarray:
    return np.stack([gen_w2_expert(cfg, e) for e in range(cfg.E)])


def gen_fc1_bias(cfg: LayerConfig) -> np.ndarray:
    """Optional FC1 bias, fp32 [E, N1] in the logical [gate | linear] order: 0.1 N(0,1)."""
    return (0.1 * _rng(cfg.seed, 6).standard_normal((cfg.E, cfg.N1))).astype(np.float32)


def gen_feat_scale(cfg: LayerConfig) -> np.ndarray:
    """Optional per-feature scale of the activation, fp32 [E, F]: 1 + 0.25 N(0,1)."""
    return (1.0 + 0.25 * _rng(cfg.seed, 7).standard_normal((cfg.E, cfg.F))).astype(np.float32)


def gen_rht_mask(cfg: LayerConfig) -> int:
    """The 16 random signs of the NVFP4 weight-gradient rotation, as a mask (bit j set: -1)."""
    return int(np.dot(_rng(cfg.seed, 8).integers(0, 2, 16), 1 << np.arange(16)))


def gen_bf16_matrix(seed: int, M: int, N: int, scale: float = 1.0, outlier_rows: int = 0):
    """A standalone bf16 matrix for quantiser tests: N(0,1)*scale, with a few rows carrying
    large-magnitude outliers and exact zeros so every scale-exponent path is exercised."""
    r = _rng(seed, 7)
    a = r.standard_normal((M, N), dtype=np.float32) * np.float32(scale)
    if outlier_rows:
        rows = r.choice(M, size=min(outlier_rows, M), replace=False)
        a[rows] *= np.float32(2.0) ** r.integers(-40, 40, size=(len(rows), 1)).astype(np.float32)
        a[rows[: max(1, len(rows) // 4)], : min(N, 64)] = 0.0
    return round_to_bf16_bits(a)
