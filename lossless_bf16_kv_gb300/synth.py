"""Seeded synthetic inputs for the SplitZip codec.

This module holds only random-number recipes (no part of the codec's
arithmetic).  It serves both the CUDA path and the CPU oracle's tests: a tensor
is drawn once (on the GPU, or on the CPU where no GPU is present) and the same
bytes go to both sides.

The recipes stand in for the real key/value activations the pages measure on
(Qwen3-32B on WikiText-2, "SplitZip: Ultra-Fast Lossless KV Compression for
Disaggregated LLM Serving", section Reproducing Paper Artifact Scripts), which
are not available here; no item of that dataset is reproduced.

All draws are fp32 from a ``torch.Generator`` seeded once per tensor, then cast
to BF16 or FP8 E5M2 with PyTorch's round-to-nearest-even conversion.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable

import torch

KV_HEADS = 8
HEAD_DIM = 128
OUTLIER_P = 0.001
OUTLIER_SCALE = 100.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) drawn in fp32, cast to BF16."""
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def _kv_layer_fp32(g: torch.Generator, tokens: int, device) -> torch.Tensor:
    """One layer's [2, tokens, 8, 128] fp32 key/value values.

    Per-(head, channel) scale s = exp(N(0,1)) (log-normal, mu=0, sigma=1), drawn
    first and shared by K and V; values N(0,1) * s; 0.1% of entries (Bernoulli
    mask) multiplied by 100 as outliers.
    """
    scale = torch.exp(torch.randn((KV_HEADS, HEAD_DIM), generator=g, dtype=torch.float32,
                                  device=device))
    v = torch.randn((2, tokens, KV_HEADS, HEAD_DIM), generator=g, dtype=torch.float32,
                    device=device)
    v.mul_(scale)
    mask = torch.rand((2, tokens, KV_HEADS, HEAD_DIM), generator=g, dtype=torch.float32,
                      device=device) < OUTLIER_P
    return torch.where(mask, v * OUTLIER_SCALE, v)


def kv_cache(layers: int, tokens: int, seed: int, device="cpu", dtype=torch.bfloat16,
             squeeze_single: bool = False) -> torch.Tensor:
    """KV cache [layers, 2, tokens, 8, 128], generated layer by layer with fresh
    per-layer scales from one generator.  ``dtype`` is torch.bfloat16 or
    torch.float8_e5m2 (cast directly from fp32, not through BF16)."""
    g = _gen(seed, device)
    out = torch.empty((layers, 2, tokens, KV_HEADS, HEAD_DIM), dtype=dtype, device=device)
    for layer in range(layers):
        out[layer].copy_(_kv_layer_fp32(g, tokens, device).to(dtype))
    if squeeze_single and layers == 1:
        return out[0]
    return out


def student_t_scaled_bf16(shape, seed: int, df: float = 1.5, u_lo: float = -20.0,
                          u_hi: float = 20.0, device="cpu") -> torch.Tensor:
    """t(df) * 2**U with U ~ Uniform[u_lo, u_hi] (continuous), cast to BF16.

    t = Z / sqrt(V / df) with Z ~ N(0,1) and V ~ chi-square(df) = 2 * Gamma(df/2).
    """
    g = _gen(seed, device)
    z = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    alpha = torch.full(shape, df / 2.0, dtype=torch.float32, device=device)
    v = 2.0 * torch._standard_gamma(alpha, generator=g)
    del alpha
    t = z / torch.sqrt(v / df)
    del z, v
    u = torch.rand(shape, generator=g, dtype=torch.float32, device=device) * (u_hi - u_lo) + u_lo
    t.mul_(torch.exp2(u))
    return t.to(torch.bfloat16)


@dataclass(frozen=True)
class Workload:
    """One seeded workload: the tensor to encode, the tensor to calibrate on,
    the chunk size and the element format ('bf16' or 'e5m2')."""
    name: str
    fmt: str
    shape: tuple
    chunk: int
    make: Callable[[object], torch.Tensor]
    make_calib: Callable[[object], torch.Tensor]
    description: str

    @property
    def numel(self) -> int:
        return math.prod(self.shape)

    @property
    def nbytes(self) -> int:
        return self.numel * (2 if self.fmt == "bf16" else 1)


def _n01_calib(device):
    return normal_bf16((1024, 4096), seed=1, device=device)


WORKLOADS = {
    "n01_1024x4096": Workload(
        "n01_1024x4096", "bf16", (1024, 4096), 1024,
        lambda d: normal_bf16((1024, 4096), seed=0, device=d), _n01_calib,
        "BF16 [1024, 4096] N(0,1) seed 0; codebook from N(0,1) seed 1 of the same shape"),
    "kv_layer_32k": Workload(
        "kv_layer_32k", "bf16", (2, 32768, 8, 128), 1024,
        lambda d: kv_cache(1, 32768, seed=0, device=d, squeeze_single=True),
        lambda d: kv_cache(1, 32768, seed=1, device=d, squeeze_single=True),
        "single-layer KV BF16 [2, 32768, 8, 128], log-normal channel scales, 0.1% x100 "
        "outliers; codebook from seed 1"),
    "kv_prefill_64L_16k": Workload(
        "kv_prefill_64L_16k", "bf16", (64, 2, 16384, 8, 128), 1024,
        lambda d: kv_cache(64, 16384, seed=0, device=d),
        lambda d: kv_cache(64, 1024, seed=1, device=d),
        "64-layer prefill KV BF16 [64, 2, 16384, 8, 128] (2^31 elements, 4.29 GB); "
        "codebook from a [64, 2, 1024, 8, 128] seed-1 sample"),
    "kv_prefill_4L_16k": Workload(
        "kv_prefill_4L_16k", "bf16", (4, 2, 16384, 8, 128), 1024,
        lambda d: kv_cache(4, 16384, seed=0, device=d),
        lambda d: kv_cache(4, 1024, seed=1, device=d),
        "4-layer prefill KV BF16 [4, 2, 16384, 8, 128] (2^27 elements, 268 MB > L2): the "
        "profiling-size cut of the 64-layer workload"),
    "kv_prefill_4L_16k_e5m2": Workload(
        "kv_prefill_4L_16k_e5m2", "e5m2", (4, 2, 16384, 8, 128), 1024,
        lambda d: kv_cache(4, 16384, seed=0, device=d, dtype=torch.float8_e5m2),
        lambda d: kv_cache(4, 1024, seed=1, device=d, dtype=torch.float8_e5m2),
        "4-layer prefill KV E5M2 (2^27 elements, 134 MB > L2): profiling-size cut"),
    "escape_stress_t15": Workload(
        "escape_stress_t15", "bf16", (8192, 8192), 1024,
        lambda d: student_t_scaled_bf16((8192, 8192), seed=0, device=d), _n01_calib,
        "BF16 [8192, 8192] t(1.5) * 2^U, U ~ U[-20, 20]; N(0,1) codebook"),
    "escape_stress_t15_u4": Workload(
        "escape_stress_t15_u4", "bf16", (8192, 8192), 1024,
        lambda d: student_t_scaled_bf16((8192, 8192), seed=0, u_lo=-4.0, u_hi=4.0, device=d),
        _n01_calib,
        "BF16 [8192, 8192] t(1.5) * 2^U, U ~ U[-4, 4]; N(0,1) codebook"),
    "kv_prefill_64L_16k_e5m2": Workload(
        "kv_prefill_64L_16k_e5m2", "e5m2", (64, 2, 16384, 8, 128), 1024,
        lambda d: kv_cache(64, 16384, seed=0, device=d, dtype=torch.float8_e5m2),
        lambda d: kv_cache(64, 1024, seed=1, device=d, dtype=torch.float8_e5m2),
        "FP8 E5M2 KV [64, 2, 16384, 8, 128] (2^31 elements, 2.15 GB) from the prefill "
        "generator; codebook from a seed-1 sample"),
}


def raw_bits(t: torch.Tensor) -> torch.Tensor:
    """Bit-pattern view: int16 for BF16, uint8 for E5M2 (same storage)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float8_e5m2:
        return t.view(torch.uint8)
    raise TypeError(f"unsupported dtype {t.dtype}")


def all_bf16_patterns() -> torch.Tensor:
    """Every one of the 65536 BF16 bit patterns, in order."""
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)


def all_e5m2_patterns() -> torch.Tensor:
    """Every one of the 256 E5M2 bit patterns, in order."""
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2)
