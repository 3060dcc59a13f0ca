"""Seeded synthetic inputs for the INT8ConvRot linear layer.

This module holds random-number recipes and workload shapes only -- none of
the layer's arithmetic.  It is the one module that both the oracle-side tests
and the GPU-side tests/benchmark use to draw inputs.

Shapes and layer counts come from the page "INT8ConvRot GEMM vs fp16 on M1 Max
with Metal, MPSMatrix, and MLX", section "Testing the MPS weight-only INT8 path
in isolation", per-shape table (448 int8 weights in 6 (N, K) shapes, all timed
at M = 1024).  The quantized UNet checkpoint those shapes come from is not
available; these generators stand in for its weights and activations.

Recipe (stated once, used everywhere):
  X      fp16 [M, K]: standard normal draws (fp32), then ``n_out`` random
         K-columns multiplied by 50 (activation outliers, the reason for the
         rotation), then rounded to fp16.  n_out = round(0.01 K), except the
         tiny case, which uses 4.
  W      fp32 [N, K]: normal with standard deviation 1/sqrt(K).
  lora_down fp16 [R, K], lora_up fp16 [N, R]: normal with std 0.01.
Each array comes from its own numpy PCG64 stream keyed by (seed, stream id), so
changing one size never changes another array.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

OUTLIER_SCALE = 50.0

# (N, K, layer count) -- the six weight shapes of the quantized UNet.
SWEEP_SHAPES = (
    (2048, 2048, 168),
    (256, 2048, 84),
    (6144, 256, 84),
    (2048, 1024, 56),
    (8192, 2048, 28),
    (2048, 8192, 28),
)
SWEEP_M = 1024


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def n_outliers(K: int) -> int:
    return int(round(0.01 * K))


def make_x(M: int, K: int, seed: int, n_out: int | None = None) -> np.ndarray:
    """fp16 activations [M, K] with ``n_out`` outlier columns scaled by 50."""
    rng = _rng(seed, 0)
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = n_outliers(K) if n_out is None else n_out
    if n_out:
        cols = rng.permutation(K)[:n_out]
        x[:, cols] *= OUTLIER_SCALE
    return x.astype(np.float16)


def make_w(N: int, K: int, seed: int) -> np.ndarray:
    """fp32 weights [N, K] with std 1/sqrt(K)."""
    rng = _rng(seed, 1)
    return (rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K)))


def make_lora(N: int, K: int, R: int, seed: int):
    """fp16 lora_down [R, K] and lora_up [N, R], std 0.01."""
    rng = _rng(seed, 2)
    down = (rng.standard_normal((R, K), dtype=np.float32) * np.float32(0.01)).astype(np.float16)
    up = (rng.standard_normal((N, R), dtype=np.float32) * np.float32(0.01)).astype(np.float16)
    return down, up


def make_int8(shape, seed: int, stream: int = 3, low: int = -128, high: int = 127) -> np.ndarray:
    """Uniform int8 values in [low, high] (for exact-product tests)."""
    return _rng(seed, stream).integers(low, high + 1, size=shape, dtype=np.int64).astype(np.int8)


@dataclass(frozen=True)
class Config:
    name: str
    M: int
    N: int
    K: int
    seed: int
    n_out: int | None = None
    R: int = 0
    lora_scale: float = 0.0
    notes: str = ""


# The five workloads.  The tiny case (M=64, K=256, N=256, 4 outlier columns,
# seed 0) is small enough for the oracle in a fraction of a second.
TINY = Config("tiny", 64, 256, 256, seed=0, n_out=4,
              notes="one Hadamard group; 4 outlier columns x50")
ATTN = Config("attn", 1024, 2048, 2048, seed=1,
              notes="attention-projection sized; 1% outlier columns x50")
LORA = Config("lora", 4096, 2048, 8192, seed=4, R=32, lora_scale=0.8,
              notes="unmerged LoRA rank 32, scale 0.8, on the unrotated X")
M_SWEEP_MS = (1, 16, 128, 4096, 16384)
M_SWEEP_SHAPES = ((8192, 2048), (2048, 8192))


def sweep_configs(seed: int = 2):
    """The six M=1024 layer shapes with their layer counts."""
    out = []
    for i, (N, K, count) in enumerate(SWEEP_SHAPES):
        out.append((Config(f"sweep_{N}x{K}", SWEEP_M, N, K, seed=seed * 1000 + i), count))
    return out


def m_sweep_configs(seed: int = 3):
    out = []
    for j, (N, K) in enumerate(M_SWEEP_SHAPES):
        for i, M in enumerate(M_SWEEP_MS):
            out.append(Config(f"msweep_M{M}_{N}x{K}", M, N, K, seed=seed * 1000 + 10 * j + i))
    return out


def sweep_total_ops(M: int = SWEEP_M) -> float:
    """2*M*N*K summed over the 448 layers (integer multiply-adds count 2)."""
    return float(sum(2 * M * N * K * c for N, K, c in SWEEP_SHAPES))


def make_inputs(cfg: Config):
    """X, W (and lora_down, lora_up when R > 0) for a config."""
    X = make_x(cfg.M, cfg.K, cfg.seed, cfg.n_out)
    W = make_w(cfg.N, cfg.K, cfg.seed)
    if cfg.R:
        down, up = make_lora(cfg.N, cfg.K, cfg.R, cfg.seed)
    else:
        down = up = None
    return X, W, down, up
