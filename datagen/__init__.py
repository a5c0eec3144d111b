"""Seeded synthetic inputs for the FP8 up-projection workloads.

This module only draws random numbers and rounds them to bf16 storage; it holds
none of the FP8 method's arithmetic (no amax, no scale, no FP8 cast, no GEMM).
Both the CPU oracle's tests and the GPU tests/bench take their inputs from here.

Every tensor is returned as ``np.uint16`` bf16 bit patterns (row-major).
Seeds follow ``numpy.random.default_rng(1000 * config + tensor_index)``; the tiny
forward workload uses seed 0 for x and seed 1 for W.

Workloads (shapes and distributions):

* tiny forward: x [256 x 128] ~ N(0,1), W [128 x 512] ~ N(0, 0.02)
* GPT-2-small up-projection forward: x [8192 x 768] ~ N(0,1) with 0.1 % of the
  entries multiplied by 100, W [768 x 3072] ~ N(0, 0.02)
* backward: M=16384, K=1024, N=4096; dy log-normal magnitudes
  (median 1e-4, sigma of the natural log = 2, random sign), x ~ N(0,1),
  W ~ N(0, 0.02)
* fine-grained forward: x [16384 x 4096] = z * std_c with std_c = 10**U(-1,1)
  per column, W [4096 x 14336] ~ N(0, 0.02)
* delayed-scaling loop: 12 layers, W_l [1536 x 6144] ~ N(0, 0.02), x [32768 x 1536],
  dy [32768 x 6144] drawn once and shared, per-step weight perturbation N(0, 1e-3)
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "f32_from_bf16_bits", "normal_bf16", "outlier_normal_bf16",
    "lognormal_grad_bf16", "channel_scaled_bf16", "perturbation_f32", "WORKLOADS", "workload_inputs",
]


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits.

    Only used to store synthetic inputs in bf16; NaN inputs are not produced here.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return bf16_bits_from_f32(z)


def outlier_normal_bf16(seed: int, shape, frac: float = 1e-3, factor: float = 100.0) -> np.ndarray:
    """N(0,1) in bf16, then round(frac * numel) positions drawn without replacement are
    multiplied by ``factor`` in float32 and re-rounded to bf16."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    x = bf16_bits_from_f32(z)
    n = int(np.prod(shape))
    k = int(round(frac * n))
    if k:
        pos = rng.choice(n, size=k, replace=False)
        flat = x.reshape(-1)
        flat[pos] = bf16_bits_from_f32(f32_from_bf16_bits(flat[pos]) * np.float32(factor))
    return x


def lognormal_grad_bf16(seed: int, shape, median: float = 1e-4, sigma_log: float = 2.0) -> np.ndarray:
    """sign * median * exp(sigma_log * z), z ~ N(0,1), sign = +-1 with equal odds."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    sign = rng.integers(0, 2, size=shape, dtype=np.int8)
    mag = (np.float32(median) * np.exp(np.float32(sigma_log) * z)).astype(np.float32)
    mag[sign == 1] *= np.float32(-1.0)
    return bf16_bits_from_f32(mag)


def channel_scaled_bf16(seed: int, shape) -> np.ndarray:
    """x[:, c] = z * std_c with std_c = 10**U(-1, 1) drawn once per column."""
    rng = np.random.default_rng(seed)
    rows, cols = shape
    std = (10.0 ** rng.uniform(-1.0, 1.0, size=cols)).astype(np.float32)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    z *= std[None, :]
    return bf16_bits_from_f32(z)


def perturbation_f32(seed: int, shape, std: float = 1e-3) -> np.ndarray:
    """The simulated optimizer step's additive noise, N(0, std), float32."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    z *= np.float32(std)
    return z


# Workload table: name -> shapes.  ``scale`` divides the token count for reduced runs.
WORKLOADS = {
    "tiny_fwd": dict(cfg=1, M=256, K=128, N=512),
    "gpt2s_upproj_fwd": dict(cfg=2, M=8192, K=768, N=3072),
    "upproj_bwd": dict(cfg=3, M=16384, K=1024, N=4096),
    "finegrained_fwd": dict(cfg=4, M=16384, K=4096, N=14336),
    "delayed_loop": dict(cfg=5, M=32768, K=1536, N=6144, layers=12, steps=50, hist_len=16),
}


def workload_inputs(name: str, M: int | None = None, K: int | None = None, N: int | None = None) -> dict:
    """Inputs of a named workload, optionally at other sizes (same distributions and seeds)."""
    w = dict(WORKLOADS[name])
    M = w["M"] if M is None else M
    K = w["K"] if K is None else K
    N = w["N"] if N is None else N
    cfg = w["cfg"]
    base = 1000 * cfg
    if name == "tiny_fwd":
        return dict(x=normal_bf16(0, (M, K)), w=normal_bf16(1, (K, N), 0.02), M=M, K=K, N=N)
    if name == "gpt2s_upproj_fwd":
        return dict(x=outlier_normal_bf16(base + 0, (M, K)), w=normal_bf16(base + 1, (K, N), 0.02),
                    M=M, K=K, N=N)
    if name == "upproj_bwd":
        return dict(x=normal_bf16(base + 0, (M, K)), w=normal_bf16(base + 1, (K, N), 0.02),
                    dy=lognormal_grad_bf16(base + 2, (M, N)), M=M, K=K, N=N)
    if name == "finegrained_fwd":
        return dict(x=channel_scaled_bf16(base + 0, (M, K)), w=normal_bf16(base + 1, (K, N), 0.02),
                    M=M, K=K, N=N)
    if name == "delayed_loop":
        layers = w["layers"]
        return dict(x=normal_bf16(base + 0, (M, K)), dy=lognormal_grad_bf16(base + 2, (M, N)),
                    w=[normal_bf16(base + 100 + l, (K, N), 0.02) for l in range(layers)],
                    M=M, K=K, N=N, layers=layers, steps=w["steps"], hist_len=w["hist_len"],
                    perturb_seed=lambda layer, step: base + 10_000 + 100 * step + layer)
    raise KeyError(name)
