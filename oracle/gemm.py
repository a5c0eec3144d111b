"""Scaled FP8 matmuls and the error bound (oracle; test infrastructure).

Source: "#84 FP8 Precision" page, "Explanation" and its code: the FP8 matmul takes
the two quantised operands and one scale per operand and returns a high-precision
result; "Hardware precision": FP8 tensor cores.  "FP8 stability guardrails" page,
"Real products, models, and research": per-tile / per-block scales (DeepSeek-V3).

Definitions (A [M,K] and B [N,K] are code arrays, both contracted over K):
* per-tensor:   C_ij = bf16( fl32(d_a * d_b) * sum_k a_ik * b_jk )
* block scaled: C_ij = bf16( sum_kb fl32(d_a[i,kb] * d_b[kb, j // 128]) * P_ij,kb ),
                P_ij,kb = sum over k in K-block kb of a_ik * b_jk
with a, b the decoded FP8 values, every sum exact (fp64 of short products) and bf16 the
round-to-nearest-even rounding of the real result.
Accepted error of an fp32-accumulating implementation:
    |C - C_ref| <= 1e-3 * sum_k |a_ik * b_jk| * d_a * d_b + 1 bf16 ulp(C_ref).

Pins (tests/test_oracle_gemm.py): integer-valued products summed exactly and compared
with Python integer arithmetic, the identity operand, and the bf16 rounding against
torch's fp32->bf16 conversion.
"""
from __future__ import annotations

import numpy as np

from . import fp8

TILE = 128
REL_TOL = 1e-3


def bf16_round(x) -> np.ndarray:
    """Round real values (fp64) to bf16 with ties to even; returns the rounded fp64 values."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, ex = np.frexp(np.where(fin, x, 1.0))          # |x| in [2^(ex-1), 2^ex)
    e = np.maximum(ex - 1, -126)                       # bf16 exponent, subnormals share -126
    ulp_exp = e - 7                                    # 8 significant bits
    q = np.ldexp(np.where(fin, x, 0.0), -ulp_exp)
    r = np.rint(q)                                     # round half to even
    val = np.ldexp(r, ulp_exp)
    val = np.where(np.abs(val) >= 2.0 ** 128, np.copysign(np.inf, x), val)
    out[fin] = val[fin]
    return out


def bf16_ulp(c) -> np.ndarray:
    """Spacing of bf16 numbers at |c| (fp64)."""
    c = np.asarray(c, dtype=np.float64)
    _, ex = np.frexp(np.where(np.isfinite(c) & (c != 0), c, 1.0))
    e = np.where(np.isfinite(c) & (c != 0), np.maximum(ex - 1, -126), -126)
    return np.ldexp(1.0, e - 7)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _dec(codes, fmt):
    return fp8.decode_array(codes, fmt)


def scaled_mm(a_codes, fa, b_codes, fb, d_a, d_b):
    """Per-tensor scaled matmul; returns (C_ref fp64 bf16-rounded, sum|a*b| fp64, dd)."""
    A = _dec(a_codes, fa)
    B = _dec(b_codes, fb)
    S = A @ B.T
    mag = np.abs(A) @ np.abs(B).T
    dd = np.float32(np.float32(d_a) * np.float32(d_b))
    return bf16_round(np.float64(dd) * S), mag * float(d_a) * float(d_b), dd


def scaled_mm_sampled(a_codes, fa, b_codes, fb, d_a, d_b, rows, cols):
    """The same definition for selected outputs (rows[i], cols[i]) only."""
    A = _dec(a_codes[rows], fa)
    B = _dec(b_codes[cols], fb)
    S = np.einsum("ik,ik->i", A, B)
    mag = np.einsum("ik,ik->i", np.abs(A), np.abs(B))
    dd = np.float32(np.float32(d_a) * np.float32(d_b))
    return bf16_round(np.float64(dd) * S), mag * float(d_a) * float(d_b)


def block_scaled_mm(a_codes, fa, d_a, b_codes, fb, d_b):
    """1x128-tile scaled A [M,K] (d_a [M, K/128]) times 128x128-block scaled B given as
    [N,K] codes with d_b [K/128, N/128].  Returns (C_ref, bound magnitude)."""
    A = _dec(a_codes, fa)
    B = _dec(b_codes, fb)
    M, K = A.shape
    N = B.shape[0]
    KB = K // TILE
    acc = np.zeros((M, N), dtype=np.float64)
    mag = np.zeros((M, N), dtype=np.float64)
    nb = np.arange(N) // TILE
    for kb in range(KB):
        ks = slice(kb * TILE, (kb + 1) * TILE)
        P = A[:, ks] @ B[:, ks].T
        Pm = np.abs(A[:, ks]) @ np.abs(B[:, ks]).T
        sc = (d_a[:, kb][:, None].astype(np.float32) * d_b[kb, nb][None, :].astype(np.float32)).astype(np.float32)
        acc += sc.astype(np.float64) * P
        mag += sc.astype(np.float64) * Pm
    return bf16_round(acc), mag


def block_scaled_mm_sampled(a_codes, fa, d_a, b_codes, fb, d_b, rows, cols):
    A = _dec(a_codes[rows], fa)
    B = _dec(b_codes[cols], fb)
    K = A.shape[1]
    acc = np.zeros(len(rows))
    mag = np.zeros(len(rows))
    for kb in range(K // TILE):
        ks = slice(kb * TILE, (kb + 1) * TILE)
        P = np.einsum("ik,ik->i", A[:, ks], B[:, ks])
        Pm = np.einsum("ik,ik->i", np.abs(A[:, ks]), np.abs(B[:, ks]))
        sc = (d_a[rows, kb].astype(np.float32) * d_b[kb, cols // TILE].astype(np.float32)).astype(np.float32)
        acc += sc.astype(np.float64) * P
        mag += sc.astype(np.float64) * Pm
    return bf16_round(acc), mag


def within_bound(c_test, c_ref, mag):
    """Boolean mask: |c_test - c_ref| <= 1e-3 * mag + ulp_bf16(c_ref)."""
    c_test = np.asarray(c_test, dtype=np.float64)
    err = np.abs(c_test - c_ref)
    return err <= REL_TOL * mag + bf16_ulp(c_ref)
