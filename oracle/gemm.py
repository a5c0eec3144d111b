"""Scaled FP8 matmuls and the error bound (oracle; test infrastructure).

Source: "#84 FP8 Precision" page, "Explanation" and its code: the FP8 matmul takes
the two quantised operands and one scale per operand and returns a high-precision
result; "Hardware precision": FP8 tensor cores.  "FP8 stability guardrails" page,
"Real products, models, and research": per-tile / per-block scales (DeepSeek-V3).

Definitions (A [M,K] and B [N,K] are code arrays, both contracted over K):
* per-tensor:   C_ij = bf16( fl32(d_a * d_b) * sum_k a_ik * b_jk )
* block scaled: C_ij = bf16( sum_kb fl32(d_a[i,kb] * d_b[kb, j // 128]) * P_ij,kb ),
                P_ij,kb = sum over k in K-block kb of a_ik * b_jk
* MX scaled:    C_ij = bf16( sum_g 2^(e_a[i,g] + e_b[j,g]) * P_ij,g ), P_ij,g the sum over the
                g-th group of 32 consecutive k (power-of-two scales, one per row and group)
with a, b the decoded FP8 values, the sums taken over the reals and bf16 the
round-to-nearest-even rounding of the real result.

How exactly each function meets the definition:
* ``scaled_mm_sampled`` and ``block_scaled_mm_sampled`` are exact.  Every finite E4M3
  value is an integer multiple of 2^-9 and every finite E5M2 value one of 2^-16, so each
  sum is an integer (Python's unbounded ints) times a power of two, the scales are exact
  rationals, and the final bf16 rounding is done on the exact rational.
* ``scaled_mm`` and ``block_scaled_mm`` sum in fp64 (a library matmul).  The products are
  exact in fp64; the sums are exact while every partial sum fits 53 bits (always for
  E4M3 x E4M3 products, multiples of 2^-18 below 2^17.6, up to K = 2^17; for a product
  with an E5M2 operand only while partial sums stay below 2^28).  Otherwise the rounding
  error of any summation order is at most K * 2^-53 * sum_k |a_ik b_jk| (the standard
  bound for recursive summation), below 1e-10 of the accepted error for K <= 2^20; the
  result can then differ from the exact definition only where the real result lies that
  close to a bf16 rounding boundary.
Accepted error of an fp32-accumulating implementation:
    |C - C_ref| <= 1e-3 * sum_k |a_ik * b_jk| * d_a * d_b + 1 bf16 ulp(C_ref).

Pins (tests/test_oracle_gemm.py): exact rational brute force (Python ``Fraction``) on
non-square shapes of every format pair, integer-valued products, the identity operand,
the bf16 rounding against torch's fp32->bf16 conversion, a sum whose small term fp64
summation loses and the exact reference keeps, and the block-scaled form's reduction to
the per-tensor form.
"""
from __future__ import annotations

from fractions import Fraction

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


# Every finite code of the format is an integer multiple of 2^-SHIFT (the smallest subnormal).
_SHIFT = {fp8.E4M3: 9, fp8.E5M2: 16}


def _int_table(fmt):
    """int64[256]: decode(c) * 2^SHIFT for every finite code (exact integers, |v| < 2^32),
    and the mask of the finite codes."""
    tab = fp8.decode_table(fmt)
    fin = np.isfinite(tab)
    out = np.zeros(256, dtype=np.int64)
    out[fin] = np.ldexp(tab[fin], _SHIFT[fmt]).astype(np.int64)
    assert np.array_equal(np.ldexp(out[fin].astype(np.float64), -_SHIFT[fmt]), tab[fin])
    return out, fin


def _exact_row_dots(ai, bi):
    """Exact sum_k ai[n, k] * bi[n, k] for int64 arrays with entries below 2^32 in magnitude,
    as Python ints.  ai is split as hi * 2^16 + lo (|hi| < 2^16, 0 <= lo < 2^16) so that each
    product stays below 2^48 and a chunk of 2^13 of them below 2^61 in int64."""
    n, K = ai.shape
    lo = ai & 0xFFFF
    hi = ai >> 16
    out = [0] * n
    ch = 1 << 13
    for k0 in range(0, K, ch):
        b = bi[:, k0:k0 + ch]
        s_hi = np.einsum("ik,ik->i", hi[:, k0:k0 + ch], b)
        s_lo = np.einsum("ik,ik->i", lo[:, k0:k0 + ch], b)
        for i in range(n):
            out[i] += (int(s_hi[i]) << 16) + int(s_lo[i])
    return out


def bf16_round_exact(v) -> float:
    """Round an exact rational (Fraction or int) to bf16, ties to even; returns a float."""
    v = Fraction(v)
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a < 2^(e+2)
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                                            # subnormals share 2^-126
    q = a / Fraction(2) ** (e - 7)                              # 8 significant bits
    r = q.numerator // q.denominator
    rem = q - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    mag = Fraction(r) * Fraction(2) ** (e - 7)
    out = float("inf") if mag >= Fraction(2) ** 128 else float(mag)
    return -out if v < 0 else out


def _sampled_ints(a_codes, fa, b_codes, fb, rows, cols):
    ta, oka = _int_table(fa)
    tb, okb = _int_table(fb)
    A = np.asarray(a_codes)[rows]
    B = np.asarray(b_codes)[cols]
    if not (oka[A].all() and okb[B].all()):
        raise ValueError("NaN or infinite codes among the sampled operands: use scaled_mm")
    return ta[A], tb[B], A, B


def scaled_mm_sampled(a_codes, fa, b_codes, fb, d_a, d_b, rows, cols):
    """The per-tensor definition for selected outputs (rows[i], cols[i]), computed exactly
    (integer sums); returns (C_ref, bound magnitude sum|a*b| * d_a * d_b)."""
    ai, bi, A, B = _sampled_ints(a_codes, fa, b_codes, fb, rows, cols)
    sums = _exact_row_dots(ai, bi)
    dd = Fraction(float(np.float32(np.float32(d_a) * np.float32(d_b))))
    unit = Fraction(1, 1 << (_SHIFT[fa] + _SHIFT[fb]))
    ref = np.array([bf16_round_exact(dd * s * unit) for s in sums], dtype=np.float64)
    mag = np.einsum("ik,ik->i", np.abs(_dec(A, fa)), np.abs(_dec(B, fb)))
    return ref, mag * float(d_a) * float(d_b)


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
    """The block-scaled definition for selected outputs, computed exactly: per K block an
    integer sum, times the exact fp32 scale product, summed as rationals, rounded once."""
    ai, bi, A, B = _sampled_ints(a_codes, fa, b_codes, fb, rows, cols)
    K = ai.shape[1]
    unit = Fraction(1, 1 << (_SHIFT[fa] + _SHIFT[fb]))
    tot = [Fraction(0)] * len(rows)
    mag = np.zeros(len(rows))
    Ad, Bd = np.abs(_dec(A, fa)), np.abs(_dec(B, fb))
    for kb in range(K // TILE):
        ks = slice(kb * TILE, (kb + 1) * TILE)
        sums = _exact_row_dots(ai[:, ks], bi[:, ks])
        sc = (d_a[rows, kb].astype(np.float32) * d_b[kb, cols // TILE].astype(np.float32)).astype(np.float32)
        for i in range(len(rows)):
            if sums[i]:
                tot[i] += Fraction(float(sc[i])) * sums[i]
        mag += sc.astype(np.float64) * np.einsum("ik,ik->i", Ad[:, ks], Bd[:, ks])
    ref = np.array([bf16_round_exact(t * unit) for t in tot], dtype=np.float64)
    return ref, mag


MX = 32


def mx_scaled_mm(a_codes, fa, e_a, b_codes, fb, e_b):
    """MX-scaled A [M,K] (exponents e_a [M, K/32]) times B [N,K] (e_b [N, K/32]).  Every
    term is a code product times a power of two, so each group's sum scaled by 2^(e_a + e_b)
    and the sum over groups are exact in fp64 while the partial sums fit 53 bits (the
    sampled form below is exact always).  Returns (C_ref, bound magnitude)."""
    A = _dec(a_codes, fa)
    B = _dec(b_codes, fb)
    M, K = A.shape
    acc = np.zeros((M, B.shape[0]))
    mag = np.zeros((M, B.shape[0]))
    for g in range(K // MX):
        ks = slice(g * MX, (g + 1) * MX)
        sc = np.ldexp(1.0, (np.asarray(e_a)[:, g][:, None] + np.asarray(e_b)[:, g][None, :]).astype(np.int64))
        acc += sc * (A[:, ks] @ B[:, ks].T)
        mag += sc * (np.abs(A[:, ks]) @ np.abs(B[:, ks]).T)
    return bf16_round(acc), mag


def mx_scaled_mm_sampled(a_codes, fa, e_a, b_codes, fb, e_b, rows, cols):
    """The MX definition for selected outputs, exactly: integer group sums times exact powers
    of two, rounded once."""
    ai, bi, A, B = _sampled_ints(a_codes, fa, b_codes, fb, rows, cols)
    K = ai.shape[1]
    unit = Fraction(1, 1 << (_SHIFT[fa] + _SHIFT[fb]))
    ea = np.asarray(e_a)[rows]
    eb = np.asarray(e_b)[cols]
    tot = [Fraction(0)] * len(rows)
    mag = np.zeros(len(rows))
    Ad, Bd = np.abs(_dec(A, fa)), np.abs(_dec(B, fb))
    for g in range(K // MX):
        ks = slice(g * MX, (g + 1) * MX)
        sums = _exact_row_dots(ai[:, ks], bi[:, ks])
        for i in range(len(rows)):
            if sums[i]:
                tot[i] += Fraction(2) ** int(ea[i, g] + eb[i, g]) * sums[i]
        mag += np.ldexp(1.0, (ea[:, g] + eb[:, g]).astype(np.int64)) * np.einsum("ik,ik->i", Ad[:, ks], Bd[:, ks])
    ref = np.array([bf16_round_exact(t * unit) for t in tot], dtype=np.float64)
    return ref, mag


def within_bound(c_test, c_ref, mag):
    """Boolean mask: |c_test - c_ref| <= 1e-3 * mag + ulp_bf16(c_ref)."""
    c_test = np.asarray(c_test, dtype=np.float64)
    err = np.abs(c_test - c_ref)
    return err <= REL_TOL * mag + bf16_ulp(c_ref)
