"""Pins of the oracle's scaled matmuls: exact rational brute force on tiny shapes with
non-square operands (full and sampled forms, every format pair), the identity operand, the
bf16 rounding (fp64 and exact-rational forms) against torch's fp32->bf16 conversion, a sum
whose small term fp64 summation loses, the block-scaled form's reductions to the
per-tensor form, and the bound."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8, gemm


def rand_codes(rng, shape, fmt):
    """Random finite codes (no NaN / inf)."""
    tab = fp8.decode_table(fmt)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c])], dtype=np.uint8)
    return rng.choice(ok, size=shape)


@pytest.mark.parametrize("fa,fb", [(fp8.E4M3, fp8.E4M3), (fp8.E5M2, fp8.E4M3), (fp8.E4M3, fp8.E5M2)])
def test_brute_force_rational_tiny(fa, fb):
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 7
    A = rand_codes(rng, (M, K), fa)
    B = rand_codes(rng, (N, K), fb)
    d_a, d_b = np.float32(0.375), np.float32(1.0 / 3.0)
    ref, mag, dd = gemm.scaled_mm(A, fa, B, fb, d_a, d_b)
    assert ref.shape == (M, N)
    dd_exact = Fraction(float(np.float32(d_a * d_b)))
    assert Fraction(float(dd)) == dd_exact
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(fp8.decode(int(A[i, k]), fa)) * Fraction(fp8.decode(int(B[j, k]), fb)) for k in range(K))
            exact = float(dd_exact * s)        # float64 of the exact product (one rounding)
            want = gemm.bf16_round(np.array([exact]))[0]
            assert ref[i, j] == want, (i, j)
            m = sum(abs(Fraction(fp8.decode(int(A[i, k]), fa)) * Fraction(fp8.decode(int(B[j, k]), fb))) for k in range(K))
            assert mag[i, j] == pytest.approx(float(m) * float(d_a) * float(d_b), rel=1e-15)


def test_integer_products_exact():
    # codes whose values are small integers: E4M3 1, 2, 3 = 0x38, 0x40, 0x44
    vals = {0x38: 1, 0x40: 2, 0x44: 3, 0xB8: -1, 0xC0: -2}
    rng = np.random.default_rng(1)
    keys = np.array(list(vals), dtype=np.uint8)
    A = rng.choice(keys, size=(4, 9))
    B = rng.choice(keys, size=(6, 9))
    ref, _, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 1.0, 1.0)
    want = np.array([[sum(vals[int(A[i, k])] * vals[int(B[j, k])] for k in range(9)) for j in range(6)] for i in range(4)])
    assert np.array_equal(ref, want.astype(np.float64))


@pytest.mark.parametrize("fa,one", [(fp8.E4M3, 0x38), (fp8.E5M2, 0x3C)])
def test_identity_operand(fa, one):
    rng = np.random.default_rng(2)
    K = 16
    A = rand_codes(rng, (10, K), fa)
    B = np.zeros((K, K), dtype=np.uint8)
    B[np.arange(K), np.arange(K)] = one
    # d has 8 significant bits, so decode(A) * d has at most 12 and is exact in float32:
    # torch's float32 -> bf16 conversion then rounds the exact product once
    d = np.float32(float(torch.tensor(0.0123).to(torch.bfloat16)))
    prod = fp8.decode_array(A, fa) * np.float64(d)
    assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)
    ref, _, _ = gemm.scaled_mm(A, fa, B, fa, d, 1.0)
    want = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ref, want)


def test_bf16_round_against_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(10.0) ** rng.integers(-40, 38, 100000).astype(np.float32),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.3895e38, 3.4e38, 1e-40, -1e-40, 2 ** -133, 3 * 2 ** -134], dtype=np.float32),
    ]).astype(np.float32)
    v = v[np.isfinite(v)]
    ours = gemm.bf16_round(v.astype(np.float64))
    theirs = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)


def test_block_scaled_reduces_to_per_tensor():
    rng = np.random.default_rng(5)
    M, N, K = 4, 256, 256
    A = rand_codes(rng, (M, K), fp8.E4M3)
    B = rand_codes(rng, (N, K), fp8.E4M3)
    da = np.full((M, K // 128), 0.5, dtype=np.float32)
    db = np.full((K // 128, N // 128), 0.25, dtype=np.float32)
    blk, bmag = gemm.block_scaled_mm(A, fp8.E4M3, da, B, fp8.E4M3, db)
    ref, mag, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 0.5, 0.25)
    assert np.array_equal(blk, ref)
    assert np.allclose(bmag, mag, rtol=1e-15)


def test_block_scaled_rational_with_distinct_scales():
    rng = np.random.default_rng(6)
    M, N, K = 2, 256, 256
    A = rand_codes(rng, (M, K), fp8.E5M2)
    B = rand_codes(rng, (N, K), fp8.E4M3)
    da = rng.uniform(0.1, 2, size=(M, 2)).astype(np.float32)
    db = rng.uniform(0.1, 2, size=(2, 2)).astype(np.float32)
    blk, _ = gemm.block_scaled_mm(A, fp8.E5M2, da, B, fp8.E4M3, db)
    for i in range(M):
        for j in (0, 1, 127, 128, 200, 255):
            tot = Fraction(0)
            for kb in range(2):
                sc = Fraction(float(np.float32(da[i, kb] * db[kb, j // 128])))
                p = sum(Fraction(fp8.decode(int(A[i, k]), fp8.E5M2)) * Fraction(fp8.decode(int(B[j, k]), fp8.E4M3))
                        for k in range(kb * 128, kb * 128 + 128))
                tot += sc * p
            want = gemm.bf16_round(np.array([float(tot)]))[0]
            assert blk[i, j] == want
    # sampled form agrees with the full form
    rows = np.array([0, 1, 1]); cols = np.array([5, 130, 255])
    s, _ = gemm.block_scaled_mm_sampled(A, fp8.E5M2, da, B, fp8.E4M3, db, rows, cols)
    assert np.array_equal(s, blk[rows, cols])
    for t, (i, j) in enumerate(zip(rows, cols)):
        tot = Fraction(0)
        for kb in range(2):
            sc = Fraction(float(np.float32(da[i, kb] * db[kb, j // 128])))
            tot += sc * sum(Fraction(fp8.decode(int(A[i, k]), fp8.E5M2)) * Fraction(fp8.decode(int(B[j, k]), fp8.E4M3))
                            for k in range(kb * 128, kb * 128 + 128))
        assert s[t] == gemm.bf16_round_exact(tot)


def test_sampled_matches_full():
    rng = np.random.default_rng(8)
    A = rand_codes(rng, (9, 40), fp8.E4M3)
    B = rand_codes(rng, (11, 40), fp8.E5M2)
    full, mag, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E5M2, 0.7, 1.3)
    rows = rng.integers(0, 9, 30); cols = rng.integers(0, 11, 30)
    s, m = gemm.scaled_mm_sampled(A, fp8.E4M3, B, fp8.E5M2, 0.7, 1.3, rows, cols)
    assert np.array_equal(s, full[rows, cols])
    assert np.allclose(m, mag[rows, cols], rtol=1e-15)


def test_bound_rejects_planted_errors():
    ref = np.array([1.0, 100.0, 0.0])
    mag = np.array([0.0, 0.0, 0.0])
    assert gemm.within_bound(ref, ref, mag).all()
    one_ulp = ref + gemm.bf16_ulp(ref)
    assert gemm.within_bound(one_ulp, ref, mag).all()
    two_ulp = ref + 2 * gemm.bf16_ulp(ref)
    assert not gemm.within_bound(two_ulp, ref, mag).any()
    # a transposed result fails on a non-symmetric product
    rng = np.random.default_rng(9)
    A = rand_codes(rng, (6, 32), fp8.E4M3)
    B = rand_codes(rng, (6, 32), fp8.E4M3)
    r, m, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 1.0, 1.0)
    assert not gemm.within_bound(r.T, r, m).all()


@pytest.mark.parametrize("fa,fb", [(fp8.E4M3, fp8.E4M3), (fp8.E5M2, fp8.E4M3), (fp8.E4M3, fp8.E5M2),
                                   (fp8.E5M2, fp8.E5M2)])
def test_exact_sampled_against_fraction(fa, fb):
    """The sampled reference is the definition computed exactly: rational brute force over
    random finite codes of every format pair (extremes included) and random fp32 scales."""
    rng = np.random.default_rng(12)
    M, N, K = 5, 6, 300
    A = rand_codes(rng, (M, K), fa)
    B = rand_codes(rng, (N, K), fb)
    A[0, :4] = [0x7E if fa == fp8.E4M3 else 0x7B, 0x01, 0xFE if fa == fp8.E4M3 else 0xFB, 0x80]
    d_a, d_b = np.float32(rng.uniform(1e-3, 10)), np.float32(rng.uniform(1e-3, 10))
    rows = np.repeat(np.arange(M), N)
    cols = np.tile(np.arange(N), M)
    ref, mag = gemm.scaled_mm_sampled(A, fa, B, fb, d_a, d_b, rows, cols)
    dd = Fraction(float(np.float32(d_a * d_b)))
    for t, (i, j) in enumerate(zip(rows, cols)):
        s = sum(Fraction(fp8.decode(int(A[i, k]), fa)) * Fraction(fp8.decode(int(B[j, k]), fb)) for k in range(K))
        want = gemm.bf16_round_exact(dd * s)
        assert ref[t] == want, (i, j)
        m = sum(abs(Fraction(fp8.decode(int(A[i, k]), fa)) * Fraction(fp8.decode(int(B[j, k]), fb))) for k in range(K))
        assert mag[t] == pytest.approx(float(m) * float(d_a) * float(d_b), rel=1e-12)


def test_exact_sampled_keeps_a_term_fp64_summation_loses():
    """Sixty-four E5M2-max x E4M3-max products, one product of the smallest subnormals, then
    the negated large products: the real sum is 2^-25. fp64 summation in this order loses the
    small term (the partial sum is near 2^30.6, whose fp64 spacing is 2^-22); the exact
    reference keeps it."""
    big_a, big_b = 0x7B, 0x7E                 # 57344 (E5M2) and 448 (E4M3)
    A = np.array([[big_a] * 64 + [0x01] + [big_a | 0x80] * 64], dtype=np.uint8)
    B = np.array([[big_b] * 64 + [0x01] + [big_b] * 64], dtype=np.uint8)
    vals = [fp8.decode(int(a), fp8.E5M2) * fp8.decode(int(b), fp8.E4M3) for a, b in zip(A[0], B[0])]
    acc = 0.0
    for v in vals:                            # left-to-right fp64 summation
        acc += v
    assert acc == 0.0
    ref, _ = gemm.scaled_mm_sampled(A, fp8.E5M2, B, fp8.E4M3, 1.0, 1.0, np.array([0]), np.array([0]))
    assert ref[0] == 2.0 ** -25


def test_bf16_round_exact_against_torch_and_ties():
    rng = np.random.default_rng(13)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000)).astype(np.float32)
    v = np.concatenate([v[np.isfinite(v)], np.array([3.3895e38, 1e-40, -1e-40, 2 ** -133], dtype=np.float32)])
    theirs = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([gemm.bf16_round_exact(Fraction(float(x))) for x in v])
    assert np.array_equal(ours, theirs)
    # exact ties between bf16 neighbours (1 + 2^-8 lies halfway between 1 and 1 + 2^-7)
    assert gemm.bf16_round_exact(Fraction(1) + Fraction(1, 256)) == 1.0
    assert gemm.bf16_round_exact(Fraction(1) + Fraction(3, 256)) == 1.0 + 2 ** -6
    assert gemm.bf16_round_exact(-(Fraction(1) + Fraction(1, 256) + Fraction(1, 2 ** 60))) == -(1.0 + 2 ** -7)
    assert gemm.bf16_round_exact(Fraction(2) ** 128) == float("inf")
    assert gemm.bf16_round_exact(Fraction(3, 2 ** 135)) == 2.0 ** -133      # 1.5 subnormal ulps -> even


def test_mx_reduces_to_per_tensor_with_equal_exponents():
    rng = np.random.default_rng(70)
    A = rand_codes(rng, (5, 128), fp8.E4M3)
    B = rand_codes(rng, (7, 128), fp8.E5M2)
    ea = np.full((5, 4), -3)
    eb = np.full((7, 4), 2)
    mx_full, mx_mag = gemm.mx_scaled_mm(A, fp8.E4M3, ea, B, fp8.E5M2, eb)
    ref, mag, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E5M2, 2.0 ** -3, 2.0 ** 2)
    assert np.array_equal(mx_full, ref)
    assert np.allclose(mx_mag, mag, rtol=1e-15)


@pytest.mark.parametrize("fa,fb", [(fp8.E4M3, fp8.E4M3), (fp8.E5M2, fp8.E4M3)])
def test_mx_rational_with_distinct_exponents(fa, fb):
    rng = np.random.default_rng(71)
    M, N, K = 3, 4, 96
    A = rand_codes(rng, (M, K), fa)
    B = rand_codes(rng, (N, K), fb)
    ea = rng.integers(-30, 30, size=(M, K // 32))
    eb = rng.integers(-30, 30, size=(N, K // 32))
    full, _ = gemm.mx_scaled_mm(A, fa, ea, B, fb, eb)
    rows = np.repeat(np.arange(M), N)
    cols = np.tile(np.arange(N), M)
    samp, _ = gemm.mx_scaled_mm_sampled(A, fa, ea, B, fb, eb, rows, cols)
    for t, (i, j) in enumerate(zip(rows, cols)):
        tot = Fraction(0)
        for g in range(K // 32):
            sc = Fraction(2) ** int(ea[i, g] + eb[j, g])
            tot += sc * sum(Fraction(fp8.decode(int(A[i, k]), fa)) * Fraction(fp8.decode(int(B[j, k]), fb))
                            for k in range(32 * g, 32 * g + 32))
        want = gemm.bf16_round_exact(tot)
        assert samp[t] == want
        assert full[i, j] == want
