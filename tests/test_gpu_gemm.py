"""GPU parity of the tcgen05 FP8 GEMM against the oracle's exact products:
|C - C_ref| <= 1e-3 * sum_k |a b| d_a d_b + 1 bf16 ulp(C_ref), element by element."""
import numpy as np
import pytest
import torch

from oracle import fp8, gemm

from gpu_util import dev_u8, f32_scalar, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


FMT = {0: fp8.E4M3, 1: fp8.E5M2}


def rand_codes(rng, shape, fmt, spread=1.0):
    """Codes of scaled normal values (finite), with a few +-max and subnormal codes."""
    v = rng.standard_normal(size=shape) * spread
    c = fp8.cast(v, fmt)
    flat = c.reshape(-1)
    k = max(1, flat.size // 500)
    idx = rng.choice(flat.size, size=k, replace=False)
    mx = fp8.max_code(fmt)
    flat[idx[: k // 3]] = mx
    flat[idx[k // 3: 2 * k // 3]] = 0x80 | mx
    flat[idx[2 * k // 3:]] = rng.integers(1, 4, size=len(idx[2 * k // 3:])) | (rng.integers(0, 2, size=len(idx[2 * k // 3:])) << 7)
    return c


def run_mm(g, A, fa, B, fb, da, db, lda=None, ldb=None, ldc=None):
    M, K = A.shape
    N = B.shape[0]
    lda = lda or -(-K // 16) * 16
    ldb = ldb or -(-K // 16) * 16
    ldc = ldc or -(-N // 8) * 8
    Ad = torch.zeros(M, lda, dtype=torch.uint8, device="cuda")
    Ad[:, :K] = dev_u8(A)
    Bd = torch.zeros(N, ldb, dtype=torch.uint8, device="cuda")
    Bd[:, :K] = dev_u8(B)
    C = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(Ad, fa, Bd, fb, M, N, K, lda, ldb, g.FP8_GRAN_TENSOR, f32_scalar(da), f32_scalar(db), C, ldc)
    torch.cuda.synchronize()
    return host_bf16_f64(C)


def assert_close(got, ref, mag):
    ok = gemm.within_bound(got, ref, mag)
    if not ok.all():
        i = np.argwhere(~ok)[:8]
        pytest.fail(f"{(~ok).sum()} of {ok.size} outside the bound; e.g. {[(tuple(j), got[tuple(j)], ref[tuple(j)]) for j in i]}")


CASES = [
    # M, N, K, fa, fb
    (256, 512, 128, 0, 0),     # tiny forward shape
    (128, 256, 128, 0, 0),     # one tile
    (300, 200, 208, 0, 0),     # ragged M, N and K tail
    (129, 257, 64, 1, 0),      # K < one block
    (1, 16, 16, 0, 1),
    (16, 8, 32, 1, 1),
    (640, 768, 384, 1, 0),
    (4096, 4096, 256, 0, 0),   # 512 tiles: several per CTA
    (8192, 560, 256, 1, 0),    # 192-wide tiles, ragged last tile
]


@pytest.mark.parametrize("M,N,K,fa,fb", CASES)
def test_scaled_mm_against_exact(g, M, N, K, fa, fb):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    A = rand_codes(rng, (M, K), FMT[fa], 30.0)
    B = rand_codes(rng, (N, K), FMT[fb], 30.0)
    da, db = np.float32(rng.uniform(0.001, 0.1)), np.float32(rng.uniform(0.001, 0.1))
    got = run_mm(g, A, fa, B, fb, da, db)
    ref, mag, _ = gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)
    assert_close(got[:, :N], ref, mag)


def test_padded_leading_dimensions(g):
    rng = np.random.default_rng(3)
    M, N, K = 200, 264, 160
    A = rand_codes(rng, (M, K), fp8.E4M3)
    B = rand_codes(rng, (N, K), fp8.E5M2)
    got = run_mm(g, A, 0, B, 1, 0.5, 0.25, lda=192, ldb=176, ldc=272)
    ref, mag, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E5M2, 0.5, 0.25)
    assert_close(got[:, :N], ref, mag)
    assert np.isnan(got[:, N:]).all()  # columns beyond N untouched


@pytest.mark.parametrize("fa,one", [(0, 0x38), (1, 0x3C)])
def test_identity_operand_is_exact(g, fa, one):
    rng = np.random.default_rng(4)
    K = 256
    A = rand_codes(rng, (384, K), FMT[fa])
    B = np.zeros((K, K), dtype=np.uint8)
    B[np.arange(K), np.arange(K)] = one
    d = np.float32(0.01171875)  # 3 * 2^-8
    got = run_mm(g, A, fa, B, fa, d, 1.0)
    ref, _, _ = gemm.scaled_mm(A, FMT[fa], B, FMT[fa], d, 1.0)
    assert np.array_equal(got[:, :K], ref)


def test_integer_sums_are_exact(g):
    # values in {-2,-1,0,1,2}: every partial sum is an integer below 2^24, so fp32
    # accumulation is exact and the result must equal the exact bf16 rounding
    rng = np.random.default_rng(5)
    M, N, K = 256, 512, 1024
    vals = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40], dtype=np.uint8)
    A = rng.choice(vals, size=(M, K))
    B = rng.choice(vals, size=(N, K))
    got = run_mm(g, A, 0, B, 0, 1.0, 1.0)
    ref, _, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 1.0, 1.0)
    assert np.array_equal(got[:, :N], ref)


def test_k_zero_writes_zeros(g):
    C = torch.full((8, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    one = f32_scalar(1.0)
    g.fp8_scaled_mm(None, 0, None, 0, 8, 16, 0, 16, 16, g.FP8_GRAN_TENSOR, one, one, C, 16)
    torch.cuda.synchronize()
    assert (C.float() == 0).all()


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 384, 512), (300, 512, 1024), (1024, 1280, 640),
                                   # single CTAs at M = 128, CTA pairs above; ragged M; several tiles
                                   (128, 896, 512), (300, 896, 1024), (1024, 1792, 640), (512, 2688, 256)])
def test_block_scaled_against_exact(g, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = rand_codes(rng, (M, K), fp8.E4M3, 100.0)
    B = rand_codes(rng, (N, K), fp8.E4M3, 100.0)
    da = (10.0 ** rng.uniform(-4, -1, size=(M, K // 128))).astype(np.float32)
    db = (10.0 ** rng.uniform(-4, -1, size=(K // 128, N // 128))).astype(np.float32)
    Ad, Bd = dev_u8(A), dev_u8(B)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(Ad, 0, Bd, 0, M, N, K, K, K, g.FP8_GRAN_BLOCK_128x128, torch.from_numpy(da).cuda(),
                    torch.from_numpy(db).cuda(), C, N)
    torch.cuda.synchronize()
    ref, mag = gemm.block_scaled_mm(A, fp8.E4M3, da, B, fp8.E4M3, db)
    assert_close(host_bf16_f64(C), ref, mag)


def test_block_scaled_padded_ldc(g):
    """A padded ldc: the stores leave the padding columns alone."""
    M, N, K, ldc = 384, 896, 384, 960
    rng = np.random.default_rng(17)
    A = rand_codes(rng, (M, K), fp8.E4M3, 100.0)
    B = rand_codes(rng, (N, K), fp8.E4M3, 100.0)
    da = (10.0 ** rng.uniform(-4, -1, size=(M, K // 128))).astype(np.float32)
    db = (10.0 ** rng.uniform(-4, -1, size=(K // 128, N // 128))).astype(np.float32)
    C = torch.full((M, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(dev_u8(A), 0, dev_u8(B), 0, M, N, K, K, K, g.FP8_GRAN_BLOCK_128x128, torch.from_numpy(da).cuda(),
                    torch.from_numpy(db).cuda(), C, ldc)
    torch.cuda.synchronize()
    ref, mag = gemm.block_scaled_mm(A, fp8.E4M3, da, B, fp8.E4M3, db)
    got = host_bf16_f64(C)
    assert_close(got[:, :N], ref, mag)
    assert np.all(got[:, N:] == 7.0)


def test_gemm_rejections(g):
    one = f32_scalar(1.0)
    A = torch.zeros(16, 32, dtype=torch.uint8, device="cuda")
    C = torch.zeros(16, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm(A, 0, A, 0, 16, 16, 24, 24, 32, g.FP8_GRAN_TENSOR, one, one, C, 16)
    assert e.value.status == g.FP8_ERR_ALIGNMENT
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm(A, 0, A, 0, 16, 16, 32, 32, 32, g.FP8_GRAN_BLOCK_128x128, one, one, C, 16)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED
    g.fp8_poll_device_error()
