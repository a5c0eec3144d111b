"""GPU parity of the split-K GEMM (fp8_scaled_mm_ws) against the oracle's exact products,
with the same bound as fp8_scaled_mm: |C - C_ref| <= 1e-3 * sum_k |a b| d_a d_b + 1 bf16 ulp.
Shapes are ones the library splits (few output tiles, long K): single-CTA and CTA-pair tiles,
ragged M, N and K."""
import numpy as np
import pytest
import torch

from oracle import fp8, gemm

from gpu_util import dev_u8, f32_scalar, host_bf16_f64
from test_gpu_gemm import FMT, assert_close, rand_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def run_ws(g, A, fa, B, fb, da, db, ws, nbytes):
    M, K = A.shape
    N = B.shape[0]
    lda = ldb = -(-K // 16) * 16
    ldc = -(-N // 8) * 8
    Ad = torch.zeros(M, lda, dtype=torch.uint8, device="cuda")
    Ad[:, :K] = dev_u8(A)
    Bd = torch.zeros(N, ldb, dtype=torch.uint8, device="cuda")
    Bd[:, :K] = dev_u8(B)
    C = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm_ws(Ad, fa, Bd, fb, M, N, K, lda, ldb, g.FP8_GRAN_TENSOR, f32_scalar(da), f32_scalar(db), C, ldc,
                       ws, nbytes)
    torch.cuda.synchronize()
    return host_bf16_f64(C)[:, :N]


SPLIT_CASES = [
    # M, N, K, fa, fb
    (256, 512, 4096, 0, 0),    # single-CTA 128-wide tiles, 32 K blocks in two halves
    (300, 520, 4000, 1, 0),    # ragged M, N and last K block
    (1024, 768, 8192, 0, 1),   # CTA-pair 256-wide tiles
    (768, 3072, 8192, 0, 1),   # the GPT-2-small weight gradient: pairs
]


@pytest.mark.parametrize("M,N,K,fa,fb", SPLIT_CASES)
def test_split_k_against_exact(g, M, N, K, fa, fb):
    nbytes = g.fp8_scaled_mm_workspace_bytes(M, N, K)
    assert nbytes > 0, "the library should split this shape"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(M + 3 * N + K)
    A = rand_codes(rng, (M, K), FMT[fa], 30.0)
    B = rand_codes(rng, (N, K), FMT[fb], 30.0)
    da, db = np.float32(rng.uniform(0.001, 0.1)), np.float32(rng.uniform(0.001, 0.1))
    got = run_ws(g, A, fa, B, fb, da, db, ws, nbytes)
    ref, mag, _ = gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)
    assert_close(got, ref, mag)
    # the same inputs give the same bits, whichever of a tile's two units finishes last; the
    # workspace is reusable without clearing
    again = run_ws(g, A, fa, B, fb, da, db, ws, nbytes)
    assert np.array_equal(got.view(np.uint64), again.view(np.uint64))
    g.fp8_poll_device_error()


def test_workspace_reused_across_shapes_and_small_workspace_falls_back(g):
    rng = np.random.default_rng(11)
    shapes = [(256, 512, 4096), (1024, 768, 8192), (256, 512, 4096)]
    big = max(g.fp8_scaled_mm_workspace_bytes(*s) for s in shapes)
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for M, N, K in shapes:
        A = rand_codes(rng, (M, K), fp8.E4M3, 20.0)
        B = rand_codes(rng, (N, K), fp8.E4M3, 20.0)
        ref, mag, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 0.01, 0.02)
        assert_close(run_ws(g, A, 0, B, 0, 0.01, 0.02, ws, big), ref, mag)
        # too small (and null) workspaces run the unsplit GEMM: still within the bound
        assert_close(run_ws(g, A, 0, B, 0, 0.01, 0.02, ws, 256), ref, mag)
        assert_close(run_ws(g, A, 0, B, 0, 0.01, 0.02, None, 0), ref, mag)


def test_unsplit_shapes_need_no_workspace(g):
    assert g.fp8_scaled_mm_workspace_bytes(8192, 3072, 768) == 0    # fills the GPU as it is
    assert g.fp8_scaled_mm_workspace_bytes(16384, 14336, 4096) == 0
    assert g.fp8_scaled_mm_workspace_bytes(0, 16, 16) == 0


def test_ws_rejections(g):
    one = f32_scalar(1.0)
    A = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    C = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_ws(A, 0, A, 0, 128, 128, 256, 256, 256, g.FP8_GRAN_BLOCK_128x128, one, one, C, 128, ws, 1024)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_ws(A, 0, A, 0, 128, 128, 256, 256, 256, g.FP8_GRAN_TENSOR, one, one, C, 128,
                           ws[8:].data_ptr(), 1000)
    assert e.value.status == g.FP8_ERR_ALIGNMENT
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_ws(A, 0, A, 0, 128, 128, 256, 256, 256, g.FP8_GRAN_TENSOR, one, one, C, 128, ws, -1)
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    g.fp8_poll_device_error()


def test_grouped_pair_against_exact(g):
    """Two GEMMs of different shapes and formats in one launch (the backward's dgrad and a
    split weight gradient), each against its exact product; then each alone."""
    rng = np.random.default_rng(21)
    shapes = [(384, 640, 4096, 0, 1), (4096, 384, 640, 1, 0)]  # wgrad-like (splits), dgrad-like
    probs, refs, outs, ops = [], [], [], []
    for M, N, K, fa, fb in shapes:
        A = rand_codes(rng, (M, K), FMT[fa], 20.0)
        B = rand_codes(rng, (N, K), FMT[fb], 20.0)
        da, db = np.float32(rng.uniform(0.001, 0.05)), np.float32(rng.uniform(0.001, 0.05))
        Ad, Bd = dev_u8(A), dev_u8(B)
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        sa, sb = f32_scalar(da), f32_scalar(db)
        ops.append((Ad, Bd, sa, sb))
        outs.append(C)
        probs.append(g.mm_problem(Ad, fa, Bd, fb, M, N, K, K, K, sa, sb, C, N))
        refs.append(gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)[:2])
    nbytes = g.fp8_scaled_mm_grouped_workspace_bytes(probs)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace without clearing
        g.fp8_scaled_mm_grouped(probs, ws, nbytes)
        torch.cuda.synchronize()
        for C, (ref, mag) in zip(outs, refs):
            assert_close(host_bf16_f64(C), ref, mag)
    g.fp8_scaled_mm_grouped(probs[:1])  # one problem, no workspace
    torch.cuda.synchronize()
    assert_close(host_bf16_f64(outs[0]), *refs[0])
    g.fp8_poll_device_error()


def test_grouped_rejections(g):
    one = f32_scalar(1.0)
    A = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    C = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    ok = g.mm_problem(A, 0, A, 0, 128, 128, 256, 256, 256, one, one, C, 128)
    bad_k = g.mm_problem(A, 0, A, 0, 128, 128, 0, 256, 256, one, one, C, 128)
    bad_ld = g.mm_problem(A, 0, A, 0, 128, 128, 256, 264, 256, one, one, C, 128)  # lda % 16 != 0
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_grouped([ok, bad_k])
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_grouped([ok, bad_ld])
    assert e.value.status == g.FP8_ERR_ALIGNMENT
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_scaled_mm_grouped([ok, ok, ok])
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    g.fp8_poll_device_error()


GROUP_CASES = [
    # (M, N, K, fa, fb) x 2: single CTAs (a problem with M <= 128), ragged N and K
    ((96, 520, 1000, 0, 1), (640, 200, 336, 1, 0)),
    # CTA pairs, units of very different lengths (explicit schedule)
    ((512, 512, 8192, 0, 0), (1024, 256, 256, 1, 0)),
    # CTA pairs, units of one length (round robin)
    ((512, 768, 1024, 0, 1), (768, 512, 1024, 1, 0)),
]


@pytest.mark.parametrize("pa,pb", GROUP_CASES)
def test_grouped_shapes_against_exact(g, pa, pb):
    rng = np.random.default_rng(pa[0] + pb[2])
    probs, refs, outs, keep = [], [], [], []
    for M, N, K, fa, fb in (pa, pb):
        A = rand_codes(rng, (M, K), FMT[fa], 25.0)
        B = rand_codes(rng, (N, K), FMT[fb], 25.0)
        da, db = np.float32(rng.uniform(0.001, 0.05)), np.float32(rng.uniform(0.001, 0.05))
        lda = ldb = -(-K // 16) * 16
        ldc = -(-N // 8) * 8
        Ad = torch.zeros(M, lda, dtype=torch.uint8, device="cuda")
        Ad[:, :K] = dev_u8(A)
        Bd = torch.zeros(N, ldb, dtype=torch.uint8, device="cuda")
        Bd[:, :K] = dev_u8(B)
        C = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
        sa, sb = f32_scalar(da), f32_scalar(db)
        keep.append((Ad, Bd, sa, sb))
        outs.append((C, N))
        probs.append(g.mm_problem(Ad, fa, Bd, fb, M, N, K, lda, ldb, sa, sb, C, ldc))
        refs.append(gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)[:2])
    nbytes = g.fp8_scaled_mm_grouped_workspace_bytes(probs)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    for w, nb in ((ws, nbytes), (None, 0)):
        for C, _ in outs:
            C.fill_(float("nan"))
        g.fp8_scaled_mm_grouped(probs, w, nb)
        torch.cuda.synchronize()
        for (C, N), (ref, mag) in zip(outs, refs):
            assert_close(host_bf16_f64(C)[:, :N], ref, mag)
            assert np.isnan(host_bf16_f64(C)[:, N:]).all()  # padding columns untouched
    g.fp8_poll_device_error()
