"""GPU parity on shapes whose tile raster ends in a short group: the GEMMs sweep the output
in groups of 16 (per-tensor) or 32 (block-scaled and MX on CTA pairs) row blocks of 256, and
the kernels map work units to tiles with host-computed multipliers, including one for the
last group's row count. These shapes have several groups and a one-row-block last group, on
the single-problem, split-K, grouped, block-scaled and MX launches; every output is compared
with the oracle within the GEMM bound (1e-3 * sum|a b| d_a d_b + 1 bf16 ulp)."""
import numpy as np
import pytest
import torch

from oracle import fp8, gemm

from gpu_util import dev_u8, f32_scalar, host_bf16_f64
from test_gpu_gemm import FMT, assert_close, rand_codes
from test_gpu_mx import small_int_codes, sf_tile

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def _dev_ab(A, B):
    return dev_u8(A), dev_u8(B)


@pytest.mark.parametrize("M,N,K,fa,fb", [(4352, 640, 384, 0, 1),   # 17 pair rows: groups of 16 and 1
                                         (4480, 384, 256, 1, 0)])  # 17.5: the last pair half empty
def test_per_tensor_short_last_group(g, M, N, K, fa, fb):
    rng = np.random.default_rng(M + 3 * N + K)
    A = rand_codes(rng, (M, K), FMT[fa], 20.0)
    B = rand_codes(rng, (N, K), FMT[fb], 20.0)
    da, db = np.float32(0.03), np.float32(0.07)
    Ad, Bd = _dev_ab(A, B)
    ref, mag, _ = gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(Ad, fa, Bd, fb, M, N, K, K, K, g.FP8_GRAN_TENSOR, f32_scalar(da), f32_scalar(db), C, N)
    torch.cuda.synchronize()
    assert_close(host_bf16_f64(C), ref, mag)
    # the same through the workspace entry point (split K where the shape asks for it)
    wsb = g.fp8_scaled_mm_workspace_bytes(M, N, K)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    C2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm_ws(Ad, fa, Bd, fb, M, N, K, K, K, g.FP8_GRAN_TENSOR, f32_scalar(da), f32_scalar(db), C2, N, ws, wsb)
    torch.cuda.synchronize()
    assert_close(host_bf16_f64(C2), ref, mag)


def test_split_k_short_last_group(g):
    """17 pair tiles of a long contraction: too few to fill the GPU, so each is split over the
    halves of K; compared on 2048 sampled outputs with the exact reference."""
    M, N, K = 4352, 256, 8192
    assert g.fp8_scaled_mm_workspace_bytes(M, N, K) > 0  # (the shape splits)
    rng = np.random.default_rng(11)
    A = rand_codes(rng, (M, K), fp8.E4M3, 10.0)
    B = rand_codes(rng, (N, K), fp8.E5M2, 10.0)
    da, db = np.float32(0.01), np.float32(0.02)
    Ad, Bd = _dev_ab(A, B)
    wsb = g.fp8_scaled_mm_workspace_bytes(M, N, K)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm_ws(Ad, 0, Bd, 1, M, N, K, K, K, g.FP8_GRAN_TENSOR, f32_scalar(da), f32_scalar(db), C, N, ws, wsb)
    torch.cuda.synchronize()
    got = host_bf16_f64(C)
    rows = np.concatenate([rng.integers(0, M, 1792), rng.integers(M - 256, M, 256)])  # the last group too
    cols = rng.integers(0, N, rows.size)
    ref, mag = gemm.scaled_mm_sampled(A, fp8.E4M3, B, fp8.E5M2, da, db, rows, cols)
    assert_close(got[rows, cols], ref, mag)


def test_grouped_short_last_group(g):
    """Two problems in one launch, the first with a short last raster group."""
    rng = np.random.default_rng(5)
    shapes = [(4352, 384, 256, 0, 0), (768, 640, 512, 1, 0)]
    probs, keep = [], []
    for M, N, K, fa, fb in shapes:
        A = rand_codes(rng, (M, K), FMT[fa], 20.0)
        B = rand_codes(rng, (N, K), FMT[fb], 20.0)
        da, db = np.float32(rng.uniform(0.01, 0.1)), np.float32(rng.uniform(0.01, 0.1))
        Ad, Bd = _dev_ab(A, B)
        sa, sb = f32_scalar(da), f32_scalar(db)
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        probs.append(g.mm_problem(Ad, fa, Bd, fb, M, N, K, K, K, sa, sb, C, N))
        keep.append((A, fa, B, fb, da, db, C, Ad, Bd, sa, sb))
    wsb = g.fp8_scaled_mm_grouped_workspace_bytes(probs)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    g.fp8_scaled_mm_grouped(probs, ws, wsb)
    torch.cuda.synchronize()
    for A, fa, B, fb, da, db, C, *_ in keep:
        ref, mag, _ = gemm.scaled_mm(A, FMT[fa], B, FMT[fb], da, db)
        assert_close(host_bf16_f64(C), ref, mag)


def test_block_scaled_short_last_group(g):
    """33 pair rows: one group of 32 and one of 1 (block-scaled raster groups hold 32)."""
    M, N, K = 8448, 384, 256
    rng = np.random.default_rng(21)
    A = rand_codes(rng, (M, K), fp8.E4M3, 100.0)
    B = rand_codes(rng, (N, K), fp8.E4M3, 100.0)
    da = (10.0 ** rng.uniform(-4, -1, size=(M, K // 128))).astype(np.float32)
    db = (10.0 ** rng.uniform(-4, -1, size=(K // 128, N // 128))).astype(np.float32)
    Ad, Bd = _dev_ab(A, B)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(Ad, 0, Bd, 0, M, N, K, K, K, g.FP8_GRAN_BLOCK_128x128, torch.from_numpy(da).cuda(),
                    torch.from_numpy(db).cuda(), C, N)
    torch.cuda.synchronize()
    ref, mag = gemm.block_scaled_mm(A, fp8.E4M3, da, B, fp8.E4M3, db)
    assert_close(host_bf16_f64(C), ref, mag)


def test_mx_short_last_group(g):
    """The MX GEMM on CTA pairs over 33 pair rows, exact on small-integer codes."""
    M, N, K = 8448, 256, 256
    rng = np.random.default_rng(31)
    A, _ = small_int_codes(rng, (M, K), fp8.E4M3)
    B, _ = small_int_codes(rng, (N, K), fp8.E4M3)
    ea = rng.integers(-4, 5, size=(M, K // 32))
    eb = rng.integers(-4, 5, size=(N, K // 32))
    sa = dev_u8(sf_tile((ea + 127).astype(np.uint8)))
    sb = dev_u8(sf_tile((eb + 127).astype(np.uint8)))
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm(dev_u8(A), 0, dev_u8(B), 0, M, N, K, K, K, g.FP8_GRAN_MX_1x32, sa, sb, C, N)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    ref, _ = gemm.mx_scaled_mm(A, fp8.E4M3, ea, B, fp8.E4M3, eb)
    assert np.array_equal(gemm.bf16_round(ref), ref)  # (the products and sums are exact in bf16)
    np.testing.assert_array_equal(host_bf16_f64(C), ref)
