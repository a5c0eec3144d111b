"""Operands read MN-major: fp8_scaled_mm_t (C = A^T B with A [K, M] and B [K, N] row-major) and
fp8_linear_bwd_mn (the weight gradient from x's and dy's codes as the casts write them, with no
transposed copies) against the oracle.

Small shapes in full (single CTAs and CTA pairs, 128- and 256-wide tiles, ragged M, N and K,
every format pair, split K through the workspace); the backward's dx bit for bit against
fp8_linear_bwd (the same dgrad launch) and dW against the oracle; the backward workload at full
size on sampled outputs."""
import numpy as np
import pytest
import torch

from datagen import lognormal_grad_bf16, normal_bf16, workload_inputs
from oracle import fp8, gemm, quant

from gpu_util import dev_bf16, dev_u8, empty_u8, f32_scalar, host_bf16_f64, host_u8

pytestmark = pytest.mark.gpu
FMTS = {0: fp8.E4M3, 1: fp8.E5M2}


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def finite_codes(rng, shape, fmt):
    ok = np.array([c for c in range(256) if np.isfinite(fp8.decode(c, fmt))], dtype=np.uint8)
    return rng.choice(ok, size=shape)


def within(got, ref, mag):
    ok = gemm.within_bound(got, ref, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"


@pytest.mark.parametrize("M,N,K,fa,fb", [(128, 256, 128, 0, 0), (112, 208, 64, 0, 1), (384, 512, 256, 0, 1),
                                         (304, 704, 160, 1, 0), (1024, 1536, 512, 0, 1), (640, 128, 1024, 1, 1),
                                         (256, 384, 8192, 0, 1)])
def test_scaled_mm_t_against_oracle(g, M, N, K, fa, fb):
    rng = np.random.default_rng(M + 3 * N + K)
    A = finite_codes(rng, (K, M), FMTS[fa])      # [K, M], the contraction along rows
    B = finite_codes(rng, (K, N), FMTS[fb])
    da, db = np.float32(rng.uniform(0.01, 2)), np.float32(rng.uniform(0.01, 2))
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    wsb = g.fp8_scaled_mm_workspace_bytes(M, N, K)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    g.fp8_scaled_mm_t(dev_u8(A), fa, dev_u8(B), fb, M, N, K, M, N, f32_scalar(da), f32_scalar(db), C, N, ws, wsb)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    ref, mag, _ = gemm.scaled_mm(np.ascontiguousarray(A.T), FMTS[fa], np.ascontiguousarray(B.T), FMTS[fb], da, db)
    within(host_bf16_f64(C), ref, mag)


@pytest.mark.parametrize("pa,pb", [((640, 384, 256, 0, 1), (256, 640, 384, 1, 0)),
                                   ((1024, 1536, 4096, 0, 1), (4096, 1024, 512, 1, 0))])
def test_grouped_mn_major_beside_k_major(g, pa, pb):
    """One grouped launch of an MN-major problem (A [K, M], B [K, N]) beside a K-major one, split
    K through the workspace; each against the oracle."""
    rng = np.random.default_rng(pa[0] + pb[2])
    probs, keep = [], []
    for (M, N, K, fa, fb), mn in ((pa, 1), (pb, 0)):
        sa, sb = np.float32(rng.uniform(0.05, 2)), np.float32(rng.uniform(0.05, 2))
        if mn:
            A, B = finite_codes(rng, (K, M), FMTS[fa]), finite_codes(rng, (K, N), FMTS[fb])
            Ar, Br, lda, ldb = A.T, B.T, M, N
        else:
            A, B = finite_codes(rng, (M, K), FMTS[fa]), finite_codes(rng, (N, K), FMTS[fb])
            Ar, Br, lda, ldb = A, B, K, K
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        Ad, Bd, da, db = dev_u8(A), dev_u8(B), f32_scalar(sa), f32_scalar(sb)
        keep += [Ad, Bd, da, db]
        probs.append(g.mm_problem(Ad, fa, Bd, fb, M, N, K, lda, ldb, da, db, C, N, mn_major=mn))
        keep.append((C, np.ascontiguousarray(Ar), FMTS[fa], np.ascontiguousarray(Br), FMTS[fb], sa, sb))
    nbytes = g.fp8_scaled_mm_grouped_workspace_bytes(probs)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    g.fp8_scaled_mm_grouped(probs, ws, nbytes)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    for C, A, fa, B, fb, sa, sb in (k for k in keep if isinstance(k, tuple)):
        ref, mag, _ = gemm.scaled_mm(A, fa, B, fb, sa, sb)
        within(host_bf16_f64(C), ref, mag)


def test_scaled_mm_t_padded_leading_dimensions(g):
    rng = np.random.default_rng(5)
    M, N, K, lda, ldb, ldc = 200, 300, 256, 224, 320, 304
    A = finite_codes(rng, (K, lda), fp8.E4M3)
    B = finite_codes(rng, (K, ldb), fp8.E5M2)
    C = torch.zeros(M, ldc, dtype=torch.bfloat16, device="cuda")
    g.fp8_scaled_mm_t(dev_u8(A), 0, dev_u8(B), 1, M, N, K, lda, ldb, f32_scalar(0.5), f32_scalar(0.25), C, ldc)
    torch.cuda.synchronize()
    ref, mag, _ = gemm.scaled_mm(np.ascontiguousarray(A[:, :M].T), fp8.E4M3, np.ascontiguousarray(B[:, :N].T),
                                 fp8.E5M2, 0.5, 0.25)
    got = host_bf16_f64(C)
    within(got[:, :N], ref, mag)
    assert np.all(got[:, N:] == 0)


def run_forward(g, x_b, w_b, M, K, N):
    x, w = dev_bf16(x_b), dev_bf16(w_b)
    wst, xst = g.TensorState(), g.TensorState()
    wq, wqT, xq, xqT = empty_u8(K, N), empty_u8(N, K), empty_u8(M, K), empty_u8(K, M)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T, C = g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT
    g.fp8_requantize_weights(w, K, N, T, C, wst, wq, wqT)
    g.fp8_linear_fwd(x, M, K, N, wqT, wst, None, xst, T, C, xq, xqT, None, y)
    return wst, xst, wq, xq, xqT


@pytest.mark.parametrize("M,K,N", [(256, 128, 512), (2048, 384, 1536), (1040, 256, 272)])
def test_linear_bwd_mn_against_transposed_path_and_oracle(g, M, K, N):
    x_b = normal_bf16(7400 + M, (M, K))
    w_b = normal_bf16(7401 + M, (K, N), 0.02)
    dy_b = lognormal_grad_bf16(7402 + M, (M, N))
    wst, xst, wq, xq, xqT = run_forward(g, x_b, w_b, M, K, N)
    dy = dev_bf16(dy_b)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    C = g.FP8_SCALE_CURRENT
    wsb = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st_t, st_m = g.TensorState(), g.TensorState()
    dyq_t, dyqT, dx_t, dw_t = empty_u8(M, N), empty_u8(N, M), bf(M, K), bf(K, N)
    g.fp8_linear_bwd_ws(dy, M, K, N, xqT, xst, wq, wst, st_t, C, dyq_t, dyqT, dx_t, dw_t, ws, wsb)
    dyq_m, dx_m, dw_m = empty_u8(M, N), bf(M, K), bf(K, N)
    g.fp8_linear_bwd_mn(dy, M, K, N, xq, xst, wq, wst, st_m, C, dyq_m, dx_m, dw_m, ws, wsb)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    assert torch.equal(dyq_m, dyq_t)
    assert torch.equal(dx_m.view(torch.int16), dx_t.view(torch.int16))
    a, b = st_t.snapshot(), st_m.snapshot()
    for k in ("scale", "scale_inv", "amax_cur", "overflow", "underflow"):
        assert a[k] == b[k], k
    og = quant.quantize_tensor(dy_b, fp8.E5M2)
    ox = quant.quantize_tensor(x_b, fp8.E4M3)
    assert np.array_equal(host_u8(dyq_m), og["q"])
    ref, mag, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    within(host_bf16_f64(dw_m), ref, mag)


def test_linear_bwd_mn_wgrad_only_and_empty_batch(g):
    M, K, N = 512, 256, 768
    x_b = normal_bf16(7500, (M, K))
    w_b = normal_bf16(7501, (K, N), 0.02)
    dy_b = lognormal_grad_bf16(7502, (M, N))
    wst, xst, wq, xq, xqT = run_forward(g, x_b, w_b, M, K, N)
    st = g.TensorState()
    dyq, dw = empty_u8(M, N), torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    g.fp8_linear_bwd_mn(dev_bf16(dy_b), M, K, N, xq, xst, wq, wst, st, g.FP8_SCALE_CURRENT, dyq, None, dw)
    torch.cuda.synchronize()
    og = quant.quantize_tensor(dy_b, fp8.E5M2)
    ox = quant.quantize_tensor(x_b, fp8.E4M3)
    ref, mag, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    within(host_bf16_f64(dw), ref, mag)
    # an empty token batch writes dW as zeros
    dw0 = torch.full((K, N), 1.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_linear_bwd_mn(None, 0, K, N, None, xst, wq, wst, g.TensorState(), g.FP8_SCALE_CURRENT, None, None, dw0)
    torch.cuda.synchronize()
    assert float(dw0.float().abs().max()) == 0.0


@pytest.mark.slow
def test_linear_bwd_mn_full_size(g):
    """The backward workload (M=16384, K=1024, N=4096) through the MN-major path: 4096 sampled
    outputs of dx and of dW against the exact sampled reference."""
    w_in = workload_inputs("upproj_bwd")
    M, K, N = w_in["M"], w_in["K"], w_in["N"]
    wst, xst, wq, xq, xqT = run_forward(g, w_in["x"], w_in["w"], M, K, N)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    st = g.TensorState()
    dyq, dx, dw = empty_u8(M, N), bf(M, K), bf(K, N)
    wsb = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    g.fp8_linear_bwd_mn(dev_bf16(w_in["dy"]), M, K, N, xq, xst, wq, wst, st, g.FP8_SCALE_CURRENT, dyq, dx, dw, ws, wsb)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    og = quant.quantize_tensor(w_in["dy"], fp8.E5M2)
    ox = quant.quantize_tensor(w_in["x"], fp8.E4M3)
    ow = quant.quantize_tensor(w_in["w"], fp8.E4M3)
    assert np.array_equal(host_u8(dyq), og["q"])
    rng = np.random.default_rng(33)
    r, c = rng.integers(0, M, 4096), rng.integers(0, K, 4096)
    ref, mag = gemm.scaled_mm_sampled(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"], r, c)
    within(host_bf16_f64(dx)[r, c], ref, mag)
    r, c = rng.integers(0, K, 4096), rng.integers(0, N, 4096)
    ref, mag = gemm.scaled_mm_sampled(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"], r, c)
    within(host_bf16_f64(dw)[r, c], ref, mag)
