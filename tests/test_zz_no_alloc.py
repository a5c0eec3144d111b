"""The allocation-free backward entry point against the scratch-taking one.

fp8_linear_bwd_noalloc serves callers that cannot allocate device memory when they call
the backward (a framework that passes only its input and output tensors and forbids side
allocations, or a C program without a device allocator of its own): it keeps the E5M2
codes of dy in a static array inside the library. This file is collected last so that a
run stopping at its first failure has already run every other test.

Two calls in a row (different dy, so the second call must not reuse the first call's codes)
are compared with fp8_linear_bwd on the same inputs, through the C ABI: dx and dW within the
tolerance the other GEMM tests use (1e-3 * sum|a b| d_a d_b + 1 bf16 ulp, magnitudes from the
oracle) and the dy scaling state bit for bit. A shape beyond the static array is rejected."""
import numpy as np
import pytest
import torch

from datagen import lognormal_grad_bf16, normal_bf16
from oracle import fp8, gemm, quant

from gpu_util import dev_bf16, empty_u8, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def within(a, b, mag):
    ok = gemm.within_bound(a, b, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"


def test_noalloc_backward_matches_scratch_backward_twice(g):
    M, K, N = 1024, 384, 1536
    x_b = normal_bf16(7100, (M, K))
    w_b = normal_bf16(7101, (K, N), 0.02)
    x, w = dev_bf16(x_b), dev_bf16(w_b)
    wst, xst = g.TensorState(), g.TensorState()
    wq, wqT, xq, xqT = empty_u8(K, N), empty_u8(N, K), empty_u8(M, K), empty_u8(K, M)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T, C = g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT
    g.fp8_requantize_weights(w, K, N, T, C, wst, wq, wqT)
    g.fp8_linear_fwd(x, M, K, N, wqT, wst, None, xst, T, C, xq, xqT, None, y)
    ox = quant.quantize_tensor(x_b, fp8.E4M3)
    ow = quant.quantize_tensor(w_b, fp8.E4M3)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    for call, seed in enumerate((7102, 7103)):
        dy_b = lognormal_grad_bf16(seed, (M, N))
        dy = dev_bf16(dy_b)
        # existing entry point, caller-provided scratch
        st_ref = g.TensorState()
        dyq, dyqT = empty_u8(M, N), empty_u8(N, M)
        dx_ref, dw_ref = bf(M, K), bf(K, N)
        g.fp8_linear_bwd(dy, M, K, N, xqT, xst, wq, wst, st_ref, C, dyq, dyqT, dx_ref, dw_ref)
        # allocation-free entry point
        st_na = g.TensorState()
        dx_na, dw_na = bf(M, K), bf(K, N)
        g.fp8_linear_bwd_noalloc(dy, M, K, N, xqT, xst, wq, wst, st_na, C, dx_na, dw_na)
        torch.cuda.synchronize()
        g.fp8_poll_device_error()
        a, b = st_ref.snapshot(), st_na.snapshot()
        for k in ("scale", "scale_inv", "amax_cur", "overflow", "underflow"):
            assert a[k] == b[k], (call, k)
        og = quant.quantize_tensor(dy_b, fp8.E5M2)
        _, mag_dx, _ = gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"])
        _, mag_dw, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
        within(host_bf16_f64(dx_na), host_bf16_f64(dx_ref), mag_dx)
        within(host_bf16_f64(dw_na), host_bf16_f64(dw_ref), mag_dw)


def test_noalloc_backward_rejects_shapes_beyond_the_static_array(g):
    """Shapes whose codes do not fit the 64 MiB array are refused before anything runs."""
    st = g.TensorState()
    tiny = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never touched: the call is refused
    # with wgrad: 2 x 32 Mi codes plus padding exceeds 64 MiB
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_linear_bwd_noalloc(tiny, 8192, 64, 4096 + 16, tiny, st, tiny, st, st, g.FP8_SCALE_CURRENT, tiny, tiny)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED and "static array" in e.value.detail
    # dgrad only: 64 Mi + 128 Ki codes exceed 64 MiB
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_linear_bwd_noalloc(tiny, 8192, 64, 8192 + 16, tiny, st, tiny, st, st, g.FP8_SCALE_CURRENT, tiny, None)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED and "static array" in e.value.detail
    torch.cuda.synchronize()
    assert float(tiny.float().abs().sum()) == float(tiny.float().abs().sum())  # context still usable
