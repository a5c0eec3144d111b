"""The allocation-free backward entry point against the scratch-taking one.

fp8_linear_bwd_noalloc serves callers that cannot allocate device memory when they call
the backward (a framework that passes only its input and output tensors and forbids side
allocations, or a C program without a device allocator of its own): it keeps the E5M2
codes of dy in a static array inside the library. This file is collected last so that a
run stopping at its first failure has already run every other test.

Two calls in a row (different dy, so the second call must not reuse the first call's codes)
are compared with fp8_linear_bwd on the same inputs, through the C ABI. Both run the same
kernels on the same codes, so dx and dW must be bit-identical, and the dy scaling state
too; both are also checked against the oracle's exact sampled reference within the GEMM
bound (1e-3 * sum|a b| d_a d_b + 1 bf16 ulp). The dgrad-only form (no dW: no transposed
codes) is checked the same way. A further call leaves the device's free memory unchanged.
A shape beyond the static array is rejected."""
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


def bits_equal(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


class Forward:
    """A layer whose forward ran: the cached weight codes and the saved x codes."""

    def __init__(self, g, M, K, N, seed):
        self.M, self.K, self.N = M, K, N
        self.x_b = normal_bf16(seed, (M, K))
        self.w_b = normal_bf16(seed + 1, (K, N), 0.02)
        x, w = dev_bf16(self.x_b), dev_bf16(self.w_b)
        self.wst, self.xst = g.TensorState(), g.TensorState()
        self.wq, self.wqT, self.xq, self.xqT = empty_u8(K, N), empty_u8(N, K), empty_u8(M, K), empty_u8(K, M)
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        T, C = g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT
        g.fp8_requantize_weights(w, K, N, T, C, self.wst, self.wq, self.wqT)
        g.fp8_linear_fwd(x, M, K, N, self.wqT, self.wst, None, self.xst, T, C, self.xq, self.xqT, None, y)
        self.ox = quant.quantize_tensor(self.x_b, fp8.E4M3)
        self.ow = quant.quantize_tensor(self.w_b, fp8.E4M3)


def oracle_check(f, dy_b, dx, dw):
    """dx (and dW) against the oracle's exact sampled reference."""
    og = quant.quantize_tensor(dy_b, fp8.E5M2)
    rng = np.random.default_rng(int(dy_b[0, 0]))
    r, c = rng.integers(0, f.M, 2048), rng.integers(0, f.K, 2048)
    ref, mag = gemm.scaled_mm_sampled(og["q"], fp8.E5M2, f.ow["q"], fp8.E4M3, og["d"], f.ow["d"], r, c)
    within(host_bf16_f64(dx)[r, c], ref, mag)
    if dw is not None:
        r, c = rng.integers(0, f.K, 2048), rng.integers(0, f.N, 2048)
        ref, mag = gemm.scaled_mm_sampled(f.ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, f.ox["d"], og["d"], r, c)
        within(host_bf16_f64(dw)[r, c], ref, mag)


def run_pair(g, f, dy_b, with_dw):
    """fp8_linear_bwd (caller scratch) and fp8_linear_bwd_noalloc on the same dy."""
    M, K, N = f.M, f.K, f.N
    C = g.FP8_SCALE_CURRENT
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    dy = dev_bf16(dy_b)
    st_ref, st_na = g.TensorState(), g.TensorState()
    dyq, dyqT = empty_u8(M, N), (empty_u8(N, M) if with_dw else None)
    dx_ref, dx_na = bf(M, K), bf(M, K)
    dw_ref, dw_na = (bf(K, N), bf(K, N)) if with_dw else (None, None)
    g.fp8_linear_bwd(dy, M, K, N, f.xqT, f.xst, f.wq, f.wst, st_ref, C, dyq, dyqT, dx_ref, dw_ref)
    g.fp8_linear_bwd_noalloc(dy, M, K, N, f.xqT, f.xst, f.wq, f.wst, st_na, C, dx_na, dw_na)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    a, b = st_ref.snapshot(), st_na.snapshot()
    for k in ("scale", "scale_inv", "amax_cur", "overflow", "underflow"):
        assert a[k] == b[k], k
    assert bits_equal(dx_na, dx_ref)
    if with_dw:
        assert bits_equal(dw_na, dw_ref)
    return dx_na, dw_na


def test_noalloc_backward_matches_scratch_backward_twice(g):
    f = Forward(g, 1024, 384, 1536, 7100)
    for seed in (7102, 7103):
        dy_b = lognormal_grad_bf16(seed, (f.M, f.N))
        dx, dw = run_pair(g, f, dy_b, with_dw=True)
        oracle_check(f, dy_b, dx, dw)


def test_noalloc_dgrad_only_matches_scratch_backward_twice(g):
    """dW not requested: the array holds only the row-major dy codes (a larger M*N fits)."""
    f = Forward(g, 2048, 256, 2048, 7200)
    for seed in (7202, 7203):
        dy_b = lognormal_grad_bf16(seed, (f.M, f.N))
        dx, _ = run_pair(g, f, dy_b, with_dw=False)
        oracle_check(f, dy_b, dx, None)


def test_noalloc_backward_allocates_no_device_memory(g):
    """After a first call (which looks up the array's address), a second call changes the
    device's free memory by nothing."""
    f = Forward(g, 512, 256, 1024, 7300)
    dy = dev_bf16(lognormal_grad_bf16(7302, (f.M, f.N)))
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    dx, dw, st = bf(f.M, f.K), bf(f.K, f.N), g.TensorState()
    C = g.FP8_SCALE_CURRENT
    g.fp8_linear_bwd_noalloc(dy, f.M, f.K, f.N, f.xqT, f.xst, f.wq, f.wst, st, C, dx, dw)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    g.fp8_linear_bwd_noalloc(dy, f.M, f.K, f.N, f.xqT, f.xst, f.wq, f.wst, st, C, dx, dw)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    g.fp8_poll_device_error()
    assert free1 == free0


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
