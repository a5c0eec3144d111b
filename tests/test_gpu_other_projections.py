"""The same FP8 path on the transformer block's other projections (QKV: d -> 3d,
down-projection: 4d -> d, attention output: d -> d): forward and backward through the C ABI
against the oracle, in full at reduced token counts and on sampled outputs at 8192 tokens."""
import numpy as np
import pytest
import torch

from datagen import normal_bf16, lognormal_grad_bf16
from oracle import fp8, gemm, quant

from gpu_util import dev_bf16, empty_u8, host_u8, host_bf16_f64

pytestmark = pytest.mark.gpu

D = 768
SHAPES = {"qkv": (D, 3 * D), "down": (4 * D, D), "attn_out": (D, D)}


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def run(g, M, K, N, seed):
    x_b = normal_bf16(seed, (M, K))
    w_b = normal_bf16(seed + 1, (K, N), 0.02)
    dy_b = lognormal_grad_bf16(seed + 2, (M, N))
    T, C = g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT
    wst, xst, gst = g.TensorState(), g.TensorState(), g.TensorState()
    wq, wqT, xq, xqT = empty_u8(K, N), empty_u8(N, K), empty_u8(M, K), empty_u8(K, M)
    dyq, dyqT = empty_u8(M, N), empty_u8(N, M)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    y, dx, dw = bf(M, N), bf(M, K), bf(K, N)
    g.fp8_requantize_weights(dev_bf16(w_b), K, N, T, C, wst, wq, wqT)
    g.fp8_linear_fwd(dev_bf16(x_b), M, K, N, wqT, wst, None, xst, T, C, xq, xqT, None, y)
    g.fp8_linear_bwd(dev_bf16(dy_b), M, K, N, xqT, xst, wq, wst, gst, C, dyq, dyqT, dx, dw)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    ox, ow, og = quant.quantize_tensor(x_b, fp8.E4M3), quant.quantize_tensor(w_b, fp8.E4M3), quant.quantize_tensor(dy_b, fp8.E5M2)
    assert np.array_equal(host_u8(xq), ox["q"]) and np.array_equal(host_u8(wqT), ow["qT"])
    assert np.array_equal(host_u8(dyq), og["q"])
    return (ox, ow, og), (host_bf16_f64(y), host_bf16_f64(dx), host_bf16_f64(dw))


def check(got, ref, mag):
    ok = gemm.within_bound(got, ref, mag)
    assert ok.all(), f"{(~ok).sum()} outside the bound"


@pytest.mark.parametrize("name", list(SHAPES))
def test_projection_reduced_tokens_in_full(g, name):
    K, N = SHAPES[name]
    M = 400
    (ox, ow, og), (y, dx, dw) = run(g, M, K, N, 3100 + K + N)
    r, m, _ = gemm.scaled_mm(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"])
    check(y, r, m)
    r, m, _ = gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"])
    check(dx, r, m)
    r, m, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    check(dw, r, m)


@pytest.mark.parametrize("name", list(SHAPES))
def test_projection_full_tokens_sampled(g, name):
    K, N = SHAPES[name]
    M = 8192
    (ox, ow, og), (y, dx, dw) = run(g, M, K, N, 3200 + K + N)
    rng = np.random.default_rng(K + N)
    for got, (a, fa, b, fb, da, db), (R, Cc) in (
            (y, (ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"]), (M, N)),
            (dx, (og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"]), (M, K)),
            (dw, (ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"]), (K, N))):
        r, c = rng.integers(0, R, 2048), rng.integers(0, Cc, 2048)
        ref, mag = gemm.scaled_mm_sampled(a, fa, b, fb, da, db, r, c)
        assert np.isfinite(got).all()
        check(got[r, c], ref, mag)
