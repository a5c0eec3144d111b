"""GPU parity of the backward pass through fp8_linear_bwd_ws: dgrad and wgrad in one grouped
launch, the weight gradient split over its token contraction through the workspace. Codes and
the dy state bit for bit; GEMM outputs within 1e-3 * sum|a b| d_a d_b + 1 bf16 ulp, in full at
a small size and on sampled outputs at the GPT-2-small size."""
import numpy as np
import pytest
import torch

from datagen import normal_bf16, lognormal_grad_bf16
from oracle import fp8, gemm, quant

from gpu_util import host_u8, host_bf16_f64
from test_gpu_linear import Step, assert_close, assert_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def backward_ws(g, s, ws, nbytes):
    g.fp8_linear_bwd_ws(s.dy, s.M, s.K, s.N, s.xqT, s.xst, s.wq, s.wst, s.gst, s.mode, s.dyq, s.dyqT, s.dx, s.dw,
                        ws, nbytes)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    return host_bf16_f64(s.dx), host_bf16_f64(s.dw)


@pytest.mark.parametrize("M,K,N", [(4096, 256, 512), (4096, 384, 640)])
def test_grouped_split_backward_against_exact(g, M, K, N):
    nbytes = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    assert nbytes > 0, "the weight gradient of this shape should split"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    x = normal_bf16(M + 5, (M, K))
    w = normal_bf16(K + 6, (K, N), 0.02)
    dy = lognormal_grad_bf16(N + 7, (M, N))
    s = Step(g, x, w, dy, M, K, N)
    s.forward()
    dx, dw = backward_ws(g, s, ws, nbytes)
    ow, ox, og = quant.quantize_tensor(w, fp8.E4M3), quant.quantize_tensor(x, fp8.E4M3), quant.quantize_tensor(dy, fp8.E5M2)
    assert np.array_equal(host_u8(s.dyq), og["q"]) and np.array_equal(host_u8(s.dyqT), og["qT"])
    assert_state(s.gst, og, og["overflow"], og["underflow"])
    rdx, mdx, _ = gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"])
    rdw, mdw, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    assert_close(dx, rdx, mdx)
    assert_close(dw, rdw, mdw)
    # the same call again (workspace reused without clearing): the same bits
    dx2, dw2 = backward_ws(g, s, ws, nbytes)
    assert np.array_equal(dx.view(np.uint64), dx2.view(np.uint64))
    assert np.array_equal(dw.view(np.uint64), dw2.view(np.uint64))
    # without a workspace: one grouped launch, no split, within the same bound
    s.dx.zero_()
    s.dw.zero_()
    s.backward()
    torch.cuda.synchronize()
    assert_close(host_bf16_f64(s.dx), rdx, mdx)
    assert_close(host_bf16_f64(s.dw), rdw, mdw)


def test_gpt2_small_backward_grouped(g):
    """M=8192 tokens, d=768, 4d=3072: dgrad [8192 x 768] and the split wgrad [768 x 3072] in
    one launch; 4096 sampled outputs of each against the oracle."""
    M, K, N = 8192, 768, 3072
    nbytes = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    x = normal_bf16(31, (M, K))
    w = normal_bf16(32, (K, N), 0.02)
    dy = lognormal_grad_bf16(33, (M, N))
    s = Step(g, x, w, dy, M, K, N)
    s.forward()
    dx, dw = backward_ws(g, s, ws, nbytes)
    ow, ox, og = quant.quantize_tensor(w, fp8.E4M3), quant.quantize_tensor(x, fp8.E4M3), quant.quantize_tensor(dy, fp8.E5M2)
    assert np.array_equal(host_u8(s.dyqT), og["qT"])
    rng = np.random.default_rng(2)
    r, c = rng.integers(0, M, 4096), rng.integers(0, K, 4096)
    ref, mag = gemm.scaled_mm_sampled(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"], r, c)
    assert_close(dx[r, c], ref, mag)
    r, c = rng.integers(0, K, 4096), rng.integers(0, N, 4096)
    ref, mag = gemm.scaled_mm_sampled(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"], r, c)
    assert_close(dw[r, c], ref, mag)


def test_linear_bwd_ws_rejections(g):
    s = Step(g, normal_bf16(1, (256, 128)), normal_bf16(2, (128, 256), 0.02), lognormal_grad_bf16(3, (256, 256)),
             256, 128, 256)
    s.forward()
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_linear_bwd_ws(s.dy, 256, 128, 256, s.xqT, s.xst, s.wq, s.wst, s.gst, 0, s.dyq, s.dyqT, s.dx, s.dw,
                            ws[8:].data_ptr(), 1000)
    assert e.value.status == g.FP8_ERR_ALIGNMENT
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_linear_bwd_ws(s.dy, 256, 128, 256, s.xqT, s.xst, s.wq, s.wst, s.gst, 0, s.dyq, s.dyqT, s.dx, s.dw,
                            ws, -1)
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    g.fp8_poll_device_error()
