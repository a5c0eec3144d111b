"""GPU parity of the forward / backward compositions and of the weight cache refresh,
at small ragged sizes in full and at the workloads' full sizes on sampled outputs.
Codes, amaxes, scales and counters are compared bit for bit; GEMM outputs within
1e-3 * sum|a b| d_a d_b + 1 bf16 ulp."""
import numpy as np
import pytest
import torch

from datagen import workload_inputs, normal_bf16, lognormal_grad_bf16, channel_scaled_bf16
from oracle import fp8, gemm, quant

from gpu_util import dev_bf16, empty_u8, host_u8, host_bf16_f64

pytestmark = pytest.mark.gpu
SAMPLES = 4096


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def assert_close(got, ref, mag):
    ok = gemm.within_bound(got, ref, mag)
    if not ok.all():
        i = np.argwhere(~ok)[:8]
        pytest.fail(f"{(~ok).sum()} of {ok.size} outside the bound; e.g. {[(tuple(j), got[tuple(j)], ref[tuple(j)]) for j in i]}")


def assert_state(st, o, overflow, underflow):
    s = st.snapshot()
    assert np.float32(s["amax_cur"]) == o["amax"]
    assert np.float32(s["scale"]) == o["s"] and np.float32(s["scale_inv"]) == o["d"]
    assert s["overflow"] == overflow and s["underflow"] == underflow


class Step:
    """Device buffers and one forward + backward through the C ABI (per-tensor, current)."""

    def __init__(self, g, x, w, dy, M, K, N, mode=0):
        self.g, self.M, self.K, self.N, self.mode = g, M, K, N, mode
        self.x, self.w = dev_bf16(x), dev_bf16(w)
        self.dy = dev_bf16(dy) if dy is not None else None
        self.wst, self.xst, self.gst = g.TensorState(), g.TensorState(), g.TensorState()
        self.wq, self.wqT = empty_u8(K, N), empty_u8(N, K)
        self.xq, self.xqT = empty_u8(M, K), empty_u8(K, M)
        self.y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        if dy is not None:
            self.dyq, self.dyqT = empty_u8(M, N), empty_u8(N, M)
            self.dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
            self.dw = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")

    def forward(self):
        g = self.g
        g.fp8_requantize_weights(self.w, self.K, self.N, g.FP8_GRAN_TENSOR, self.mode, self.wst, self.wq, self.wqT)
        g.fp8_linear_fwd(self.x, self.M, self.K, self.N, self.wqT, self.wst, None, self.xst, g.FP8_GRAN_TENSOR,
                         self.mode, self.xq, self.xqT, None, self.y)

    def backward(self):
        g = self.g
        g.fp8_linear_bwd(self.dy, self.M, self.K, self.N, self.xqT, self.xst, self.wq, self.wst, self.gst, self.mode,
                         self.dyq, self.dyqT, self.dx, self.dw)


@pytest.mark.parametrize("M,K,N", [(256, 128, 512), (512, 256, 768), (400, 320, 272)])
def test_forward_backward_small(g, M, K, N):
    x = normal_bf16(M + 1, (M, K))
    w = normal_bf16(K + 2, (K, N), 0.02)
    dy = lognormal_grad_bf16(N + 3, (M, N))
    s = Step(g, x, w, dy, M, K, N)
    s.forward()
    s.backward()
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    ow, ox, og = quant.quantize_tensor(w, fp8.E4M3), quant.quantize_tensor(x, fp8.E4M3), quant.quantize_tensor(dy, fp8.E5M2)
    assert np.array_equal(host_u8(s.wq), ow["q"]) and np.array_equal(host_u8(s.wqT), ow["qT"])
    assert np.array_equal(host_u8(s.xq), ox["q"]) and np.array_equal(host_u8(s.xqT), ox["qT"])
    assert np.array_equal(host_u8(s.dyq), og["q"]) and np.array_equal(host_u8(s.dyqT), og["qT"])
    assert_state(s.wst, ow, ow["overflow"], ow["underflow"])
    assert_state(s.xst, ox, ox["overflow"], ox["underflow"])
    assert_state(s.gst, og, og["overflow"], og["underflow"])
    y, my, _ = gemm.scaled_mm(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"])
    dx, mdx, _ = gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"])
    dw, mdw, _ = gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    assert_close(host_bf16_f64(s.y), y, my)
    assert_close(host_bf16_f64(s.dx), dx, mdx)
    assert_close(host_bf16_f64(s.dw), dw, mdw)


@pytest.mark.parametrize("mode", [0, 1])
def test_empty_token_batch(g, mode):
    """M = 0 (a batch, or an expert, with no tokens): the layer calls accept empty buffers as
    null pointers, the forward writes nothing, the weight gradient of no tokens is zero and
    the x and dy states get unit scales and a zero amax."""
    K, N = 256, 512
    w = normal_bf16(9, (K, N), 0.02)
    wd = dev_bf16(w)
    wst, xst, gst = g.TensorState(), g.TensorState(), g.TensorState()
    wq, wqT = empty_u8(K, N), empty_u8(N, K)
    g.fp8_requantize_weights(wd, K, N, g.FP8_GRAN_TENSOR, mode, wst, wq, wqT)
    xst.scale.fill_(5.0)
    gst.scale.fill_(5.0)
    g.fp8_linear_fwd(None, 0, K, N, wqT, wst, None, xst, g.FP8_GRAN_TENSOR, mode, None, None, None, None)
    dx = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((K, N), 7.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_linear_bwd(None, 0, K, N, None, xst, wq, wst, gst, mode, None, None, dx, dw)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    assert (dw.float() == 0).all()
    for st in (xst, gst):
        snap = st.snapshot()
        assert snap["scale"] == 1.0 and snap["scale_inv"] == 1.0 and snap["amax_cur"] == 0.0
        assert snap["overflow"] == 0 and snap["underflow"] == 0


def test_tiny_forward_workload_in_full(g):
    w = workload_inputs("tiny_fwd")
    M, K, N = w["M"], w["K"], w["N"]
    s = Step(g, w["x"], w["w"], None, M, K, N)
    s.forward()
    torch.cuda.synchronize()
    ow, ox = quant.quantize_tensor(w["w"], fp8.E4M3), quant.quantize_tensor(w["x"], fp8.E4M3)
    assert np.array_equal(host_u8(s.xq), ox["q"]) and np.array_equal(host_u8(s.wqT), ow["qT"])
    y, my, _ = gemm.scaled_mm(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"])
    assert_close(host_bf16_f64(s.y), y, my)


def test_gpt2_small_forward_full_size(g):
    """x [8192 x 768] with 0.1 % outliers x100, W [768 x 3072]: all codes and state bit-exact,
    4096 sampled outputs within the bound, no non-finite output."""
    w = workload_inputs("gpt2s_upproj_fwd")
    M, K, N = w["M"], w["K"], w["N"]
    s = Step(g, w["x"], w["w"], None, M, K, N)
    s.forward()
    torch.cuda.synchronize()
    ow, ox = quant.quantize_tensor(w["w"], fp8.E4M3), quant.quantize_tensor(w["x"], fp8.E4M3)
    assert np.array_equal(host_u8(s.xq), ox["q"]) and np.array_equal(host_u8(s.xqT), ox["qT"])
    assert np.array_equal(host_u8(s.wqT), ow["qT"]) and np.array_equal(host_u8(s.wq), ow["q"])
    assert_state(s.xst, ox, ox["overflow"], ox["underflow"])
    assert ox["underflow"] > 0  # the outliers push the small values below the E4M3 range
    y = host_bf16_f64(s.y)
    assert np.isfinite(y).all()
    rng = np.random.default_rng(0)
    r, c = rng.integers(0, M, SAMPLES), rng.integers(0, N, SAMPLES)
    ref, mag = gemm.scaled_mm_sampled(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"], r, c)
    assert_close(y[r, c], ref, mag)


@pytest.mark.slow
def test_backward_full_size(g):
    """M=16384, K=1024, N=4096; log-normal dy in E5M2: every code and the state bit-exact;
    4096 sampled dgrad and wgrad outputs within the bound."""
    w = workload_inputs("upproj_bwd")
    M, K, N = w["M"], w["K"], w["N"]
    s = Step(g, w["x"], w["w"], w["dy"], M, K, N)
    s.forward()
    s.backward()
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    ow, ox, og = (quant.quantize_tensor(w["w"], fp8.E4M3), quant.quantize_tensor(w["x"], fp8.E4M3),
                  quant.quantize_tensor(w["dy"], fp8.E5M2))
    assert np.array_equal(host_u8(s.dyq), og["q"])
    assert np.array_equal(host_u8(s.dyqT), og["qT"])
    assert np.array_equal(host_u8(s.xqT), ox["qT"])
    assert_state(s.gst, og, og["overflow"], og["underflow"])
    assert og["underflow"] > 0
    rng = np.random.default_rng(1)
    dx, dw = host_bf16_f64(s.dx), host_bf16_f64(s.dw)
    assert np.isfinite(dx).all() and np.isfinite(dw).all()
    r, c = rng.integers(0, M, SAMPLES), rng.integers(0, K, SAMPLES)
    ref, mag = gemm.scaled_mm_sampled(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"], r, c)
    assert_close(dx[r, c], ref, mag)
    r, c = rng.integers(0, K, SAMPLES), rng.integers(0, N, SAMPLES)
    ref, mag = gemm.scaled_mm_sampled(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"], r, c)
    assert_close(dw[r, c], ref, mag)


def _block_forward(g, x, wm, M, K, N):
    xd, wd = dev_bf16(x), dev_bf16(wm)
    wq, wqT = empty_u8(K, N), empty_u8(N, K)
    wsi = torch.empty(K // 128, N // 128, dtype=torch.float32, device="cuda")
    xq = empty_u8(M, K)
    xsi = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    xst = g.TensorState()
    g.fp8_requantize_weights(wd, K, N, g.FP8_GRAN_BLOCK_128x128, 0, None, wq, wqT, wsi)
    g.fp8_linear_fwd(xd, M, K, N, wqT, None, wsi, xst, g.FP8_GRAN_BLOCK_128x128, 0, xq, None, xsi, y)
    torch.cuda.synchronize()
    return wq, wqT, wsi, xq, xsi, y


@pytest.mark.parametrize("M,K,N", [(300, 512, 640), (1024, 1024, 2048)])
def test_block_scaled_forward_small(g, M, K, N):
    x = channel_scaled_bf16(M + K, (M, K))
    wm = normal_bf16(N, (K, N), 0.02)
    wq, wqT, wsi, xq, xsi, y = _block_forward(g, x, wm, M, K, N)
    ow = quant.quantize_block_128x128(wm, fp8.E4M3)
    ox = quant.quantize_tile_1x128(x, fp8.E4M3)
    assert np.array_equal(host_u8(wqT), ow["qT"]) and np.array_equal(wsi.cpu().numpy(), ow["d"])
    assert np.array_equal(host_u8(xq), ox["q"]) and np.array_equal(xsi.cpu().numpy(), ox["d"])
    ref, mag = gemm.block_scaled_mm(ox["q"], fp8.E4M3, ox["d"], ow["qT"], fp8.E4M3, ow["d"])
    assert_close(host_bf16_f64(y), ref, mag)


@pytest.mark.slow
def test_finegrained_forward_full_size(g):
    """x [16384 x 4096] with per-channel std 10^U(-1,1) in 1x128 tiles, W [4096 x 14336] in
    128x128 blocks: sampled rows' codes and tile scales, sampled column blocks' codes and
    block scales bit-exact; a grid of sampled outputs within the bound."""
    w = workload_inputs("finegrained_fwd")
    M, K, N = w["M"], w["K"], w["N"]
    wq, wqT, wsi, xq, xsi, y = _block_forward(g, w["x"], w["w"], M, K, N)
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(M, 48, replace=False))
    nbs = np.sort(rng.choice(N // 128, 3, replace=False))
    ox = quant.quantize_tile_1x128(w["x"][rows], fp8.E4M3)
    assert np.array_equal(host_u8(xq)[rows], ox["q"])
    assert np.array_equal(xsi.cpu().numpy()[rows], ox["d"])
    cols, wT_rows, d_w = [], [], np.empty((K // 128, N // 128), dtype=np.float32)
    wqT_h, wsi_h = host_u8(wqT), wsi.cpu().numpy()
    for nb in nbs:
        ob = quant.quantize_block_128x128(w["w"][:, nb * 128:(nb + 1) * 128], fp8.E4M3)
        assert np.array_equal(wqT_h[nb * 128:(nb + 1) * 128], ob["qT"])
        assert np.array_equal(wsi_h[:, nb], ob["d"][:, 0])
        d_w[:, nb] = ob["d"][:, 0]
        pick = np.sort(rng.choice(128, 16, replace=False))
        cols.extend(nb * 128 + pick)
        wT_rows.append(ob["qT"][pick])
    cols = np.array(cols)
    bT = np.zeros((N, K), dtype=np.uint8)
    bT[cols] = np.concatenate(wT_rows)
    aq = np.zeros((M, K), dtype=np.uint8)
    aq[rows] = ox["q"]
    da = np.zeros((M, K // 128), dtype=np.float32)
    da[rows] = ox["d"]
    rr, cc = np.meshgrid(rows, cols, indexing="ij")
    rr, cc = rr.reshape(-1), cc.reshape(-1)
    ref, mag = gemm.block_scaled_mm_sampled(aq, fp8.E4M3, da, bT, fp8.E4M3, d_w, rr, cc)
    got = host_bf16_f64(y)
    assert np.isfinite(got).all()
    assert_close(got[rr, cc], ref, mag)
