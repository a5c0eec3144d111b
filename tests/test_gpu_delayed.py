"""The delayed-scaling training loop on the GPU against the oracle's trajectory.

Reduced size (all layers and steps, fewer tokens and a narrower d): every layer-step's
scaling state (history, count, scale, scale_inv, amax, counters) and codes bit-exact;
GEMM outputs within the bound at a few steps. Full size: the loop's shapes for two of
the twelve layers, the weight's state and codes every step, the x and dy states every
step, sampled outputs at the first and last steps. Odd layers (and layer 11 at full size)
run the backward with the wgrad reading x_q and dy_q MN-major, the others with the
transposed copies."""
import numpy as np
import pytest
import torch

from datagen import normal_bf16, lognormal_grad_bf16, perturbation_f32, workload_inputs
from oracle import fp8, gemm, linear, quant

from gpu_util import dev_bf16, empty_u8, host_u8, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def assert_close(got, ref, mag):
    ok = gemm.within_bound(got, ref, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"


class Layer:
    """One layer's step through the library. mn: the backward through fp8_linear_bwd_mn (the
    wgrad reads x_q and dy_q MN-major, split K through a workspace, as bench.py times it);
    otherwise fp8_linear_bwd with the transposed copies."""

    def __init__(self, g, w_bits, M, K, N, hist, mn=False):
        self.g, self.M, self.K, self.N, self.mn = g, M, K, N, mn
        self.w = dev_bf16(w_bits)
        self.wst, self.xst, self.gst = g.TensorState(hist), g.TensorState(hist), g.TensorState(hist)
        self.wq, self.wqT = empty_u8(K, N), empty_u8(N, K)
        self.xq, self.xqT = empty_u8(M, K), empty_u8(K, M)
        self.dyq, self.dyqT = empty_u8(M, N), empty_u8(N, M)
        bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
        self.y, self.dx, self.dw = bf(M, N), bf(M, K), bf(K, N)
        self.wsb = g.fp8_linear_bwd_workspace_bytes(M, K, N)
        self.ws = torch.zeros(max(self.wsb, 16), dtype=torch.uint8, device="cuda")

    def step(self, x, dy, delta):
        g, D, T = self.g, self.g.FP8_SCALE_DELAYED, self.g.FP8_GRAN_TENSOR
        if delta is not None:  # simulated optimizer step (harness, not the library)
            self.w.copy_((self.w.float() + delta).to(torch.bfloat16))
        g.fp8_requantize_weights(self.w, self.K, self.N, T, D, self.wst, self.wq, self.wqT)
        g.fp8_linear_fwd(x, self.M, self.K, self.N, self.wqT, self.wst, None, self.xst, T, D, self.xq,
                         None if self.mn else self.xqT, None, self.y)
        if self.mn:
            g.fp8_linear_bwd_mn(dy, self.M, self.K, self.N, self.xq, self.xst, self.wq, self.wst, self.gst, D,
                                self.dyq, self.dx, self.dw, self.ws, self.wsb)
        else:
            g.fp8_linear_bwd(dy, self.M, self.K, self.N, self.xqT, self.xst, self.wq, self.wst, self.gst, D,
                             self.dyq, self.dyqT, self.dx, self.dw)
        for st in (self.wst, self.xst, self.gst):
            g.fp8_history_commit(st)


def same_state(snap, o):
    assert snap["count"] == o["count"]
    assert np.array_equal(snap["hist"], o["hist"])
    assert np.float32(snap["scale"]) == o["scale"] and np.float32(snap["scale_inv"]) == o["scale_inv"]
    assert np.float32(snap["amax_cur"]) == o["amax_cur"]
    assert snap["overflow"] == o["overflow"] and snap["underflow"] == o["underflow"]


def test_delayed_loop_reduced_trajectory(g):
    L, T, H = 3, 50, 16
    M, K, N = 256, 256, 512
    x_b = normal_bf16(5000, (M, K))
    dy_b = lognormal_grad_bf16(5002, (M, N))
    w_b = [normal_bf16(5100 + l, (K, N), 0.02) for l in range(L)]
    delta = lambda l, t: perturbation_f32(15000 + 100 * t + l, (K, N), 1e-3)
    x, dy = dev_bf16(x_b), dev_bf16(dy_b)
    layers = [Layer(g, w_b[l], M, K, N, H, mn=(l % 2 == 1)) for l in range(L)]  # both backward paths
    recs = {}

    def on_step(t, l, rec):
        recs[(t, l)] = rec

    # run the oracle lazily per step to keep memory small: collect the whole trajectory
    linear.training_loop(x_b, dy_b, w_b, T, H, delta, with_gemm=False, on_step=on_step)
    check_gemm_at = {0, 1, 16, 17, 49}
    for t in range(T):
        for l in range(L):
            d = None if t == 0 else torch.from_numpy(delta(l, t)).cuda()
            layers[l].step(x, dy, d)
            r = recs[(t, l)]
            lay = layers[l]
            same_state(lay.wst.snapshot(), r["state"]["w"])
            same_state(lay.xst.snapshot(), r["state"]["x"])
            same_state(lay.gst.snapshot(), r["state"]["dy"])
            assert np.array_equal(host_u8(lay.wq), r["w"]["q"]), (t, l)
            assert np.array_equal(host_u8(lay.wqT), r["w"]["qT"])
            assert np.array_equal(host_u8(lay.dyq), r["dy"]["q"])
            if t in check_gemm_at:
                wo, xo, go = r["w"], r["x"], r["dy"]
                assert np.array_equal(host_u8(lay.xq), xo["q"])
                if not lay.mn:
                    assert np.array_equal(host_u8(lay.xqT), xo["qT"]) and np.array_equal(host_u8(lay.dyqT), go["qT"])
                yr, ym, _ = gemm.scaled_mm(xo["q"], fp8.E4M3, wo["qT"], fp8.E4M3, xo["d"], wo["d"])
                dxr, dxm, _ = gemm.scaled_mm(go["q"], fp8.E5M2, wo["q"], fp8.E4M3, go["d"], wo["d"])
                dwr, dwm, _ = gemm.scaled_mm(xo["qT"], fp8.E4M3, go["qT"], fp8.E5M2, xo["d"], go["d"])
                assert_close(host_bf16_f64(lay.y), yr, ym)
                assert_close(host_bf16_f64(lay.dx), dxr, dxm)
                assert_close(host_bf16_f64(lay.dw), dwr, dwm)
            # invariant: the bootstrap step never saturates
            if t == 0:
                assert r["state"]["w"]["overflow"] == 0 and r["state"]["x"]["overflow"] == 0
    g.fp8_poll_device_error()


@pytest.mark.slow
def test_delayed_loop_full_size(g):
    """Full shapes (32768 tokens, d 1536 -> 6144, history 16, 50 steps) for layers 0 and 11
    of the 12: the weight's whole state and codes every step against the oracle; the x and
    dy casts in full at step 0, and after it their states follow from it (the same tensors
    every step, so amax_eff equals the step-0 amax and the counters grow by the step-0
    counts). At the first and the last step, 4096 sampled outputs of each GEMM against the
    oracle's exact sampled reference: the forward (contraction 1536), dgrad (E5M2 x E4M3,
    contraction 6144) and wgrad (E4M3 x E5M2, contraction over all 32768 tokens)."""
    wl = workload_inputs("delayed_loop", M=32768)
    M, K, N, T, H = wl["M"], wl["K"], wl["N"], wl["steps"], wl["hist_len"]
    x_b, dy_b = wl["x"], wl["dy"]
    x, dy = dev_bf16(x_b), dev_bf16(dy_b)
    ox0 = quant.quantize_tensor(x_b, fp8.E4M3)
    og0 = quant.quantize_tensor(dy_b, fp8.E5M2)
    rng = np.random.default_rng(9)
    for l in (0, 11):  # layer 11 through the MN-major backward, as the bench runs it
        lay = Layer(g, wl["w"][l], M, K, N, H, mn=(l == 11))
        ws = quant.DelayedState(H)
        w_host = wl["w"][l].copy()
        for t in range(T):
            delta = None
            if t >= 1:
                dnp = perturbation_f32(wl["perturb_seed"](l, t), (K, N), 1e-3)
                delta = torch.from_numpy(dnp).cuda()
                w_host = linear.perturb_master(w_host, dnp)
            lay.step(x, dy, delta)
            wo = ws.quantize(w_host, fp8.E4M3)
            ws.commit()
            same_state(lay.wst.snapshot(), ws.snapshot())
            assert np.array_equal(host_u8(lay.wqT), wo["qT"]), (l, t)
            for st, o0 in ((lay.xst, ox0), (lay.gst, og0)):
                snap = st.snapshot()
                n = t + 1
                assert snap["count"] == n
                assert np.all(snap["hist"][:min(n, H)] == o0["amax"]) and np.all(snap["hist"][min(n, H):] == 0)
                assert np.float32(snap["scale"]) == o0["s"] and np.float32(snap["scale_inv"]) == o0["d"]
                assert snap["overflow"] == n * o0["overflow"] and snap["underflow"] == n * o0["underflow"]
            if t == 0:
                assert np.array_equal(host_u8(lay.xq), ox0["q"])
                assert np.array_equal(host_u8(lay.dyq), og0["q"])
            if t in (0, T - 1):
                # the x and dy codes of every step equal step 0's (same tensors, same scale)
                S = 4096
                r, c = rng.integers(0, M, S), rng.integers(0, N, S)
                ref, mag = gemm.scaled_mm_sampled(ox0["q"], fp8.E4M3, wo["qT"], fp8.E4M3, ox0["d"], wo["d"], r, c)
                assert_close(host_bf16_f64(lay.y)[r, c], ref, mag)
                r, c = rng.integers(0, M, S), rng.integers(0, K, S)
                ref, mag = gemm.scaled_mm_sampled(og0["q"], fp8.E5M2, wo["q"], fp8.E4M3, og0["d"], wo["d"], r, c)
                assert_close(host_bf16_f64(lay.dx)[r, c], ref, mag)
                r, c = rng.integers(0, K, S), rng.integers(0, N, S)
                ref, mag = gemm.scaled_mm_sampled(ox0["qT"], fp8.E4M3, og0["qT"], fp8.E5M2, ox0["d"], og0["d"], r, c)
                assert_close(host_bf16_f64(lay.dw)[r, c], ref, mag)
        del lay
        torch.cuda.empty_cache()
    g.fp8_poll_device_error()
