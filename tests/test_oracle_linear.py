"""Pins of the oracle's forward/backward compositions and the delayed-scaling loop:
layouts checked against an unquantised fp64 product, and the loop's state checked
against amaxes recomputed from the master weights it was given."""
import numpy as np

from datagen import normal_bf16, lognormal_grad_bf16, perturbation_f32
from oracle import fp8, gemm, linear, quant


def test_forward_backward_layouts_track_fp64_product():
    M, K, N = 64, 128, 96
    x = normal_bf16(1, (M, K))
    w = normal_bf16(2, (K, N), 0.02)
    dy = normal_bf16(3, (M, N), 1e-2)
    ws = quant.quantize_tensor(w, fp8.E4M3)
    xs = quant.DelayedState()
    gs = quant.DelayedState()
    xo, y, _ = linear.forward(x, ws["qT"], ws["d"], xs, delayed=False)
    go, dx, _, dw, _ = linear.backward(dy, xo, ws["q"], ws["d"], gs, delayed=False)
    X = quant.widen_bf16(x).astype(np.float64)
    W = quant.widen_bf16(w).astype(np.float64)
    G = quant.widen_bf16(dy).astype(np.float64)
    # FP8 quantisation keeps ~2-3 significant bits; the products must still correlate
    # strongly and have the right shape (a transposed operand would not)
    for got, want in ((y, X @ W), (dx, G @ W.T), (dw, X.T @ G)):
        assert got.shape == want.shape
        c = np.corrcoef(got.reshape(-1), want.reshape(-1))[0, 1]
        assert c > 0.97, c


def test_training_loop_state_against_recomputed_amaxes():
    M, K, N, L, T, H = 32, 128, 128, 2, 7, 3
    x = normal_bf16(10, (M, K))
    dy = lognormal_grad_bf16(11, (M, N))
    ws = [normal_bf16(20 + l, (K, N), 0.02) for l in range(L)]
    seen = {}

    def rec(t, l, r):
        seen[(t, l)] = r

    linear.training_loop(x, dy, ws, T, H, lambda l, t: perturbation_f32(100 * t + l, (K, N), 1e-3),
                         with_gemm=False, on_step=rec)
    for l in range(L):
        amaxes = [float(np.abs(quant.widen_bf16(seen[(t, l)]["w_master"])).max()) for t in range(T)]
        for t in range(T):
            st = seen[(t, l)]["state"]["w"]
            assert st["count"] == t + 1
            window = amaxes[max(0, t + 1 - H):t + 1]
            assert sorted(st["hist"][:min(t + 1, H)].tolist()) == sorted(np.float32(window).tolist())
            # the scale used at step t came from the window before its push
            eff = amaxes[0] if t == 0 else max(amaxes[max(0, t - H):t])
            assert seen[(t, l)]["w"]["s"] == quant.scales_from_amax(np.float32(eff), fp8.E4M3)[0]
        # bootstrap casts never saturate
        assert seen[(0, l)]["w"]["overflow"] == 0 and seen[(0, l)]["x"]["overflow"] == 0
        assert seen[(0, l)]["dy"]["overflow"] == 0
        # x and dy are the same every step: their histories hold one value
        assert set(seen[(T - 1, l)]["state"]["x"]["hist"].tolist()) == {float(quant.amax(x))}
    # the perturbation changed the masters
    assert not np.array_equal(seen[(T - 1, 0)]["w_master"], ws[0])


def test_perturb_master_is_one_fp32_add_rounded():
    w = normal_bf16(30, (4, 8), 0.02)
    d = perturbation_f32(31, (4, 8))
    got = quant.widen_bf16(linear.perturb_master(w, d)).astype(np.float64)
    exact = quant.widen_bf16(w).astype(np.float64) + d.astype(np.float64)
    # within half a bf16 ulp of the exact sum (plus the fp32 step)
    assert np.all(np.abs(got - exact) <= 0.5 * gemm.bf16_ulp(got) * (1 + 2 ** -15))
