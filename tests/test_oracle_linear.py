"""Pins of the oracle's forward/backward compositions and the delayed-scaling loop:
layouts checked against an unquantised fp64 product, each GEMM's scale pairing checked
exactly with power-of-two scales and integer codes, the optimizer step's bf16 rounding
against torch on constructed ties, and the loop's state checked against amaxes recomputed
from the master weights it was given."""
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


def _tie_cases():
    """fp32 values that sit exactly halfway between two bf16 neighbours (low 16 bits 0x8000),
    with an even and an odd lower neighbour, both signs, normal and subnormal, plus values a
    hair above and below a tie, and the largest finite fp32 (rounds to infinity)."""
    rng = np.random.default_rng(40)
    hi = rng.integers(0x0001, 0x7F7F, 4000).astype(np.uint32)
    hi = np.concatenate([hi, hi | 1, hi & ~np.uint32(1), np.array([0x0000, 0x0001, 0x007F, 0x3F80, 0x3F81, 0x7F7E, 0x7F7F],
                                                                   dtype=np.uint32)])
    sign = rng.integers(0, 2, hi.size).astype(np.uint32) << 31
    ties = (sign | (hi << 16) | 0x8000).astype(np.uint32)
    near = np.concatenate([ties + 1, ties - 1])
    extra = np.array([0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F7FFF], dtype=np.uint32)
    return np.concatenate([ties, near, extra]).view(np.float32)


def test_bf16_rounding_of_the_optimizer_step_against_torch_on_ties():
    """perturb_master's rounding (and datagen's, which stores every synthetic input) against
    torch's fp32 -> bf16 conversion, round to nearest with ties to even, on constructed ties."""
    import torch
    from datagen import bf16_bits_from_f32
    v = _tie_cases()
    want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(linear._bf16_bits_rne(v), want)
    assert np.array_equal(bf16_bits_from_f32(v), want)
    # the same through the optimizer step: W + delta landing exactly on a tie
    w = np.array([0x3F80, 0x3F81, 0xBF80, 0xBF81], dtype=np.uint16)      # 1, 1+2^-7, -1, -(1+2^-7)
    delta = np.array([2 ** -8, 2 ** -8, -(2 ** -8), -(2 ** -8)], dtype=np.float32)
    got = linear.perturb_master(w, delta)
    # 1 + 2^-8 ties to 1 (even); 1 + 3*2^-8 ties to 1 + 2^-6 (even); likewise negated
    assert got.tolist() == [0x3F80, 0x3F82, 0xBF80, 0xBF82]
    s = (quant.widen_bf16(w) + delta).astype(np.float32)
    assert np.array_equal(got, torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def _codes_from_values(vals, fmt):
    c = fp8.cast(np.asarray(vals, dtype=np.float64), fmt)
    assert np.array_equal(fp8.decode_array(c, fmt), np.asarray(vals, dtype=np.float64))
    return c


def test_forward_backward_scale_pairing_exact():
    """Each GEMM of the layer multiplies by its own two operands' scales: with distinct powers
    of two as d_x, d_w and d_dy and small-integer codes, y = bf16(d_x d_w S_y),
    dx = bf16(d_dy d_w S_dx) and dW = bf16(d_x d_dy S_dW), each S an integer sum worked out
    here from the code values; a swapped pairing moves a result by a power of two."""
    rng = np.random.default_rng(41)
    M, K, N = 16, 32, 48
    ints = np.array([-3, -2, -1, 0, 1, 2, 3])
    # tensors whose amax is FP8_MAX * 2^e: every element is an integer times 2^e, so the cast
    # reproduces the integers exactly and d = 2^e
    def tensor(shape, fmt, e):
        v = rng.choice(ints, size=shape).astype(np.float64)
        v.flat[0] = fp8.fp8_max(fmt)                      # the amax element (code max)
        bits = np.asarray(np.ldexp(v, e), dtype=np.float32).view(np.uint32)
        assert np.all((bits & 0xFFFF) == 0)
        return (bits >> 16).astype(np.uint16), v
    x_b, xv = tensor((M, K), fp8.E4M3, -3)
    w_b, wv = tensor((K, N), fp8.E4M3, 5)
    dy_b, gv = tensor((M, N), fp8.E5M2, -10)
    ws = quant.quantize_tensor(w_b, fp8.E4M3)
    assert ws["d"] == np.float32(2.0 ** 5)
    xs, gs = quant.DelayedState(), quant.DelayedState()
    xo, y, _ = linear.forward(x_b, ws["qT"], ws["d"], xs, delayed=False)
    go, dx, _, dw, _ = linear.backward(dy_b, xo, ws["q"], ws["d"], gs, delayed=False)
    assert xo["d"] == np.float32(2.0 ** -3) and go["d"] == np.float32(2.0 ** -10)
    assert np.array_equal(xo["q"], _codes_from_values(xv, fp8.E4M3))
    assert np.array_equal(go["q"], _codes_from_values(gv, fp8.E5M2))
    S_y = (xv @ wv).astype(np.float64)
    S_dx = (gv @ wv.T).astype(np.float64)
    S_dw = (xv.T @ gv).astype(np.float64)
    assert np.array_equal(y, gemm.bf16_round(np.ldexp(S_y, -3 + 5)))
    assert np.array_equal(dx, gemm.bf16_round(np.ldexp(S_dx, -10 + 5)))
    assert np.array_equal(dw, gemm.bf16_round(np.ldexp(S_dw, -3 - 10)))
