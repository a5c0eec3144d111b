"""Pins of the oracle's amax, scales, counters, fine-grained units and delayed state
against hand-derived values, closed forms and invariants."""
import numpy as np
import pytest

from datagen import bf16_bits_from_f32, normal_bf16
from oracle import fp8, quant


def bits(vals):
    return bf16_bits_from_f32(np.asarray(vals, dtype=np.float32))


def test_amax_hand_values():
    assert quant.amax(bits([1.0, -3.0, 2.0])) == 3.0
    assert quant.amax(bits([np.nan, -0.5, 0.25])) == 0.5           # NaN ignored
    assert quant.amax(bits([-0.0, 0.0])) == 0.0
    assert quant.amax(bits([np.nan])) == 0.0
    assert quant.amax(np.zeros(0, dtype=np.uint16)) == 0.0
    assert quant.amax(bits([1.0, -np.inf])) == np.inf


def test_scale_closed_forms():
    s, d = quant.scales_from_amax(np.float32(448.0), fp8.E4M3)
    assert s == 1.0 and d == 1.0
    s, d = quant.scales_from_amax(np.float32(57344.0), fp8.E5M2)
    assert s == 1.0 and d == 1.0
    s, d = quant.scales_from_amax(np.float32(7.0), fp8.E4M3)
    assert s == 64.0 and d == np.float32(1 / 64)
    s, d = quant.scales_from_amax(np.float32(0.5), fp8.E4M3)
    assert s == 896.0 and d == np.float32(0.5 / 448.0)
    for bad in (0.0, np.inf, np.nan):
        assert quant.scales_from_amax(np.float32(bad), fp8.E4M3) == (1.0, 1.0)
    # a subnormal amax whose quotient overflows float32 behaves like a zero amax
    tiny = np.float32(2.0 ** -133)  # the smallest bf16 subnormal
    assert quant.scales_from_amax(tiny, fp8.E4M3) == (1.0, 1.0)
    assert quant.scales_from_amax(tiny, fp8.E5M2) == (1.0, 1.0)
    # the largest amax with a finite quotient keeps the rule
    a = np.float32(2.0 ** -119)
    s, d = quant.scales_from_amax(a, fp8.E4M3)
    assert np.isfinite(s) and s == np.float32(np.float32(448.0) / a)


@pytest.mark.parametrize("fmt,maxcode", [(fp8.E4M3, 0x7E), (fp8.E5M2, 0x7B)])
def test_amax_element_hits_the_maximum_code(fmt, maxcode):
    for seed in range(20):
        x = normal_bf16(seed, (37, 53), std=10.0 ** (seed % 7 - 3))
        r = quant.quantize_tensor(x, fmt)
        xv = quant.widen_bf16(x)
        i = np.argmax(np.abs(xv))
        assert (r["q"].reshape(-1)[i] & 0x7F) == maxcode
        assert r["overflow"] == 0
        # every code is finite and within range
        dec = fp8.decode_array(r["q"], fmt)
        assert np.all(np.isfinite(dec)) and np.all(np.abs(dec) <= fp8.fp8_max(fmt))


def test_counters_hand_values():
    x = bits([500.0, -1000.0, np.inf, -np.inf, np.nan, 1e-30, -1e-30, 0.0, -0.0, 1.0, 2.0 ** -11])
    q, ov, un = quant.cast_with_scale(x, np.float32(1.0), fp8.E4M3)
    # 500, -1000, +inf, -inf exceed 448; 1e-30, -1e-30, 2^-11 round to zero
    assert ov == 4 and un == 3
    assert q.tolist() == [0x7E, 0xFE, 0x7E, 0xFE, 0x7F, 0x00, 0x80, 0x00, 0x80, 0x38, 0x00]
    q, ov, un = quant.cast_with_scale(x, np.float32(1.0), fp8.E5M2)
    # only the infinities exceed 57344; 2^-11 is a normal E5M2 value (least normal 2^-14),
    # so only the two 1e-30s flush to zero
    assert ov == 2 and un == 2
    dec = fp8.decode_array(q, fp8.E5M2)
    assert dec[10] == 2.0 ** -11


def test_counters_multiply_overflow():
    # a finite input whose scaled value overflows fp32 is counted and saturates
    x = bits([3e38, -3e38, 1.0])
    q, ov, un = quant.cast_with_scale(x, np.float32(10.0), fp8.E4M3)
    assert ov == 2 and un == 0 and q.tolist() == [0x7E, 0xFE, 0x52]   # 10 = 1.25 * 2^3 -> 0x52


def test_tile_reduces_to_tensor_on_one_tile():
    x = normal_bf16(3, (1, 128))
    t = quant.quantize_tile_1x128(x, fp8.E4M3)
    r = quant.quantize_tensor(x, fp8.E4M3)
    assert np.array_equal(t["q"], r["q"]) and t["d"][0, 0] == r["d"]


def test_tiles_are_independent_power_of_two_copies():
    base = quant.widen_bf16(normal_bf16(4, (3, 128)))
    tiles = [base * np.float32(2.0 ** p) for p in (-4, 0, 5, 9)]
    x = bf16_bits_from_f32(np.concatenate(tiles, axis=1))
    t = quant.quantize_tile_1x128(x, fp8.E5M2)
    for j in range(1, 4):
        assert np.array_equal(t["q"][:, j * 128:(j + 1) * 128], t["q"][:, :128])
    p = np.array([-4, 0, 5, 9], dtype=np.float64)
    assert np.allclose(t["d"] / t["d"][:, :1], 2.0 ** (p - p[0])[None, :], rtol=0, atol=0)


def test_block_reduces_to_tensor_and_is_independent():
    w = normal_bf16(5, (128, 128), 0.02)
    b = quant.quantize_block_128x128(w, fp8.E4M3)
    r = quant.quantize_tensor(w, fp8.E4M3)
    assert np.array_equal(b["q"], r["q"]) and b["d"][0, 0] == r["d"]
    # a 256 x 384 tensor made of scaled copies of one block
    base = quant.widen_bf16(w)
    rows = [np.concatenate([base * np.float32(2.0 ** (a + 2 * c)) for c in range(3)], axis=1) for a in range(2)]
    W = bf16_bits_from_f32(np.concatenate(rows, axis=0))
    bb = quant.quantize_block_128x128(W, fp8.E4M3)
    for a in range(2):
        for c in range(3):
            assert np.array_equal(bb["q"][a * 128:(a + 1) * 128, c * 128:(c + 1) * 128], b["q"])
            assert bb["d"][a, c] == np.float32(b["d"][0, 0] * 2.0 ** (a + 2 * c))
    assert np.array_equal(bb["qT"], bb["q"].T)


def test_delayed_state_hand_trajectory():
    st = quant.DelayedState(hist_len=3)
    amaxes = [2.0, 1.0, 4.0, 0.5, 0.25, 8.0]
    effs = []
    for a in amaxes:
        x = bits([a, -a / 2, 0.0])
        r = st.quantize(x, fp8.E4M3, delayed=True)
        effs.append(np.float32(448.0) / r["s"])
        assert st.amax_cur == a
        st.commit()
    # bootstrap uses the current amax (2); then the max over the last <= 3 pushes
    assert [float(e) for e in effs] == [2.0, 2.0, 2.0, 4.0, 4.0, 4.0]
    assert st.count == 6 and st.hist.tolist() == [0.5, 0.25, 8.0]


def test_delayed_running_max_and_commit_reset():
    """amax_cur: the running maximum of the delayed casts since the last commit (the bootstrap
    scale included), reset by the commit; a current-scaling cast sets it to its own amax."""
    st = quant.DelayedState(hist_len=2)
    r1 = st.quantize(bits([3.0, -1.0]), fp8.E4M3, delayed=True)  # bootstrap: amax 3
    assert st.amax_cur == 3.0 and r1["s"] == np.float32(448.0 / 3.0)
    r2 = st.quantize(bits([1.5]), fp8.E4M3, delayed=True)  # still bootstrap: the running max 3
    assert st.amax_cur == 3.0 and r2["s"] == r1["s"] and r2["amax"] == 1.5
    r3 = st.quantize(bits([-6.0]), fp8.E4M3, delayed=True)
    assert st.amax_cur == 6.0 and r3["s"] == np.float32(448.0 / 6.0)
    st.commit()
    assert st.amax_cur == 0.0 and st.hist.tolist() == [6.0, 0.0] and st.count == 1
    r4 = st.quantize(bits([0.5]), fp8.E4M3, delayed=True)  # past bootstrap: the history's 6
    assert st.amax_cur == 0.5 and r4["s"] == np.float32(448.0 / 6.0)
    st.quantize(bits([0.25]), fp8.E4M3, delayed=False)  # current scaling: its own amax
    assert st.amax_cur == 0.25
    st.commit()
    assert st.hist.tolist() == [6.0, 0.25] and st.amax_cur == 0.0


def test_delayed_saturation_is_counted():
    st = quant.DelayedState(hist_len=4)
    st.quantize(bits([1.0, 0.5]), fp8.E4M3)
    st.commit()
    assert st.overflow == 0
    # the tensor doubled: elements above the old amax saturate and are counted
    r = st.quantize(bits([2.0, 1.5, 1.0, -1.25]), fp8.E4M3)
    assert r["overflow"] == 3
    assert r["q"].tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert st.overflow == 3


def test_current_mode_ignores_history():
    st = quant.DelayedState(hist_len=4)
    st.quantize(bits([100.0]), fp8.E4M3)
    st.commit()
    r = st.quantize(bits([1.0]), fp8.E4M3, delayed=False)
    assert r["s"] == 448.0


# ---------------------------------------------------------------------------------------
# MX units: power-of-two scales per 32 elements along the contraction dimension
# ---------------------------------------------------------------------------------------
def _mx_exponent_by_search(a, fmt):
    """The definition read directly: the smallest integer e in [-127, 127] with
    FP8_MAX * 2^e >= a (searched upward; the clamps at both ends), 0 for zero or non-finite."""
    if not (np.isfinite(a) and a > 0):
        return 0
    mx = fp8.fp8_max(fmt)
    for e in range(-127, 128):
        if mx * 2.0 ** e >= a:
            return e
    return 127


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_mx_exponent_against_search(fmt):
    rng = np.random.default_rng(60)
    v = np.abs(rng.standard_normal(3000) * 10.0 ** rng.uniform(-45, 38, 3000)).astype(np.float32)
    mx = np.float32(fp8.fp8_max(fmt))
    edges = [mx * np.float32(2.0) ** k for k in range(-60, 60, 7)]
    edges += [np.nextafter(x, np.float32(np.inf)) for x in edges] + [np.nextafter(x, np.float32(0)) for x in edges]
    for a in list(v) + edges + [np.float32(1e-45), np.float32(3.3e38)]:
        a = np.float32(a)
        assert quant.mx_exponent(a, fmt) == _mx_exponent_by_search(float(a), fmt), a


def test_mx_exponent_hand_values():
    E4, E5 = fp8.E4M3, fp8.E5M2
    assert quant.mx_exponent(448.0, E4) == 0 and quant.mx_exponent(449.0, E4) == 1
    assert quant.mx_exponent(448.0 * 8, E4) == 3 and quant.mx_exponent(448.0 * 8 + 1, E4) == 4
    assert quant.mx_exponent(1.0, E4) == -8          # 448 * 2^-8 = 1.75 >= 1 > 0.875
    assert quant.mx_exponent(57344.0, E5) == 0 and quant.mx_exponent(57345.0, E5) == 1
    assert quant.mx_exponent(0.0, E4) == 0 and quant.mx_exponent(np.inf, E4) == 0 and quant.mx_exponent(np.nan, E5) == 0
    assert quant.mx_exponent(1e-40, E4) == -127      # clamped to the byte's range


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_mx_groups_use_the_top_binade_and_never_saturate(fmt):
    rng = np.random.default_rng(61)
    x = bits(rng.standard_normal((6, 256)) * 10.0 ** rng.uniform(-6, 6, (6, 8)).repeat(32, axis=1))
    o = quant.quantize_mx(x, fmt)
    assert o["overflow"] == 0
    mx = fp8.fp8_max(fmt)
    vals = np.abs(fp8.decode_array(o["q"], fmt)).reshape(6, 8, 32)
    top = vals.max(axis=2)
    assert np.all(top <= mx) and np.all(top >= mx / 2)   # the group's amax lands in (max/2, max]
    assert np.array_equal(o["ue8m0"].astype(np.int64), o["e"] + 127)
    # groups are independent: scaling one group by 2^5 moves only its exponent, by 5
    x2 = x.copy()
    x2[:, 64:96] = bits(quant.widen_bf16(x[:, 64:96]) * np.float32(32.0))
    o2 = quant.quantize_mx(x2, fmt)
    assert np.array_equal(o2["q"], o["q"])
    want = o["e"].copy()
    want[:, 2] += 5
    assert np.array_equal(o2["e"], want)


def test_mx_reproduces_representable_groups_exactly():
    """A group whose elements are E4M3 values times 2^e (the largest one 448 * 2^e) casts to
    exactly those codes with exponent e."""
    rng = np.random.default_rng(62)
    codes = rng.integers(0, 0x7F, size=(3, 64)).astype(np.uint8) | (rng.integers(0, 2, size=(3, 64)) << 7).astype(np.uint8)
    codes[:, 0] = 0x7E
    codes[:, 32] = 0xFE
    e = np.array([[-20, 5], [0, 17], [-3, -9]])
    vals = fp8.decode_array(codes, fp8.E4M3) * np.ldexp(1.0, np.repeat(e, 32, axis=1))
    x = bits(vals)
    assert np.array_equal(quant.widen_bf16(x).astype(np.float64), vals)
    o = quant.quantize_mx(x, fp8.E4M3)
    assert np.array_equal(o["e"], e)
    assert np.array_equal(o["q"], codes)
