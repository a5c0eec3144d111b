"""Pins of the oracle's FP8 formats and cast against facts outside the oracle itself:
the pages' printed maxima and bit counts, torch's float8 dtypes (run, not read), an
argmin search over every code for all 65,536 bf16 bit patterns, closed-form ties and
the format invariants."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_format_facts.txt")


def _facts():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = int(v)
    return out


def all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    return bits.view(np.float32)


def brute_force_cast(v, fmt):
    """Nearest finite code by exhaustive distance over every code; ties to the even code;
    |v| >= max saturates; NaN -> 0x7F; sign kept.  Independent of fp8.cast's neighbour search."""
    tab = fp8.decode_table(fmt)
    pos = [c for c in range(128) if math.isfinite(tab[c])]
    vals = tab[pos]
    top = max(pos, key=lambda c: tab[c])
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(np.where(np.isnan(v), 0.0, v))
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among the tied candidates prefer an even code
    even = np.array([c % 2 == 0 for c in pos])
    pick_even = cand & even[None, :]
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, np.argmax(pick_even, axis=1), np.argmax(cand, axis=1))
    code = np.array(pos)[idx]
    code = np.where(a >= tab[top], top, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def test_page_facts_maxima_and_bits():
    f = _facts()
    assert fp8.fp8_max(fp8.E4M3) == f["e4m3_max"]
    assert fp8.fp8_max(fp8.E5M2) == f["e5m2_max"]
    assert fp8._SPEC[fp8.E4M3]["exp_bits"] == f["e4m3_exponent_bits"]
    assert fp8._SPEC[fp8.E4M3]["man_bits"] == f["e4m3_mantissa_bits"]
    assert fp8._SPEC[fp8.E5M2]["exp_bits"] == f["e5m2_exponent_bits"]
    assert fp8._SPEC[fp8.E5M2]["man_bits"] == f["e5m2_mantissa_bits"]
    # 1 sign + exponent + mantissa = 8 bits
    for k in ("e4m3", "e5m2"):
        assert 1 + f[k + "_exponent_bits"] + f[k + "_mantissa_bits"] == 8
    # the maximum codes
    assert fp8.max_code(fp8.E4M3) == 0x7E and fp8.max_code(fp8.E5M2) == 0x7B


@pytest.mark.parametrize("fmt,tdt", [(fp8.E4M3, torch.float8_e4m3fn), (fp8.E5M2, torch.float8_e5m2)])
def test_decode_all_codes_against_torch(fmt, tdt):
    ours = fp8.decode_table(fmt)
    theirs = torch.arange(256, dtype=torch.uint8).view(tdt).to(torch.float64).numpy()
    nan_o, nan_t = np.isnan(ours), np.isnan(theirs)
    assert np.array_equal(nan_o, nan_t)
    assert np.array_equal(ours[~nan_o], theirs[~nan_t])
    # signed zero
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_decode_special_codes():
    assert math.isnan(fp8.decode(0x7F, fp8.E4M3)) and math.isnan(fp8.decode(0xFF, fp8.E4M3))
    assert sum(math.isnan(v) for v in fp8.decode_table(fp8.E4M3)) == 2
    assert fp8.decode(0x7C, fp8.E5M2) == math.inf and fp8.decode(0xFC, fp8.E5M2) == -math.inf
    assert sum(math.isnan(v) for v in fp8.decode_table(fp8.E5M2)) == 6
    # smallest subnormals and normals
    assert fp8.decode(0x01, fp8.E4M3) == 2.0 ** -9 and fp8.decode(0x08, fp8.E4M3) == 2.0 ** -6
    assert fp8.decode(0x01, fp8.E5M2) == 2.0 ** -16 and fp8.decode(0x04, fp8.E5M2) == 2.0 ** -14
    assert fp8.decode(0x38, fp8.E4M3) == 1.0 and fp8.decode(0x3C, fp8.E5M2) == 1.0


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_cast_every_bf16_pattern_against_brute_force(fmt):
    v = all_bf16_values()
    assert np.array_equal(fp8.cast(v, fmt), brute_force_cast(v, fmt))


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_cast_scaled_bf16_patterns_against_brute_force(fmt):
    # fp32 values that are not bf16: products x*s as the quantiser forms them
    rng = np.random.default_rng(7)
    v = all_bf16_values()
    s = np.float32(rng.uniform(0.5, 2.0))
    w = (v * s).astype(np.float32)
    assert np.array_equal(fp8.cast(w, fmt), brute_force_cast(w, fmt))


@pytest.mark.parametrize("fmt,tdt", [(fp8.E4M3, torch.float8_e4m3fn), (fp8.E5M2, torch.float8_e5m2)])
def test_cast_matches_torch_within_range(fmt, tdt):
    v = all_bf16_values()
    keep = np.isfinite(v) & (np.abs(v) <= fp8.fp8_max(fmt))
    v = v[keep]
    theirs = torch.from_numpy(v.copy()).to(tdt).view(torch.uint8).numpy()
    ours = fp8.cast(v, fmt)
    assert np.array_equal(ours, theirs)


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_round_trip_monotone_and_symmetric(fmt):
    tab = fp8.decode_table(fmt)
    for c in range(256):
        if math.isnan(tab[c]):
            continue
        got = int(fp8.cast(np.array([tab[c]]), fmt)[0])
        if math.isinf(tab[c]):
            assert got == (fp8.max_code(fmt) | (c & 0x80))
        else:
            assert got == c
    v = all_bf16_values()
    v = v[~np.isnan(v)]
    order = np.argsort(v, kind="stable")
    dec = fp8.decode_array(fp8.cast(v[order], fmt), fmt)
    assert np.all(np.diff(dec) >= 0)
    assert np.array_equal(fp8.cast(-v, fmt), fp8.cast(v, fmt) ^ 0x80)


def test_special_inputs():
    for fmt, mx in ((fp8.E4M3, 0x7E), (fp8.E5M2, 0x7B)):
        v = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, -1e-30, 1e-30, 1e9, -1e9], dtype=np.float32)
        got = fp8.cast(v, fmt).tolist()
        assert got == [0x7F, 0x7F, mx, 0x80 | mx, 0x00, 0x80, 0x80, 0x00, mx, 0x80 | mx]


def test_closed_form_ties():
    E = fp8.E4M3
    # 1.0 = 0x38, 1.125 = 0x39, 1.25 = 0x3A: midpoints go to the even code
    assert fp8.cast(np.array([1.0625]), E)[0] == 0x38
    assert fp8.cast(np.array([1.1875]), E)[0] == 0x3A
    # just above a midpoint goes up, just below goes down
    assert fp8.cast(np.array([np.nextafter(1.0625, 2.0)]), E)[0] == 0x39
    assert fp8.cast(np.array([np.nextafter(1.0625, 0.0)]), E)[0] == 0x38
    # subnormal / normal boundary: 7/8 * 2^-6 = 0x07, 2^-6 = 0x08; midpoint 15/16 * 2^-6 -> even 0x08
    assert fp8.cast(np.array([15 / 16 * 2.0 ** -6]), E)[0] == 0x08
    # half the smallest subnormal ties to zero (even), a bit more rounds to 0x01
    assert fp8.cast(np.array([2.0 ** -10]), E)[0] == 0x00
    assert fp8.cast(np.array([np.nextafter(2.0 ** -10, 1.0)]), E)[0] == 0x01
    # top of the range: 416 (0x7D) .. 448 (0x7E); midpoint 432 -> even 0x7E
    assert fp8.cast(np.array([432.0]), E)[0] == 0x7E
    assert fp8.cast(np.array([431.0]), E)[0] == 0x7D
    F = fp8.E5M2
    # 1.0 = 0x3C, 1.25 = 0x3D: midpoint 1.125 -> even 0x3C; 1.375 -> 0x3E
    assert fp8.cast(np.array([1.125]), F)[0] == 0x3C
    assert fp8.cast(np.array([1.375]), F)[0] == 0x3E
    # 49152 (0x7A) .. 57344 (0x7B): the midpoint 53248 goes to the even code 0x7A
    assert fp8.cast(np.array([53248.0]), F)[0] == 0x7A
    assert fp8.cast(np.array([53249.0]), F)[0] == 0x7B


def test_pins_catch_a_planted_bias_error(monkeypatch):
    """A planted mistake in the oracle (wrong E4M3 bias) must fail the pins."""
    monkeypatch.setitem(fp8._SPEC, fp8.E4M3, dict(exp_bits=4, man_bits=3, bias=8))
    assert fp8.fp8_max(fp8.E4M3) != 448
    theirs = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.decode_table(fp8.E4M3)
    ok = np.isnan(ours) == np.isnan(theirs)
    assert not np.array_equal(np.nan_to_num(ours), np.nan_to_num(theirs)) or not ok.all()
