"""FP8 formats and the saturating round-to-nearest-even cast (oracle; test infrastructure).

Source: "FP8 stability guardrails" page, section "Why FP8 is tempting and why it is
fragile": E4M3 spends 4 bits on the exponent and 3 on the mantissa and reaches 448;
E5M2 spends 5 and 2 and reaches about 57344; out-of-range values overflow or
saturate, tiny ones underflow to zero.  The speedrun page's code names the E4M3
type ``float8_e4m3fn`` ("fn": finite, no infinity).

Decode (sign-magnitude), with e the exponent field and f the mantissa field of m bits:
    e > 0:  (-1)^s * 2^(e - bias) * (1 + f / 2^m)
    e = 0:  (-1)^s * 2^(1 - bias) * (f / 2^m)          (subnormals)
E4M3: bias 7, m 3; e = 15 is an ordinary exponent; only f = 7 at e = 15 is NaN.
E5M2: bias 15, m 2; e = 31 holds +-inf (f = 0) and NaN (f != 0), as in IEEE 754.
The maxima 448 = 1.75 * 2^8 and 57344 = 1.75 * 2^15 fix both biases.

Cast of a real value v (readings where the pages are silent):
    NaN            -> code 0x7F (one canonical NaN for both formats)
    |v| >= max     -> +-max (saturation; infinities saturate too)
    otherwise      -> the nearest finite value, ties to the even code
    sign           -> kept, so a negative value that rounds to zero gives 0x80.

Pins (tests/test_oracle_fp8.py): the maxima printed on the page, all 256 codes of both
formats against torch's float8 dtypes, the cast of all 65,536 bf16 bit patterns against
an argmin search over every code, round trips, monotonicity and sign symmetry.
"""
from __future__ import annotations

import math

import numpy as np

E4M3 = "e4m3"
E5M2 = "e5m2"

_SPEC = {
    E4M3: dict(exp_bits=4, man_bits=3, bias=7),
    E5M2: dict(exp_bits=5, man_bits=2, bias=15),
}

NAN_CODE = 0x7F


def decode(code: int, fmt: str) -> float:
    """Value of one 8-bit code, as a Python float (exact)."""
    sp = _SPEC[fmt]
    m, bias = sp["man_bits"], sp["bias"]
    emax_field = (1 << sp["exp_bits"]) - 1
    s = (code >> 7) & 1
    e = (code >> m) & emax_field
    f = code & ((1 << m) - 1)
    if fmt == E4M3 and e == emax_field and f == (1 << m) - 1:
        return math.nan
    if fmt == E5M2 and e == emax_field:
        if f != 0:
            return math.nan
        return -math.inf if s else math.inf
    if e == 0:
        mag = math.ldexp(f, 1 - bias - m)
    else:
        mag = math.ldexp((1 << m) + f, e - bias - m)
    return -mag if s else mag


def decode_table(fmt: str) -> np.ndarray:
    """float64[256]: the value of every code."""
    return np.array([decode(c, fmt) for c in range(256)], dtype=np.float64)


def finite_positive(fmt: str):
    """(codes, values) of the non-negative finite codes, ascending in value.

    For sign-magnitude codes the value grows with the code, so the codes are
    0 .. max_code and the value of code c sits at index c.
    """
    tab = decode_table(fmt)
    codes = [c for c in range(128) if math.isfinite(tab[c])]
    vals = tab[codes]
    assert np.all(np.diff(vals) > 0)
    assert codes == list(range(len(codes)))
    return np.array(codes, dtype=np.int64), vals


def fp8_max(fmt: str) -> float:
    return float(finite_positive(fmt)[1][-1])


def max_code(fmt: str) -> int:
    return int(finite_positive(fmt)[0][-1])


def cast(v, fmt: str) -> np.ndarray:
    """Saturating round-to-nearest-even cast of real values (array-like, fp32 or fp64
    values) to 8-bit codes (uint8)."""
    v = np.asarray(v, dtype=np.float64)
    codes, vals = finite_positive(fmt)
    top = len(vals) - 1
    a = np.abs(v)
    nan = np.isnan(v)
    a_safe = np.where(nan, 0.0, a)
    sat = a_safe >= vals[top]
    # lower neighbour: vals[lo] <= a < vals[lo + 1]
    lo = np.searchsorted(vals, a_safe, side="right") - 1
    lo = np.clip(lo, 0, top - 1)
    hi = lo + 1
    d_lo = a_safe - vals[lo]          # exact: both operands are short floats
    d_hi = vals[hi] - a_safe
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(sat, top, mag)
    out = mag.astype(np.uint8) | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    out = np.where(nan, NAN_CODE, out).astype(np.uint8)
    return out


def decode_array(codes: np.ndarray, fmt: str) -> np.ndarray:
    """float64 values of an array of codes."""
    return decode_table(fmt)[np.asarray(codes, dtype=np.uint8)]
