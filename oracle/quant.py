"""amax, scales, the scaled cast, overflow/underflow counters, fine-grained units and
delayed scaling (oracle; test infrastructure).

Sources:
* "FP8 stability guardrails" page, "Why FP8 is tempting and why it is fragile":
  values beyond the format maximum overflow or saturate, tiny ones underflow to zero;
  the first paragraph names "overflow telemetry" as a guardrail.
* Same page, "Real products, models, and research": fine-grained tile and block
  scaling factors (DeepSeek-V3) and delayed scaling with amax history tracking
  (Transformer Engine).
* "#84 FP8 Precision" page, "Explanation": weights are divided by a scale before the
  E4M3 cast so that no value overflows the exponent range.

Definitions (readings where the pages leave a step open):
* amax = max |x| over the scaling unit, NaN ignored, -0 counts as 0; 0 when empty.
* current scaling: s = fl32(FP8_MAX / amax), d = fl32(amax / FP8_MAX) if amax is
  finite and > 0 and the quotient is finite, else s = d = 1.  Dividing by the scale d is taken as multiplying by
  s, so the cast is q = cast(fl32(float(x) * s)).
* units: the whole tensor; a 1x128 row tile along the contraction dimension; a
  128x128 block.  Dimensions that are not multiples of 128 are not tiled.
* overflow = number of non-NaN inputs with |fl32(x * s)| > FP8_MAX (infinite inputs
  included); underflow = number of non-zero non-NaN inputs whose code is +-0.
* delayed scaling: a ring of ``hist_len`` fp32 amaxes and a push count n.  A cast uses
  amax_eff = max of the filled entries when n > 0.  The state's amax_cur is the running
  maximum of the delayed casts since the last ``commit``; ``commit`` pushes it at index
  n % hist_len and resets it to 0.  In bootstrap (n == 0) a cast takes its scale from
  amax_cur after adding its own amax (its own amax when it is the first cast since the
  commit).  A current-scaling cast sets amax_cur to its own amax.  The pages record one amax
  per tensor per step; with one cast of each tensor per step, this reading and "each cast
  records its own amax" give the same history and scales.

* MX units (hardware block scaling): 32 consecutive elements along the contraction
  dimension share a power-of-two scale 2^e, stored as one UE8M0 byte e + 127.  e is the
  smallest integer with FP8_MAX * 2^e >= amax of the 32 elements, so no element saturates;
  e = 0 when that amax is zero or not finite; e is clamped to [-127, 127] (the byte's
  range without its NaN code).  The cast is the same q = cast(fl32(x * 2^-e)).

Parity: amax, scales, codes and counters are pinned by brute-force tests on small
arrays (tests/test_oracle_quant.py).  The delayed-scaling state machine is "parity
unpinned" by the pages beyond those invariants (the pages name the technique only).
"""
from __future__ import annotations

import numpy as np

from . import fp8

TILE = 128


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def amax(x_bits: np.ndarray) -> np.float32:
    v = np.abs(widen_bf16(x_bits)).reshape(-1)
    v = v[~np.isnan(v)]
    if v.size == 0:
        return np.float32(0.0)
    return np.float32(v.max())


def scales_from_amax(a, fmt: str):
    """(s, d) as float32 from an amax, per the current-scaling rule. When FP8_MAX / amax
    overflows float32 (a subnormal amax), the pair falls back to 1, 1 like a zero amax, so
    that s * d stays 1 and zeros do not become NaN (0 * inf)."""
    a = np.float32(a)
    mx = np.float32(fp8.fp8_max(fmt))
    if np.isfinite(a) and a > 0:
        with np.errstate(over="ignore"):
            s = np.float32(mx / a)
        if np.isfinite(s):
            return s, np.float32(a / mx)
    return np.float32(1.0), np.float32(1.0)


def cast_with_scale(x_bits: np.ndarray, s, fmt: str):
    """codes, overflow count, underflow count for q = cast(fl32(x * s))."""
    x = widen_bf16(x_bits)
    v = (x * np.float32(s)).astype(np.float32)            # one fp32 multiply, RNE
    q = fp8.cast(v, fmt)
    mx = fp8.fp8_max(fmt)
    notnan = ~np.isnan(x)
    overflow = int(np.count_nonzero(notnan & (np.abs(v.astype(np.float64)) > mx)))
    underflow = int(np.count_nonzero(notnan & (x != 0) & ((q & 0x7F) == 0)))
    return q, overflow, underflow


def quantize_tensor(x_bits: np.ndarray, fmt: str):
    """Per-tensor current scaling.  Returns dict(q, qT, amax, s, d, overflow, underflow)."""
    a = amax(x_bits)
    s, d = scales_from_amax(a, fmt)
    q, ov, un = cast_with_scale(x_bits, s, fmt)
    out = dict(q=q, amax=a, s=s, d=d, overflow=ov, underflow=un)
    if q.ndim == 2:
        out["qT"] = np.ascontiguousarray(q.T)
    return out


def quantize_tile_1x128(x_bits: np.ndarray, fmt: str):
    """One scale per (row, 128-column tile).  Returns dict(q, d[R, C/128], amax, s, overflow, underflow)."""
    R, C = x_bits.shape
    assert C % TILE == 0
    T = C // TILE
    q = np.empty((R, C), dtype=np.uint8)
    d = np.empty((R, T), dtype=np.float32)
    s = np.empty((R, T), dtype=np.float32)
    am = np.empty((R, T), dtype=np.float32)
    ov = un = 0
    for i in range(R):
        for t in range(T):
            unit = x_bits[i, t * TILE:(t + 1) * TILE]
            a = amax(unit)
            si, di = scales_from_amax(a, fmt)
            qi, o, u = cast_with_scale(unit, si, fmt)
            q[i, t * TILE:(t + 1) * TILE] = qi
            d[i, t], s[i, t], am[i, t] = di, si, a
            ov += o
            un += u
    return dict(q=q, d=d, s=s, amax=am, overflow=ov, underflow=un)


def quantize_block_128x128(w_bits: np.ndarray, fmt: str):
    """One scale per 128x128 block.  Returns dict(q, qT, d[R/128, C/128], amax, s, overflow, underflow)."""
    R, C = w_bits.shape
    assert R % TILE == 0 and C % TILE == 0
    A, B = R // TILE, C // TILE
    q = np.empty((R, C), dtype=np.uint8)
    d = np.empty((A, B), dtype=np.float32)
    s = np.empty((A, B), dtype=np.float32)
    am = np.empty((A, B), dtype=np.float32)
    ov = un = 0
    for a in range(A):
        for b in range(B):
            unit = w_bits[a * TILE:(a + 1) * TILE, b * TILE:(b + 1) * TILE]
            m = amax(unit)
            si, di = scales_from_amax(m, fmt)
            qi, o, u = cast_with_scale(unit, si, fmt)
            q[a * TILE:(a + 1) * TILE, b * TILE:(b + 1) * TILE] = qi
            d[a, b], s[a, b], am[a, b] = di, si, m
            ov += o
            un += u
    return dict(q=q, qT=np.ascontiguousarray(q.T), d=d, s=s, amax=am, overflow=ov, underflow=un)


MX_BLOCK = 32


def mx_exponent(a, fmt: str) -> int:
    """The MX scale exponent of a group with amax a: the smallest integer e with
    FP8_MAX * 2^e >= a, clamped to [-127, 127]; 0 for a zero or non-finite a."""
    a = float(np.float32(a))
    if not (np.isfinite(a) and a > 0):
        return 0
    mx = fp8.fp8_max(fmt)
    e = int(np.ceil(np.log2(a / mx)))
    while mx * 2.0 ** e < a:          # exact comparisons settle the logarithm's rounding
        e += 1
    while mx * 2.0 ** (e - 1) >= a:
        e -= 1
    return max(-127, min(127, e))


def quantize_mx(x_bits: np.ndarray, fmt: str):
    """MX scaling along the last axis of a [R, C] array (C % 32 == 0): one power-of-two
    scale per 32 consecutive elements of a row.  Returns dict(q [R, C], e [R, C/32] int,
    ue8m0 [R, C/32] uint8 = e + 127, amax [R, C/32], overflow, underflow)."""
    R, C = x_bits.shape
    assert C % MX_BLOCK == 0
    G = C // MX_BLOCK
    q = np.empty((R, C), dtype=np.uint8)
    e = np.empty((R, G), dtype=np.int64)
    am = np.empty((R, G), dtype=np.float32)
    ov = un = 0
    for i in range(R):
        for g in range(G):
            unit = x_bits[i, g * MX_BLOCK:(g + 1) * MX_BLOCK]
            a = amax(unit)
            ei = mx_exponent(a, fmt)
            qi, o, u = cast_with_scale(unit, np.float32(2.0 ** -ei), fmt)
            q[i, g * MX_BLOCK:(g + 1) * MX_BLOCK] = qi
            e[i, g], am[i, g] = ei, a
            ov += o
            un += u
    return dict(q=q, e=e, ue8m0=(e + 127).astype(np.uint8), amax=am, overflow=ov, underflow=un)


class DelayedState:
    """Per-tensor scaling state of one tensor role (x, W or dy) of one layer."""

    def __init__(self, hist_len: int = 16):
        self.hist_len = hist_len
        self.hist = np.zeros(hist_len, dtype=np.float32)
        self.count = 0
        self.scale = np.float32(1.0)
        self.scale_inv = np.float32(1.0)
        self.amax_cur = np.float32(0.0)
        self.overflow = 0
        self.underflow = 0

    def amax_eff(self):
        n = min(self.count, self.hist_len)
        if n == 0:
            return None
        return np.float32(self.hist[:n].max())

    def quantize(self, x_bits: np.ndarray, fmt: str, delayed: bool = True):
        """Cast with the delayed scale; in bootstrap with the running maximum including this
        tensor's amax; in current mode with this tensor's own amax."""
        cur = amax(x_bits)
        if delayed:
            self.amax_cur = np.float32(max(self.amax_cur, cur))
            eff = self.amax_eff()
            a = self.amax_cur if eff is None else eff
        else:
            self.amax_cur = cur
            a = cur
        s, d = scales_from_amax(a, fmt)
        q, ov, un = cast_with_scale(x_bits, s, fmt)
        self.scale, self.scale_inv = s, d
        self.overflow += ov
        self.underflow += un
        out = dict(q=q, s=s, d=d, amax=cur, overflow=ov, underflow=un)
        if q.ndim == 2:
            out["qT"] = np.ascontiguousarray(q.T)
        return out

    def commit(self):
        self.hist[self.count % self.hist_len] = self.amax_cur
        self.count += 1
        self.amax_cur = np.float32(0.0)

    def snapshot(self):
        return dict(hist=self.hist.copy(), count=self.count, scale=self.scale, scale_inv=self.scale_inv,
                    amax_cur=self.amax_cur, overflow=self.overflow, underflow=self.underflow)
