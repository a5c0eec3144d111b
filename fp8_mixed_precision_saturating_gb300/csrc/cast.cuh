// cast.cuh -- the scale rule and the saturating FP8 cast shared by the quantiser kernels and
// the GEMM epilogue that emits FP8 output.
//
// Sources: "FP8 stability guardrails" page, "Why FP8 is tempting and why it is fragile"
// (E4M3 max 448, E5M2 max 57344; out-of-range values saturate, tiny ones underflow);
// "#84 FP8 Precision" page, "Explanation" (divide by the scale before the cast).
//   s = FP8_MAX / amax, d = amax / FP8_MAX (IEEE fp32), or 1, 1 when amax is zero, not
//       finite, or so small that the quotient overflows
//   code = cvt.rn.satfinite(fl32(x * s)), NaN -> 0x7F
//   overflow counts |fl32(x * s)| > FP8_MAX; underflow counts x != 0 with a +-0 code.
// Each vector of 8 first compares its largest and smallest magnitude with two exact
// thresholds (make_scaler) and casts without per-element checks when nothing in it can
// saturate, flush to zero or be NaN.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "kernels.h"

namespace fp8gb {
namespace castops {

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {
  static constexpr float kMax = 448.0f;
  static constexpr float kHalfMinSub = 9.765625e-4f;  // 2^-10: half the smallest subnormal
};
template <>
struct Fmt<1> {
  static constexpr float kMax = 57344.0f;
  static constexpr float kHalfMinSub = 7.62939453125e-6f;  // 2^-17
};

// Two fp32 values -> two codes, byte 0 from `lo`, byte 1 from `hi`.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
  uint16_t r;
  if constexpr (FMT == 0) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

__device__ __forceinline__ void scales_from_amax(float a, float fmax, float& s, float& d) {
  s = 1.0f;
  d = 1.0f;
  if (a > 0.0f && a <= 3.402823466e38f) {
    const float si = __fdiv_rn(fmax, a);
    if (si <= 3.402823466e38f) {  // a subnormal amax can overflow the quotient: keep 1, 1
      s = si;
      d = __fdiv_rn(a, fmax);
    }
  }
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) {
  __nv_bfloat162 r;
  memcpy(&r, &u, sizeof(r));
  return r;
}

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 b) {
  uint32_t r;
  memcpy(&r, &b, sizeof(r));
  return r;
}

// Running max of |x| over words of two bf16, one max per half; NaN is ignored (the bf16
// maximum returns the other operand, and the running value starts at +0 and is never NaN).
__device__ __forceinline__ uint32_t absmax_h2(uint32_t m, uint32_t w) {
  return as_u32(__hmax2(as_bf2(m), as_bf2(w & 0x7FFF7FFFu)));
}

__device__ __forceinline__ uint32_t absmax_v(uint32_t m, const uint4& v) {
  return absmax_h2(absmax_h2(absmax_h2(absmax_h2(m, v.x), v.y), v.z), v.w);
}

// The larger half, as bf16 magnitude bits (non-negative bf16 order = integer order).
__device__ __forceinline__ uint32_t fold2(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

// ---------------------------------------------------------------------------------------
// exact per-element path (with counters and the canonical NaN code)
// ---------------------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ uint32_t cast_word(uint32_t w, float s, uint32_t& ov, uint32_t& un) {
  const float x0 = __uint_as_float(w << 16);
  const float x1 = __uint_as_float(w & 0xFFFF0000u);
  const float v0 = __fmul_rn(x0, s);
  const float v1 = __fmul_rn(x1, s);
  uint32_t c = cvt2<FMT>(v0, v1);
  if (x0 != x0) c = (c & 0xFF00u) | 0x7Fu;
  if (x1 != x1) c = (c & 0x00FFu) | 0x7F00u;
  ov += (fabsf(v0) > Fmt<FMT>::kMax) + (fabsf(v1) > Fmt<FMT>::kMax);
  un += ((x0 != 0.0f) & ((c & 0x7Fu) == 0u)) + ((x1 != 0.0f) & ((c & 0x7F00u) == 0u));
  return c;
}

template <int FMT>
__device__ __forceinline__ uint2 cast8_exact(uint4 v, float s, uint32_t& ov, uint32_t& un) {
  uint2 o;
  o.x = cast_word<FMT>(v.x, s, ov, un) | (cast_word<FMT>(v.y, s, ov, un) << 16);
  o.y = cast_word<FMT>(v.z, s, ov, un) | (cast_word<FMT>(v.w, s, ov, un) << 16);
  return o;
}

template <int FMT>
__device__ __forceinline__ uint8_t cast1(uint16_t b, float s, uint32_t& ov, uint32_t& un) {
  const float x = __uint_as_float(static_cast<uint32_t>(b) << 16);
  const float v = __fmul_rn(x, s);
  uint32_t c = cvt2<FMT>(v, 0.0f) & 0xFFu;
  if (x != x) c = 0x7Fu;
  ov += fabsf(v) > Fmt<FMT>::kMax;
  un += (x != 0.0f) & ((c & 0x7Fu) == 0u);
  return static_cast<uint8_t>(c);
}

// ---------------------------------------------------------------------------------------
// fast path
// ---------------------------------------------------------------------------------------
// T_ov is the largest bf16 magnitude whose scaled value fl32(|x| s) stays <= FP8_MAX, T_un
// the largest whose scaled value is <= half the smallest subnormal (code +-0). Both are
// exact: fl32(|x| s) and the cast are monotone in |x|, so |x| <= T_ov means no saturation
// and |x| > T_un means no flush to zero. NaN fails both comparisons and zeros fail the
// second, so such vectors, and any that may saturate or flush, take the exact path.
struct Scaler {
  float s;
  __nv_bfloat162 tov;
  __nv_bfloat162 tun;
};

// Largest bf16 magnitude bits b (0 .. 0x7F7F) with fl32(bf16(b) * s) <= target. `d` is the
// reciprocal scale, so fl32(target * d) lands within a few fp32 ulps of target / s and the
// two exact adjustment loops move by at most a step or two.
__device__ __forceinline__ uint32_t bf16_threshold(float s, float d, float target) {
  const float q = __fmul_rn(target, d);
  uint32_t b = min(__float_as_uint(q) >> 16, 0x7F7Fu);
  while (b < 0x7F7Fu && __fmul_rn(__uint_as_float((b + 1u) << 16), s) <= target) ++b;
  while (b > 0u && __fmul_rn(__uint_as_float(b << 16), s) > target) --b;
  return b;
}

template <int FMT>
__device__ __forceinline__ Scaler make_scaler(float s, float d) {
  Scaler c;
  c.s = s;
  const uint32_t tov = bf16_threshold(s, d, Fmt<FMT>::kMax);
  const uint32_t tun = bf16_threshold(s, d, Fmt<FMT>::kHalfMinSub);
  c.tov = as_bf2(tov | (tov << 16));
  c.tun = as_bf2(tun | (tun << 16));
  return c;
}

// 8 bf16 -> 8 codes with exact counters; with AMAX, `am` accumulates max |x| (NaN ignored)
// as two bf16 magnitudes.
template <int FMT, bool AMAX>
__device__ __forceinline__ uint2 cast8(uint4 v, const Scaler& c, uint32_t& ov, uint32_t& un, uint32_t& am) {
  const __nv_bfloat162 b0 = as_bf2(v.x & 0x7FFF7FFFu), b1 = as_bf2(v.y & 0x7FFF7FFFu);
  const __nv_bfloat162 b2 = as_bf2(v.z & 0x7FFF7FFFu), b3 = as_bf2(v.w & 0x7FFF7FFFu);
  const __nv_bfloat162 mx = __hmax2_nan(__hmax2_nan(b0, b1), __hmax2_nan(b2, b3));
  const __nv_bfloat162 mn = __hmin2_nan(__hmin2_nan(b0, b1), __hmin2_nan(b2, b3));
  if (__hble2(mx, c.tov) && __hbgt2(mn, c.tun)) {
    if constexpr (AMAX) am = as_u32(__hmax2(as_bf2(am), mx));
    const float s = c.s;
    uint2 o;
    o.x = cvt2<FMT>(__fmul_rn(__uint_as_float(v.x << 16), s), __fmul_rn(__uint_as_float(v.x & 0xFFFF0000u), s)) |
          (cvt2<FMT>(__fmul_rn(__uint_as_float(v.y << 16), s), __fmul_rn(__uint_as_float(v.y & 0xFFFF0000u), s))
           << 16);
    o.y = cvt2<FMT>(__fmul_rn(__uint_as_float(v.z << 16), s), __fmul_rn(__uint_as_float(v.z & 0xFFFF0000u), s)) |
          (cvt2<FMT>(__fmul_rn(__uint_as_float(v.w << 16), s), __fmul_rn(__uint_as_float(v.w & 0xFFFF0000u), s))
           << 16);
    return o;
  }
  if constexpr (AMAX) am = absmax_v(am, v);
  return cast8_exact<FMT>(v, c.s, ov, un);
}


// The amax a per-tensor cast uses: the history maximum in delayed mode once the history
// holds an entry, otherwise the current amax (computed by the amax pass).
__device__ __forceinline__ float effective_amax(const QuantState& st, bool delayed) {
  if (delayed) {
    const int n = *st.hist_count;
    if (n > 0) {
      const int m = min(n, st.hist_len);
      float a = 0.0f;
      for (int i = 0; i < m; ++i) a = fmaxf(a, st.hist[i]);
      return a;
    }
  }
  return *st.amax_cur;
}

__device__ __forceinline__ void atomic_max_amax(float* amax, uint32_t bf16_bits) {
  if (bf16_bits != 0) atomicMax(reinterpret_cast<unsigned int*>(amax), bf16_bits << 16);
}

}  // namespace castops
}  // namespace fp8gb
