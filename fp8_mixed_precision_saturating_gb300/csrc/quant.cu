// quant.cu -- amax reductions, scales and the saturating FP8 casts (HBM-bound kernels).
//
// Sources: "FP8 stability guardrails" page, "Why FP8 is tempting and why it is fragile"
// (E4M3 max 448, E5M2 max 57344; out-of-range values saturate, tiny ones underflow) and
// "Real products, models, and research" (1x128 tile / 128x128 block scales, delayed
// scaling with an amax history); "#84 FP8 Precision" page, "Explanation" (the tensor is
// divided by its scale before the cast).
//
// Arithmetic, identical in every kernel:
//   amax  = max |x| over the unit, NaN ignored (integer max over the bf16 magnitude bits)
//   s     = FP8_MAX / amax, d = amax / FP8_MAX (IEEE fp32 divisions), or 1, 1 when amax is
//           zero or not finite
//   code  = cvt.rn.satfinite(x * s) (one fp32 multiply), NaN -> 0x7F
//   overflow  counts |x * s| > FP8_MAX; underflow counts x != 0 whose code is +-0.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fp8gb {

namespace {

constexpr int kThreads = 256;

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {
  static constexpr float kMax = 448.0f;
};
template <>
struct Fmt<1> {
  static constexpr float kMax = 57344.0f;
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
  if (a > 0.0f && a <= 3.402823466e38f) {
    s = __fdiv_rn(fmax, a);
    d = __fdiv_rn(a, fmax);
  } else {
    s = 1.0f;
    d = 1.0f;
  }
}

// max of the bf16 magnitudes (NaN lanes zeroed) of a 32-bit word holding two bf16.
__device__ __forceinline__ uint32_t absmax2(uint32_t m, uint32_t w) {
  const uint32_t a = w & 0x7FFF7FFFu;
  const uint32_t nan = __vcmpgtu2(a, 0x7F807F80u);
  return __vmaxu2(m, a & ~nan);
}

__device__ __forceinline__ uint32_t fold2(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

// Cast one word (two bf16) with counters. Returns the two codes in bits 0..15.
template <int FMT>
__device__ __forceinline__ uint32_t cast_word(uint32_t w, float s, uint32_t& ov, uint32_t& un) {
  const float x0 = __uint_as_float(w << 16);
  const float x1 = __uint_as_float(w & 0xFFFF0000u);
  const float v0 = __fmul_rn(x0, s);
  const float v1 = __fmul_rn(x1, s);
  uint32_t c = cvt2<FMT>(v0, v1);
  if (__vcmpgtu2(w & 0x7FFF7FFFu, 0x7F807F80u)) {  // a NaN among the two: canonical code
    if (x0 != x0) c = (c & 0xFF00u) | 0x7Fu;
    if (x1 != x1) c = (c & 0x00FFu) | 0x7F00u;
  }
  ov += (fabsf(v0) > Fmt<FMT>::kMax) + (fabsf(v1) > Fmt<FMT>::kMax);
  un += ((x0 != 0.0f) & ((c & 0x7Fu) == 0u)) + ((x1 != 0.0f) & ((c & 0x7F00u) == 0u));
  return c;
}

// 8 bf16 -> 8 codes.
template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 v, float s, uint32_t& ov, uint32_t& un) {
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

// Block-wide reductions (kThreads threads). `red` holds kThreads / 32 words.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) r = max(r, red[i]);
  return r;
}

__device__ __forceinline__ void block_add_counters(uint32_t ov, uint32_t un, unsigned long long* counters,
                                                   uint32_t* red) {
  ov = __reduce_add_sync(0xFFFFFFFFu, ov);
  un = __reduce_add_sync(0xFFFFFFFFu, un);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    red[w] = ov;
    red[w + kThreads / 32] = un;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long o = 0, u = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
      o += red[i];
      u += red[i + kThreads / 32];
    }
    if (o) atomicAdd(counters + 0, o);
    if (u) atomicAdd(counters + 1, u);
  }
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

// ---------------------------------------------------------------------------------------
// amax pass (per tensor)
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                        int64_t ld, float* amax_out, const int32_t* gate_count) {
  __shared__ uint32_t red[kThreads / 32];
  if (gate_count != nullptr && *gate_count != 0) return;  // delayed mode past bootstrap
  uint32_t m = 0;
  const int64_t tid = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * kThreads;
  if (ld == cols) {
    const int64_t n = rows * cols;
    const int64_t nv = n / 8;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    int64_t i = tid;
    for (; i + 3 * nth < nv; i += 4 * nth) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(xv + i + u * nth);
#pragma unroll
      for (int u = 0; u < 4; ++u) m = absmax2(absmax2(absmax2(absmax2(m, v[u].x), v[u].y), v[u].z), v[u].w);
    }
    for (; i < nv; i += nth) {
      const uint4 v = __ldcs(xv + i);
      m = absmax2(absmax2(absmax2(absmax2(m, v.x), v.y), v.z), v.w);
    }
    for (int64_t j = nv * 8 + tid; j < n; j += nth) m = absmax2(m, x[j]);
  } else {
    const int64_t n = rows * cols;
    for (int64_t j = tid; j < n; j += nth) m = absmax2(m, x[(j / cols) * ld + (j % cols)]);
  }
  const uint32_t b = block_max_u32(fold2(m), red);
  if (threadIdx.x == 0 && b != 0) atomicMax(reinterpret_cast<unsigned int*>(amax_out), b << 16);
}

// ---------------------------------------------------------------------------------------
// per-tensor cast, row-major output (flat when contiguous)
// ---------------------------------------------------------------------------------------
template <int FMT, bool DELAYED>
__global__ void __launch_bounds__(kThreads) cast_flat_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                             QuantState st) {
  __shared__ uint32_t red[2 * kThreads / 32];
  float s, d;
  scales_from_amax(effective_amax(st, DELAYED), Fmt<FMT>::kMax, s, d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *st.scale = s;
    *st.scale_inv = d;
  }
  uint32_t ov = 0, un = 0, m = 0;
  const int64_t tid = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * kThreads;
  if (ld == cols) {
    const int64_t n = rows * cols;
    const int64_t nv = n / 16;  // 16 elements per step: 2 x 16 B in, 16 B out
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4* qv = reinterpret_cast<uint4*>(q);
    int64_t i = tid;
    for (; i + nth < nv; i += 2 * nth) {
      uint4 a[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        a[u][0] = __ldcs(xv + 2 * (i + u * nth));
        a[u][1] = __ldcs(xv + 2 * (i + u * nth) + 1);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if constexpr (DELAYED) {
          m = absmax2(absmax2(absmax2(absmax2(m, a[u][0].x), a[u][0].y), a[u][0].z), a[u][0].w);
          m = absmax2(absmax2(absmax2(absmax2(m, a[u][1].x), a[u][1].y), a[u][1].z), a[u][1].w);
        }
        const uint2 lo = cast8<FMT>(a[u][0], s, ov, un);
        const uint2 hi = cast8<FMT>(a[u][1], s, ov, un);
        __stcs(qv + i + u * nth, make_uint4(lo.x, lo.y, hi.x, hi.y));
      }
    }
    for (; i < nv; i += nth) {
      const uint4 a0 = __ldcs(xv + 2 * i), a1 = __ldcs(xv + 2 * i + 1);
      if constexpr (DELAYED) {
        m = absmax2(absmax2(absmax2(absmax2(m, a0.x), a0.y), a0.z), a0.w);
        m = absmax2(absmax2(absmax2(absmax2(m, a1.x), a1.y), a1.z), a1.w);
      }
      const uint2 lo = cast8<FMT>(a0, s, ov, un);
      const uint2 hi = cast8<FMT>(a1, s, ov, un);
      __stcs(qv + i, make_uint4(lo.x, lo.y, hi.x, hi.y));
    }
    for (int64_t j = nv * 16 + tid; j < n; j += nth) {
      if constexpr (DELAYED) m = absmax2(m, x[j]);
      q[j] = cast1<FMT>(x[j], s, ov, un);
    }
  } else {
    const int64_t n = rows * cols;
    for (int64_t j = tid; j < n; j += nth) {
      const int64_t r = j / cols, c = j % cols;
      const uint16_t b = x[r * ld + c];
      if constexpr (DELAYED) m = absmax2(m, b);
      q[r * cols + c] = cast1<FMT>(b, s, ov, un);
    }
  }
  block_add_counters(ov, un, st.counters, red);
  if constexpr (DELAYED) {
    const uint32_t b = block_max_u32(fold2(m), red);
    if (threadIdx.x == 0 && b != 0) atomicMax(reinterpret_cast<unsigned int*>(st.amax_cur), b << 16);
  }
}

// ---------------------------------------------------------------------------------------
// 128 x 128 tile cast: row-major and/or transposed codes; per-tensor or per-block scale
// ---------------------------------------------------------------------------------------
// 8x8 byte transpose: in[r] = {lo, hi} holds row r (bytes c0..c7); out[c] the column c.
__device__ __forceinline__ void transpose4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& t0,
                                           uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  const uint32_t x0 = __byte_perm(a0, a1, 0x5140), x1 = __byte_perm(a0, a1, 0x7362);
  const uint32_t y0 = __byte_perm(a2, a3, 0x5140), y1 = __byte_perm(a2, a3, 0x7362);
  t0 = __byte_perm(x0, y0, 0x5410);
  t1 = __byte_perm(x0, y0, 0x7632);
  t2 = __byte_perm(x1, y1, 0x5410);
  t3 = __byte_perm(x1, y1, 0x7632);
}

__device__ __forceinline__ void transpose8x8(const uint2 (&in)[8], uint2 (&out)[8]) {
  uint32_t t[4];
  transpose4(in[0].x, in[1].x, in[2].x, in[3].x, t[0], t[1], t[2], t[3]);
  for (int c = 0; c < 4; ++c) out[c].x = t[c];
  transpose4(in[4].x, in[5].x, in[6].x, in[7].x, t[0], t[1], t[2], t[3]);
  for (int c = 0; c < 4; ++c) out[c].y = t[c];
  transpose4(in[0].y, in[1].y, in[2].y, in[3].y, t[0], t[1], t[2], t[3]);
  for (int c = 0; c < 4; ++c) out[4 + c].x = t[c];
  transpose4(in[4].y, in[5].y, in[6].y, in[7].y, t[0], t[1], t[2], t[3]);
  for (int c = 0; c < 4; ++c) out[4 + c].y = t[c];
}

enum ScaleKind { kTensorCurrent = 0, kTensorDelayed = 1, kBlock = 2 };

// Each CTA covers one 128x128 tile; thread t handles rows 8*(t/16) .. +8 and columns
// 8*(t%16) .. +8 of it. Requires rows % 8 == 0 and cols % 8 == 0 (and, for the block
// scale, full tiles; for the transposed output, rows % 16 == 0).
template <int FMT, int SK>
__global__ void __launch_bounds__(kThreads) cast_tile_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ qT, float* unit_scale_inv,
                                                             QuantState st) {
  __shared__ __align__(128) uint8_t tT[128 * 128];
  __shared__ uint32_t red[2 * kThreads / 32];
  const int t = threadIdx.x;
  const int cg = t & 15, rg = t >> 4;
  const int64_t r0 = (int64_t)blockIdx.y * 128 + rg * 8;
  const int64_t c0 = (int64_t)blockIdx.x * 128 + cg * 8;
  const bool in = (r0 < rows) && (c0 < cols);

  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = in ? __ldcs(reinterpret_cast<const uint4*>(x + (r0 + i) * ld + c0)) : make_uint4(0, 0, 0, 0);
  }
  uint32_t m = 0;
  if constexpr (SK != kTensorCurrent) {
#pragma unroll
    for (int i = 0; i < 8; ++i) m = absmax2(absmax2(absmax2(absmax2(m, v[i].x), v[i].y), v[i].z), v[i].w);
  }
  float s, d;
  if constexpr (SK == kBlock) {
    const uint32_t b = block_max_u32(fold2(m), red);
    const float a = __uint_as_float(b << 16);
    scales_from_amax(a, Fmt<FMT>::kMax, s, d);
    if (t == 0) {
      unit_scale_inv[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = d;
      if (st.amax_cur != nullptr && b != 0) atomicMax(reinterpret_cast<unsigned int*>(st.amax_cur), b << 16);
    }
  } else {
    scales_from_amax(effective_amax(st, SK == kTensorDelayed), Fmt<FMT>::kMax, s, d);
    if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
      *st.scale = s;
      *st.scale_inv = d;
    }
  }

  uint32_t ov = 0, un = 0;
  uint2 c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = cast8<FMT>(v[i], s, ov, un);
  if (!in) ov = un = 0;
  if (in && q != nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) __stcs(reinterpret_cast<uint2*>(q + (r0 + i) * cols + c0), c[i]);
  }
  if (qT != nullptr) {
    uint2 ct[8];
    transpose8x8(c, ct);
    // tT row R = column index within the tile, 16-byte chunks XOR-swizzled by (R / 8) % 8
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int R = cg * 8 + cc;
      const int chunk = (rg >> 1) ^ ((R >> 3) & 7);
      *reinterpret_cast<uint2*>(tT + R * 128 + chunk * 16 + (rg & 1) * 8) = ct[cc];
    }
    __syncthreads();
    const int64_t colbase = (int64_t)blockIdx.x * 128;  // rows of qT
    const int64_t rowbase = (int64_t)blockIdx.y * 128;  // columns of qT
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int R = p * 32 + (t >> 3);
      const int j = t & 7;
      const int64_t gr = colbase + R;
      const int64_t gc = rowbase + j * 16;
      if (gr < cols && gc < rows) {
        const uint4 val = *reinterpret_cast<const uint4*>(tT + R * 128 + ((j ^ ((R >> 3) & 7)) * 16));
        __stcs(reinterpret_cast<uint4*>(qT + gr * rows + gc), val);
      }
    }
  }
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
  if constexpr (SK == kTensorDelayed) {
    const uint32_t b = block_max_u32(fold2(m), red);
    if (t == 0 && b != 0) atomicMax(reinterpret_cast<unsigned int*>(st.amax_cur), b << 16);
  }
}

// ---------------------------------------------------------------------------------------
// 1 x 128 tile cast: one half-warp per tile, 8 elements per lane
// ---------------------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kThreads) cast_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                              float* __restrict__ unit_scale_inv, QuantState st) {
  __shared__ uint32_t red[2 * kThreads / 32];
  const int64_t tiles_per_row = cols / 128;
  const int64_t ntiles = rows * tiles_per_row;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  uint32_t ov = 0, un = 0, mall = 0;
  constexpr int U = 2;  // tile pairs in flight per warp
  for (int64_t base = warp * 2 * U; base < ntiles; base += nwarps * 2 * U) {
    uint4 v[U];
    int64_t tile[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      tile[u] = base + 2 * u + half;
      if (tile[u] < ntiles) {
        const int64_t r = tile[u] / tiles_per_row, tc = tile[u] % tiles_per_row;
        v[u] = __ldcs(reinterpret_cast<const uint4*>(x + r * ld + tc * 128 + hl * 8));
      } else {
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t m = fold2(absmax2(absmax2(absmax2(absmax2(0u, v[u].x), v[u].y), v[u].z), v[u].w));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      mall = max(mall, m);
      float s, d;
      scales_from_amax(__uint_as_float(m << 16), Fmt<FMT>::kMax, s, d);
      uint32_t o1 = 0, u1 = 0;
      const uint2 cq = cast8<FMT>(v[u], s, o1, u1);
      if (tile[u] < ntiles) {
        const int64_t r = tile[u] / tiles_per_row, tc = tile[u] % tiles_per_row;
        __stcs(reinterpret_cast<uint2*>(q + r * cols + tc * 128 + hl * 8), cq);
        if (hl == 0) unit_scale_inv[tile[u]] = d;
        ov += o1;
        un += u1;
      }
    }
  }
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
  if (st.amax_cur != nullptr) {
    const uint32_t b = block_max_u32(mall, red);
    if (threadIdx.x == 0 && b != 0) atomicMax(reinterpret_cast<unsigned int*>(st.amax_cur), b << 16);
  }
}

__global__ void history_commit_kernel(QuantState st) {
  const int n = *st.hist_count;
  st.hist[n % st.hist_len] = *st.amax_cur;
  *st.hist_count = n + 1;
}

__global__ void selftest_wait_kernel(WaitCtl w) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    // nothing arrives on the barrier: the bounded wait must run out
    mbar_wait(smem_u32(&bar), 0, w, DEV_ERR_WAIT_SELFTEST);
  }
}

int grid_for(int64_t work_items, int per_block, int sms, int waves) {
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = (int64_t)sms * waves;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax_out,
                        const int32_t* gate_count, cudaStream_t stream) {
  const int sms = num_sms();
  const int g = grid_for(rows * cols, kThreads * 32, sms, 8);
  amax_kernel<<<g, kThreads, 0, stream>>>(static_cast<const uint16_t*>(x), rows, cols, ld, amax_out, gate_count);
  return cudaGetLastError();
}

cudaError_t launch_cast_flat(int fmt, bool delayed, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                             const QuantState& st, cudaStream_t stream) {
  const int sms = num_sms();
  const int g = grid_for(rows * cols, kThreads * 32, sms, 8);
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  if (fmt == 0) {
    if (delayed) cast_flat_kernel<0, true><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, st);
    else cast_flat_kernel<0, false><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, st);
  } else {
    if (delayed) cast_flat_kernel<1, true><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, st);
    else cast_flat_kernel<1, false><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_cast_tiles(int fmt, int scale_kind, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                              void* qT, float* unit_scale_inv, const QuantState& st, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>((rows + 127) / 128));
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  auto* tp = static_cast<uint8_t*>(qT);
#define FP8GB_TILE_LAUNCH(F, S) cast_tile_kernel<F, S><<<grid, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, tp, unit_scale_inv, st)
  if (fmt == 0) {
    if (scale_kind == kTensorCurrent) FP8GB_TILE_LAUNCH(0, kTensorCurrent);
    else if (scale_kind == kTensorDelayed) FP8GB_TILE_LAUNCH(0, kTensorDelayed);
    else FP8GB_TILE_LAUNCH(0, kBlock);
  } else {
    if (scale_kind == kTensorCurrent) FP8GB_TILE_LAUNCH(1, kTensorCurrent);
    else if (scale_kind == kTensorDelayed) FP8GB_TILE_LAUNCH(1, kTensorDelayed);
    else FP8GB_TILE_LAUNCH(1, kBlock);
  }
#undef FP8GB_TILE_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_cast_1x128(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                              float* unit_scale_inv, const QuantState& st, cudaStream_t stream) {
  const int sms = num_sms();
  const int64_t ntiles = rows * (cols / 128);
  const int g = grid_for(ntiles, 2 * (kThreads / 32) * 2, sms, 8);
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  if (fmt == 0) cast_1x128_kernel<0><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, unit_scale_inv, st);
  else cast_1x128_kernel<1><<<g, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, unit_scale_inv, st);
  return cudaGetLastError();
}

cudaError_t launch_history_commit(const QuantState& st, cudaStream_t stream) {
  history_commit_kernel<<<1, 1, 0, stream>>>(st);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(const WaitCtl& w, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(w);
  return cudaGetLastError();
}

}  // namespace fp8gb
