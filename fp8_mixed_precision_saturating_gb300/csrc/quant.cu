// quant.cu -- amax reductions, scales and the saturating FP8 casts (HBM-bound kernels).
//
// Sources: "FP8 stability guardrails" page, "Why FP8 is tempting and why it is fragile"
// (E4M3 max 448, E5M2 max 57344; out-of-range values saturate, tiny ones underflow) and
// "Real products, models, and research" (1x128 tile / 128x128 block scales, delayed
// scaling with an amax history); "#84 FP8 Precision" page, "Explanation" (the tensor is
// divided by its scale before the cast).
//
// Arithmetic, identical in every kernel:
//   amax  = max |x| over the unit, NaN ignored
//   s     = FP8_MAX / amax, d = amax / FP8_MAX (IEEE fp32 divisions); 1, 1 when amax is
//           zero or not finite, or when the quotient overflows fp32 (subnormal amax)
//   code  = cvt.rn.satfinite(x * s) (one fp32 multiply), NaN -> 0x7F
//   overflow  counts |x * s| > FP8_MAX; underflow counts x != 0 whose code is +-0.
//
// The casts are issue-bound if every element pays for its counter and NaN checks, so each
// vector of 8 first compares its largest and smallest magnitude with two exact thresholds
// (see make_scaler) and takes a check-free path when nothing in it can saturate, flush to
// zero or be NaN.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "cast.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fp8gb {

namespace {

namespace cg = cooperative_groups;
using namespace castops;
constexpr int kThreads = 256;

// ---------------------------------------------------------------------------------------
// block-wide reductions (kThreads threads); `red` holds 2 * kThreads / 32 words
// ---------------------------------------------------------------------------------------
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

// ---------------------------------------------------------------------------------------
// 128 x 128 tiles: thread t handles rows 8*(t/16) .. +8 and columns 8*(t%16) .. +8
// ---------------------------------------------------------------------------------------
// 4x4 byte transpose of the words a0..a3 (row r = bytes of a_r) into t0..t3 (columns).
__device__ __forceinline__ void transpose4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& t0,
                                           uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  const uint32_t x0 = __byte_perm(a0, a1, 0x5140), x1 = __byte_perm(a0, a1, 0x7362);
  const uint32_t y0 = __byte_perm(a2, a3, 0x5140), y1 = __byte_perm(a2, a3, 0x7362);
  t0 = __byte_perm(x0, y0, 0x5410);
  t1 = __byte_perm(x0, y0, 0x7632);
  t2 = __byte_perm(x1, y1, 0x5410);
  t3 = __byte_perm(x1, y1, 0x7632);
}

// 8x8 byte transpose: in[r] = {lo, hi} holds row r (bytes c0..c7); out[c] the column c.
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

// This thread's 8x8 patch of tile (ty, tx); zeros outside the tensor (rows, cols % 8 == 0,
// so a patch is either wholly inside or wholly outside).
// KEEP: read with normal L2 priority (an amax pass whose cast pass follows), else evict-first.
template <bool KEEP = false>
__device__ __forceinline__ bool load_patch(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                           int64_t ty, int64_t tx, uint4 (&v)[8]) {
  const int t = threadIdx.x;
  const int64_t r0 = ty * 128 + (t >> 4) * 8;
  const int64_t c0 = tx * 128 + (t & 15) * 8;
  const bool in = (r0 < rows) && (c0 < cols);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4* a = reinterpret_cast<const uint4*>(x + (r0 + i) * ld + c0);
    v[i] = in ? (KEEP ? __ldcg(a) : __ldcs(a)) : make_uint4(0, 0, 0, 0);
  }
  return in;
}

// Write a patch already transposed (ct[cc] = the codes of the tile's column cg * 8 + cc, rows
// rg * 8 .. + 8) into qT [cols, rows] through the CTA's shared buffer tT; every thread of the
// CTA must call this. Callers alternate between two buffers from tile to tile: the barrier of
// the next call orders this call's reads of one buffer before the call after next writes it.
__device__ __forceinline__ void store_patchT(const uint2 (&ct)[8], int64_t rows, int64_t cols, int64_t ty, int64_t tx,
                                             uint8_t* __restrict__ qT, uint8_t* tT) {
  const int t = threadIdx.x;
  const int cg = t & 15, rg = t >> 4;
  // tT row R = column index within the tile, 16-byte chunks XOR-swizzled by (R / 8) % 8
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const int R = cg * 8 + cc;
    const int chunk = (rg >> 1) ^ ((R >> 3) & 7);
    *reinterpret_cast<uint2*>(tT + R * 128 + chunk * 16 + (rg & 1) * 8) = ct[cc];
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int R = p * 32 + (t >> 3);
    const int j = t & 7;
    const int64_t gr = tx * 128 + R;      // row of qT
    const int64_t gc = ty * 128 + j * 16; // column of qT
    if (gr < cols && gc < rows) {
      const uint4 val = *reinterpret_cast<const uint4*>(tT + R * 128 + ((j ^ ((R >> 3) & 7)) * 16));
      *reinterpret_cast<uint4*>(qT + gr * rows + gc) = val;
    }
  }
}

// Write the patch's codes row-major into q [rows, cols] and transposed into qT [cols, rows]
// (through the CTA's shared buffer tT; every thread of the CTA must call this).
__device__ __forceinline__ void store_patch(const uint2 (&c)[8], bool in, int64_t rows, int64_t cols, int64_t ty,
                                            int64_t tx, uint8_t* __restrict__ q, uint8_t* __restrict__ qT,
                                            uint8_t* tT) {
  const int t = threadIdx.x;
  const int cg = t & 15, rg = t >> 4;
  const int64_t r0 = ty * 128 + rg * 8;
  const int64_t c0 = tx * 128 + cg * 8;
  if (in && q != nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(q + (r0 + i) * cols + c0) = c[i];
  }
  if (qT != nullptr) {
    uint2 ct[8];
    transpose8x8(c, ct);
    store_patchT(ct, rows, cols, ty, tx, qT, tT);
  }
}

// ---------------------------------------------------------------------------------------
// per-tensor quantise
// ---------------------------------------------------------------------------------------
// One cooperative launch (every CTA resident). amax_cur holds the running maximum of the
// delayed-scaling casts of the tensor since the last history commit, which pushes it into the
// history and resets it to 0; a current-scaling cast sets it to its own tensor's amax.
//   current scaling: CTA 0 zeroes amax_cur; every CTA reduces max|x| over its share; grid
//     sync; atomicMax; grid sync; scale from amax_cur; cast.
//   delayed scaling: before the history holds an entry (bootstrap) the same amax pass onto
//     amax_cur as it stands, then the scale from it; past bootstrap, one pass with the
//     history's scale that adds its amax to amax_cur with atomicMax at the end. That pass has
//     no grid-wide sync (measured: dropping the one that used to order CTA 0's zeroing of
//     amax_cur before the atomics saved ~2 us per cast, GPT-2-small to the loop's sizes; a
//     separate bootstrap-amax kernel ahead of a plain launch cost ~4 us more instead).
// The cast pass after an amax pass gets its second read of x from L2 where x fits.
__device__ __forceinline__ bool needs_amax_pass(const QuantState& st, int delayed) {
  return !delayed || *st.hist_count == 0;
}

__device__ __forceinline__ float call_amax(const QuantState& st, int delayed) {
  return effective_amax(st, delayed != 0);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Optimizer-step update of this thread's patch: W' = bf16_rne(fl32(W) + delta), one fp32 add
// per element; W' is stored back into x (in place) and returned in v. delta is row-major
// [rows, cols] fp32.
__device__ __forceinline__ void update_patch(uint16_t* __restrict__ x, const float* __restrict__ delta, int64_t cols,
                                             int64_t ld, int64_t ty, int64_t tx, bool in, uint4 (&v)[8]) {
  if (!in) return;
  const int t = threadIdx.x;
  const int64_t r0 = ty * 128 + (t >> 4) * 8;
  const int64_t c0 = tx * 128 + (t & 15) * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4* dp = reinterpret_cast<const float4*>(delta + (r0 + i) * cols + c0);
    const float4 d0 = __ldcs(dp), d1 = __ldcs(dp + 1);
    uint4& w = v[i];
    w.x = pack_bf16x2(__fadd_rn(__uint_as_float(w.x << 16), d0.x), __fadd_rn(__uint_as_float(w.x & 0xFFFF0000u), d0.y));
    w.y = pack_bf16x2(__fadd_rn(__uint_as_float(w.y << 16), d0.z), __fadd_rn(__uint_as_float(w.y & 0xFFFF0000u), d0.w));
    w.z = pack_bf16x2(__fadd_rn(__uint_as_float(w.z << 16), d1.x), __fadd_rn(__uint_as_float(w.z & 0xFFFF0000u), d1.y));
    w.w = pack_bf16x2(__fadd_rn(__uint_as_float(w.w << 16), d1.z), __fadd_rn(__uint_as_float(w.w & 0xFFFF0000u), d1.w));
    *reinterpret_cast<uint4*>(x + (r0 + i) * ld + c0) = w;
  }
}

// The first tile index >= t0 that this CTA owns (tiles are dealt out t = blockIdx.x mod grid).
__device__ __forceinline__ uint32_t first_tile(uint32_t t0) {
  const uint32_t g = gridDim.x;
  return t0 + (blockIdx.x + g - t0 % g) % g;
}

// The history count and the window maximum of effective_amax, read by a whole warp in one
// round trip: lane i loads entry i (i + 32, ... for windows longer than 32) together with the
// count, and entries at or past the count are masked afterwards. Per entry, fmaxf(h, 0) with
// the sign cleared is what effective_amax folds in (NaN and negative entries count as 0), and
// the maximum of non-negative floats is the maximum of their bit patterns. Delayed scaling only
// (the history may be absent otherwise); every lane of the warp calls it.
struct HistoryView {
  int n;       // entries pushed so far
  float amax;  // maximum over the first min(n, hist_len) entries, 0 when n == 0
};

__device__ __forceinline__ HistoryView read_history_warp(const QuantState& st) {
  const int lane = threadIdx.x & 31;
  const int n = *st.hist_count;
  uint32_t best = 0;
  for (int base = 0; base < st.hist_len; base += 32) {
    const int i = base + lane;
    const float h = i < st.hist_len ? st.hist[i] : 0.0f;
    const uint32_t b = __float_as_uint(fmaxf(h, 0.0f)) & 0x7FFFFFFFu;
    if (i < n) best = max(best, b);
  }
  HistoryView v;
  v.n = n;
  v.amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, best));
  return v;
}

// Tiled layout: rows, cols and ld multiples of 8 (rows of 16 with qT); q and/or qT. With
// UPD the tensor is first updated in place by delta (the weight-cache refresh fused with
// the optimizer step): in the amax pass when there is one, else in the cast pass, so W and
// delta are read once.
template <int FMT, bool UPD>
__global__ void __launch_bounds__(kThreads) quant_tensor_tiles_kernel(uint16_t* __restrict__ x, int64_t rows,
                                                                      int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                                      uint8_t* __restrict__ qT, QuantState st,
                                                                      int delayed, const float* __restrict__ delta) {
  __shared__ __align__(128) uint8_t tT[2][128 * 128];  // alternating transpose buffers
  __shared__ uint32_t red[2 * kThreads / 32];
  cg::grid_group grid = cg::this_grid();
  pdl_trigger();  // the next kernel may start its prologue as this one drains
  int it = 0;     // tiles written by this CTA (picks the transpose buffer)
  // tile indices in 32 bits (the host keeps a tensor below 2^31 tiles): a 64-bit division
  // is a long subroutine, and the first one stands between the CTA's start and its first load
  const uint32_t tiles_x = static_cast<uint32_t>((cols + 127) / 128);
  const uint32_t ntiles = tiles_x * static_cast<uint32_t>((rows + 127) / 128);
  const bool pass = needs_amax_pass(st, delayed);
  if (!delayed && blockIdx.x == 0 && threadIdx.x == 0) *st.amax_cur = 0.0f;
  if (pass) {
    uint32_t m = 0;
    for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const uint32_t ty = t / tiles_x, tx = t - ty * tiles_x;
      uint4 v[8];
      const bool in = load_patch<true>(x, rows, cols, ld, ty, tx, v);
      if constexpr (UPD) update_patch(x, delta, cols, ld, ty, tx, in, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = absmax_v(m, v[i]);
    }
    const uint32_t b = block_max_u32(fold2(m), red);
    grid.sync();  // (current scaling) amax_cur is zero
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
    grid.sync();  // amax_cur holds the tensor's amax
  }
  float s, d;
  scales_from_amax(call_amax(st, delayed), Fmt<FMT>::kMax, s, d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *st.scale = s;
    *st.scale_inv = d;
  }
  const Scaler sc = make_scaler<FMT>(s, d);
  uint32_t ov = 0, un = 0, m = 0;
  // after an amax pass the tiles are walked backwards: the first ones read are still in L2
  for (uint32_t tr = blockIdx.x; tr < ntiles; tr += gridDim.x) {
    const uint32_t t = pass ? ntiles - 1 - tr : tr;
    const uint32_t ty = t / tiles_x, tx = t - ty * tiles_x;
    uint4 v[8];
    const bool in = load_patch(x, rows, cols, ld, ty, tx, v);
    if constexpr (UPD) {
      if (!pass) update_patch(x, delta, cols, ld, ty, tx, in, v);
    }
    uint2 c[8];
    uint32_t o1 = 0, u1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = cast8<FMT, true>(v[i], sc, o1, u1, m);
    if (in) {
      ov += o1;
      un += u1;
    }
    store_patch(c, in, rows, cols, ty, tx, q, qT, tT[it++ & 1]);
  }
  block_add_counters(ov, un, st.counters, red);
  if (!pass) {  // delayed scaling: this cast's amax onto the running maximum
    const uint32_t b = block_max_u32(fold2(m), red);
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
  }
}

// Several tensors of one format, tiled layout, in one cooperative launch: the tiles of all
// jobs share the grid, so tensors too small to fill the GPU alone (a weight and an activation
// at GPT-2-small sizes) cost one launch's latency. Per job exactly the single-tensor
// kernel's computation: amax pass when the job needs its own amax, the job's scale, the
// cast with counters, the delayed cast's amax record. All grid-wide syncs are shared. Four
// CTAs per SM (64 registers), so GPT-2-small's weight and activation (528 tiles) take one
// round on 152 SMs.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 4) quant_tiles_many_kernel(const __grid_constant__ TileJobs J) {
  __shared__ __align__(128) uint8_t tT[2][128 * 128];  // alternating transpose buffers
  __shared__ uint32_t red[2 * kThreads / 32];
  __shared__ uint32_t s_max[kMaxJobs];
  __shared__ int s_hn[kMaxJobs];      // history counts
  __shared__ float s_ha[kMaxJobs];    // history window maxima
  int it = 0;  // tiles written by this CTA (picks the transpose buffer)
  cg::grid_group grid = cg::this_grid();
  pdl_trigger();  // the next kernel may start its prologue as this one drains
  {  // every job's scaling state in one round trip: warp j reads job j's history
    const int w = threadIdx.x >> 5;
    if (w < J.n) {
      const TileJob& jb = J.j[w];
      HistoryView h{0, 0.0f};
      if (jb.delayed) h = read_history_warp(jb.st);
      if ((threadIdx.x & 31) == 0) {
        s_hn[w] = h.n;
        s_ha[w] = h.amax;
      }
    }
  }
  __syncthreads();
  uint32_t passmask = 0;  // jobs that need their own amax first (needs_amax_pass)
#pragma unroll
  for (int j = 0; j < kMaxJobs; ++j)
    if (j < J.n && (!J.j[j].delayed || s_hn[j] == 0)) passmask |= 1u << j;
  // current scaling restarts amax_cur; delayed scaling adds to the running maximum
  if (blockIdx.x == 0 && threadIdx.x < J.n && !J.j[threadIdx.x].delayed) *J.j[threadIdx.x].st.amax_cur = 0.0f;
  if (passmask) {
#pragma unroll
    for (int j = 0; j < kMaxJobs; ++j) {
      if (threadIdx.x == 0) s_max[j] = 0;
      if (j >= J.n || !((passmask >> j) & 1u)) continue;
      const TileJob& jb = J.j[j];
      const uint32_t t0 = static_cast<uint32_t>(jb.tile0), t1 = t0 + static_cast<uint32_t>(jb.ntiles);
      const uint32_t tx_n = static_cast<uint32_t>(jb.tiles_x);
      if (first_tile(t0) >= t1) continue;  // no tile of this job here
      uint32_t m = 0;
      for (uint32_t t = first_tile(t0); t < t1; t += gridDim.x) {
        const uint32_t lt = t - t0, ty = lt / tx_n;
        uint4 v[8];
        load_patch(jb.x, jb.rows, jb.cols, jb.ld, ty, lt - ty * tx_n, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = absmax_v(m, v[i]);
      }
      const uint32_t b = block_max_u32(fold2(m), red);
      if (threadIdx.x == 0) s_max[j] = b;
    }
    grid.sync();  // every current-scaling job's amax_cur is zero
    if (threadIdx.x < J.n && ((passmask >> threadIdx.x) & 1u) && s_max[threadIdx.x] != 0)
      atomic_max_amax(J.j[threadIdx.x].st.amax_cur, s_max[threadIdx.x]);
    grid.sync();  // amax_cur holds each such job's tensor amax
  }
  __syncthreads();  // s_max is read above before the cast loop reuses it
  bool any_delayed = false;
#pragma unroll
  for (int j = 0; j < kMaxJobs; ++j) {
    if (j >= J.n) continue;
    const TileJob& jb = J.j[j];
    const bool pass = (passmask >> j) & 1u;
    any_delayed |= !pass;
    if (threadIdx.x == 0) s_max[j] = 0;
    const uint32_t t0 = static_cast<uint32_t>(jb.tile0), t1 = t0 + static_cast<uint32_t>(jb.ntiles);
    const uint32_t tx_n = static_cast<uint32_t>(jb.tiles_x);
    if (first_tile(t0) >= t1) {  // no tile of this job here
      if (blockIdx.x == 0 && threadIdx.x == 0) {        // (CTA 0 still publishes the scale)
        float sj, dj;
        scales_from_amax(pass ? *jb.st.amax_cur : s_ha[j], Fmt<FMT>::kMax, sj, dj);
        *jb.st.scale = sj;
        *jb.st.scale_inv = dj;
      }
      continue;
    }
    float sj, dj;  // call_amax: the amax pass's result, else the history maximum
    scales_from_amax(pass ? *jb.st.amax_cur : s_ha[j], Fmt<FMT>::kMax, sj, dj);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *jb.st.scale = sj;
      *jb.st.scale_inv = dj;
    }
    const Scaler sc = make_scaler<FMT>(sj, dj);
    uint32_t ov = 0, un = 0, m = 0;
    for (uint32_t t = first_tile(t0); t < t1; t += gridDim.x) {
      const uint32_t lt = t - t0, ty = lt / tx_n, tx = lt - ty * tx_n;
      uint4 v[8];
      const bool in = load_patch(jb.x, jb.rows, jb.cols, jb.ld, ty, tx, v);
      uint2 c[8];
      uint32_t o1 = 0, u1 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = cast8<FMT, true>(v[i], sc, o1, u1, m);
      if (in) {
        ov += o1;
        un += u1;
      }
      store_patch(c, in, jb.rows, jb.cols, ty, tx, jb.q, jb.qT, tT[it++ & 1]);
    }
    block_add_counters(ov, un, jb.st.counters, red);
    if (!pass) {
      const uint32_t b = block_max_u32(fold2(m), red);
      if (threadIdx.x == 0) s_max[j] = b;
    }
  }
  if (any_delayed) {  // delayed casts past bootstrap add their amax to the running maximum
    __syncthreads();  // thread 0's s_max entries
    if (threadIdx.x < J.n && !((passmask >> threadIdx.x) & 1u) && s_max[threadIdx.x] != 0)
      atomic_max_amax(J.j[threadIdx.x].st.amax_cur, s_max[threadIdx.x]);
  }
}

// Row-major layout of any shape (vector path when contiguous, element path otherwise).
template <int FMT>
__global__ void __launch_bounds__(kThreads) quant_tensor_flat_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                     int64_t cols, int64_t ld,
                                                                     uint8_t* __restrict__ q, QuantState st,
                                                                     int delayed, const int32_t* gate) {
  __shared__ uint32_t red[2 * kThreads / 32];
  // gate: run only while that history is empty (the bootstrap cast of a GEMM's FP8 output);
  // every CTA reads the same count and leaves before any grid-wide sync
  if (gate != nullptr && *gate != 0) return;
  cg::grid_group grid = cg::this_grid();
  pdl_trigger();  // the next kernel may start its prologue as this one drains
  const int64_t tid = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * kThreads;
  const int64_t n = rows * cols;
  const bool flat = (ld == cols);
  const int64_t nv = flat ? n / 16 : 0;  // 16 elements per step: 2 x 16 B in, 16 B out
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const bool pass = needs_amax_pass(st, delayed);
  if (!delayed && blockIdx.x == 0 && threadIdx.x == 0) *st.amax_cur = 0.0f;
  if (pass) {
    uint32_t m = 0;
    // read with normal L2 priority: the cast pass below walks the tensor backwards, so its
    // first reads find the lines this pass read last still in L2
    for (int64_t i = tid; i < nv; i += nth) m = absmax_v(absmax_v(m, __ldcg(xv + 2 * i)), __ldcg(xv + 2 * i + 1));
    for (int64_t j = nv * 16 + tid; j < n; j += nth) m = absmax_h2(m, x[flat ? j : (j / cols) * ld + j % cols]);
    const uint32_t b = block_max_u32(fold2(m), red);
    grid.sync();  // (current scaling) amax_cur is zero
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
    grid.sync();  // amax_cur holds the tensor's amax
  }
  float s, d;
  scales_from_amax(call_amax(st, delayed), Fmt<FMT>::kMax, s, d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *st.scale = s;
    *st.scale_inv = d;
  }
  const Scaler sc = make_scaler<FMT>(s, d);
  uint32_t ov = 0, un = 0, m = 0;
  uint4* qv = reinterpret_cast<uint4*>(q);
  // after an amax pass the tensor is walked backwards (vector nv - 1 - i), so that the first
  // reads find the lines that pass read last still in L2; a single pass walks it forwards
  // (measured faster for a lone streaming pass)
  const int64_t rv = pass ? nv - 1 : 0, sv = pass ? -1 : 1;
  int64_t i = tid;
  for (; i + nth < nv; i += 2 * nth) {
    uint4 a[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t v = rv + sv * (i + u * nth);
      a[u][0] = __ldcs(xv + 2 * v);
      a[u][1] = __ldcs(xv + 2 * v + 1);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint2 lo = cast8<FMT, true>(a[u][0], sc, ov, un, m);
      const uint2 hi = cast8<FMT, true>(a[u][1], sc, ov, un, m);
      qv[rv + sv * (i + u * nth)] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  }
  for (; i < nv; i += nth) {
    const int64_t v = rv + sv * i;
    const uint2 lo = cast8<FMT, true>(__ldcs(xv + 2 * v), sc, ov, un, m);
    const uint2 hi = cast8<FMT, true>(__ldcs(xv + 2 * v + 1), sc, ov, un, m);
    qv[v] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  for (int64_t j = nv * 16 + tid; j < n; j += nth) {
    const uint16_t b = x[flat ? j : (j / cols) * ld + j % cols];
    m = absmax_h2(m, b);
    q[j] = cast1<FMT>(b, s, ov, un);
  }
  block_add_counters(ov, un, st.counters, red);
  if (!pass) {  // delayed scaling: this cast's amax onto the running maximum
    const uint32_t b = block_max_u32(fold2(m), red);
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
  }
}


// ---------------------------------------------------------------------------------------
// 128 x 128 block scales: one CTA per block, amax of the block, then its cast
// ---------------------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kThreads) cast_block_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                              uint8_t* __restrict__ qT, float* unit_scale_inv,
                                                              QuantState st) {
  __shared__ __align__(128) uint8_t tT[128 * 128];
  __shared__ uint32_t red[2 * kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int64_t ty = blockIdx.y, tx = blockIdx.x;
  uint4 v[8];
  const bool in = load_patch(x, rows, cols, ld, ty, tx, v);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = absmax_v(m, v[i]);
  const uint32_t b = block_max_u32(fold2(m), red);
  float s, d;
  scales_from_amax(__uint_as_float(b << 16), Fmt<FMT>::kMax, s, d);
  if (threadIdx.x == 0) {
    unit_scale_inv[ty * gridDim.x + tx] = d;
    if (st.amax_cur != nullptr) atomic_max_amax(st.amax_cur, b);
  }
  const Scaler sc = make_scaler<FMT>(s, d);
  uint32_t ov = 0, un = 0, dummy = 0;
  uint2 c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = cast8<FMT, false>(v[i], sc, ov, un, dummy);
  if (!in) ov = un = 0;
  store_patch(c, in, rows, cols, ty, tx, q, qT, tT);
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
}

// ---------------------------------------------------------------------------------------
// 1 x 128 tile cast: four lanes per tile, 32 elements per lane
// ---------------------------------------------------------------------------------------
// Lane l of a tile's group of four loads the 16-byte chunks l, l+4, l+8, l+12 of the tile's
// 256 bytes, so each load instruction reads 64 contiguous bytes per tile.
template <int FMT>
__global__ void __launch_bounds__(kThreads) cast_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                              float* __restrict__ unit_scale_inv, QuantState st) {
  __shared__ uint32_t red[2 * kThreads / 32];
  pdl_wait();
  pdl_trigger();
  // tile indices in 32 bits (the host keeps a tensor below 2^31 tiles): a 64-bit division
  // per tile is a long subroutine
  const uint32_t tiles_per_row = static_cast<uint32_t>(cols / 128);
  const uint32_t ntiles = static_cast<uint32_t>(rows) * tiles_per_row;
  const int gl = threadIdx.x & 3;  // lane within the tile's group
  const uint32_t group = (blockIdx.x * kThreads + threadIdx.x) >> 2;
  const uint32_t ngroups = (gridDim.x * kThreads) >> 2;
  uint32_t ov = 0, un = 0, mall = 0;
  // every lane of a warp runs the same number of iterations (the shuffles need it)
  const uint32_t warp_first = group & ~7u;
  for (uint32_t base = warp_first; base < ntiles; base += ngroups) {
    const uint32_t tile = base + (group & 7);
    const bool ok = tile < ntiles;
    const uint32_t r = ok ? tile / tiles_per_row : 0, tc = ok ? tile - r * tiles_per_row : 0;
    const uint16_t* src = x + r * ld + tc * 128;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[j] = ok ? __ldcs(reinterpret_cast<const uint4*>(src + (j * 4 + gl) * 8)) : make_uint4(0, 0, 0, 0);
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) m = absmax_v(m, v[j]);
    m = fold2(m);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    mall = max(mall, m);
    float s, d;
    scales_from_amax(__uint_as_float(m << 16), Fmt<FMT>::kMax, s, d);
    const Scaler sc = make_scaler<FMT>(s, d);
    uint32_t o1 = 0, u1 = 0, dummy = 0;
    uint8_t* dst = q + r * cols + tc * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 cq = cast8<FMT, false>(v[j], sc, o1, u1, dummy);
      if (ok) *reinterpret_cast<uint2*>(dst + (j * 4 + gl) * 8) = cq;
    }
    if (ok) {
      if (gl == 0) unit_scale_inv[tile] = d;
      ov += o1;
      un += u1;
    }
  }
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
  if (st.amax_cur != nullptr) {
    const uint32_t b = block_max_u32(mall, red);
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
  }
}

// ---------------------------------------------------------------------------------------
// MX units: 32 consecutive elements along the contraction dimension share a power-of-two
// scale 2^e, stored as the UE8M0 byte e + 127 in the tensor cores' scale-factor layout
// ---------------------------------------------------------------------------------------
// e is the smallest integer with FP8_MAX * 2^e >= amax (nothing saturates), 0 for a zero or
// non-finite amax, at least -127. With amax = (1 + f / 128) 2^(E - 1) (bf16 exponent field
// E + 126, 7-bit fraction f) and FP8_MAX = 0.875 * 2^EMX (EMX = 9 for E4M3, 16 for E5M2):
// amax <= FP8_MAX * 2^(E - EMX) exactly when 1 + f / 128 <= 1.75, i.e. f <= 96; otherwise
// one more. A subnormal amax (below 2^-126) needs e below -127: clamped.
template <int FMT>
__device__ __forceinline__ int mx_exponent(uint32_t b) {
  constexpr int EMX = FMT == 0 ? 9 : 16;
  if (b == 0u || b >= 0x7F80u) return 0;
  const int eb = static_cast<int>(b >> 7);
  if (eb == 0) return -127;
  const int e = (eb - 126) - EMX + ((b & 0x7Fu) > 96u ? 1 : 0);
  return e < -127 ? -127 : e;
}

// 2^e for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Byte offset of the scale of MN index mn and contraction block kb (128 elements = 4 groups,
// one byte each) in atoms of 512 bytes, [ceil(MN / 128)][nkb]; inside an atom the four bytes
// of mn sit at 16 (mn % 32) + 4 ((mn / 32) % 4).
__device__ __forceinline__ int64_t mx_sf_offset(int64_t mn, int64_t kb, int64_t nkb) {
  return ((mn >> 7) * nkb + kb) * 512 + 16 * (mn & 31) + 4 * ((mn >> 5) & 3);
}

// Rows of x [rows, cols] in groups of 32 along the row (activations, contraction = cols;
// cols % 128 == 0). Four lanes per 128-element tile as in the 1 x 128 cast: lane l holds the
// 16-byte chunks l, l + 4, l + 8, l + 12, i.e. chunk l of each of the tile's four groups, so a
// group's amax is the maximum over the four lanes. The tiles of rows past the last (up to a
// multiple of 128) only write their scale bytes (e = 0).
template <int FMT>
__global__ void __launch_bounds__(kThreads) cast_mx_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                                uint8_t* __restrict__ sf, QuantState st) {
  __shared__ uint32_t red[2 * kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const uint32_t kbs = static_cast<uint32_t>(cols / 128);
  const uint32_t prow = static_cast<uint32_t>((rows + 127) & ~int64_t(127));
  const uint32_t ntiles = prow * kbs;
  const int gl = threadIdx.x & 3;
  const uint32_t group = (blockIdx.x * kThreads + threadIdx.x) >> 2;
  const uint32_t ngroups = (gridDim.x * kThreads) >> 2;
  uint32_t ov = 0, un = 0, mall = 0;
  // every lane of a warp runs the same number of iterations (the shuffles need it)
  const uint32_t warp_first = group & ~7u;
  for (uint32_t base = warp_first; base < ntiles; base += ngroups) {
    const uint32_t tile = base + (group & 7);
    const bool live = tile < ntiles;
    const uint32_t r = live ? tile / kbs : 0, kb = live ? tile - r * kbs : 0;
    const bool ok = live && r < rows;
    const uint16_t* src = x + static_cast<int64_t>(r) * ld + kb * 128;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[j] = ok ? __ldcs(reinterpret_cast<const uint4*>(src + (j * 4 + gl) * 8)) : make_uint4(0, 0, 0, 0);
    uint32_t word = 0, o1 = 0, u1 = 0, dummy = 0;
    uint2 cq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t m = fold2(absmax_v(0u, v[j]));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      mall = max(mall, m);
      const int e = mx_exponent<FMT>(m);
      cq[j] = cast8<FMT, false>(v[j], make_scaler<FMT>(pow2f(-e), pow2f(e)), o1, u1, dummy);
      word |= static_cast<uint32_t>(e + 127) << (8 * j);
    }
    if (ok) {
      uint8_t* dst = q + static_cast<int64_t>(r) * cols + kb * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint2*>(dst + (j * 4 + gl) * 8) = cq[j];
      ov += o1;
      un += u1;
    }
    if (live && gl == 0) *reinterpret_cast<uint32_t*>(sf + mx_sf_offset(r, kb, kbs)) = word;
  }
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
  if (st.amax_cur != nullptr) {
    const uint32_t b = block_max_u32(mall, red);
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
  }
}

// 8 x 8 transpose of bf16 elements: in[i] holds row i (8 halves), out[j] column j.
__device__ __forceinline__ void transpose8x8_h16(const uint4 (&in)[8], uint4 (&out)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t* a = reinterpret_cast<const uint32_t*>(&in[2 * k]);
      const uint32_t* b = reinterpret_cast<const uint32_t*>(&in[2 * k + 1]);
      w[k] = __byte_perm(a[j >> 1], b[j >> 1], (j & 1) ? 0x7632 : 0x5410);
    }
    out[j] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Columns of W [rows, cols] in groups of 32 along the column (weights, contraction = rows;
// rows % 128 == 0, cols % 8 == 0), codes written transposed into qT [cols, rows]. One CTA per
// 128 x 128 tile: each thread transposes its 8 x 8 patch in registers (a column of W becomes a
// row of 8), the CTA reduces each column's maximum over each group of 32 rows through shared
// memory, computes the 512 scales of the tile once, and casts and stores the transposed codes;
// the tile's scales are one 512-byte atom. Tiles past the last column write e = 0.
template <int FMT>
__global__ void __launch_bounds__(kThreads) cast_mx_cols_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                int64_t cols, int64_t ld, uint8_t* __restrict__ qT,
                                                                uint8_t* __restrict__ sf, QuantState st) {
  __shared__ __align__(128) uint8_t tT[128 * 128];
  __shared__ uint16_t cmax[16][128];  // per slab of 8 rows, each column's max |x| (bf16 bits)
  __shared__ Scaler scl[4][128];      // per group of 32 rows, each column's scaler
  __shared__ __align__(16) uint8_t atom[512];
  __shared__ uint32_t red[2 * kThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int64_t ty = blockIdx.y, tx = blockIdx.x;
  const int t = threadIdx.x;
  const int cg = t & 15, rg = t >> 4;
  uint4 v[8];
  const bool in = load_patch(x, rows, cols, ld, ty, tx, v);
  uint4 vt[8];
  transpose8x8_h16(v, vt);
#pragma unroll
  for (int j = 0; j < 8; ++j) cmax[rg][cg * 8 + j] = static_cast<uint16_t>(fold2(absmax_v(0u, vt[j])));
  __syncthreads();
  uint32_t mall = 0;
  for (int p = t; p < 512; p += kThreads) {
    const int c = p & 127, g = p >> 7;
    const uint32_t m = max(max(static_cast<uint32_t>(cmax[4 * g][c]), static_cast<uint32_t>(cmax[4 * g + 1][c])),
                           max(static_cast<uint32_t>(cmax[4 * g + 2][c]), static_cast<uint32_t>(cmax[4 * g + 3][c])));
    mall = max(mall, m);
    const int e = mx_exponent<FMT>(m);
    scl[g][c] = make_scaler<FMT>(pow2f(-e), pow2f(e));
    atom[16 * (c & 31) + 4 * (c >> 5) + g] = static_cast<uint8_t>(e + 127);
  }
  __syncthreads();
  const int g = rg >> 2;
  uint32_t ov = 0, un = 0, dummy = 0;
  uint2 ct[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ct[j] = cast8<FMT, false>(vt[j], scl[g][cg * 8 + j], ov, un, dummy);
  if (!in) ov = un = 0;
  store_patchT(ct, rows, cols, ty, tx, qT, tT);  // (its barrier also orders the atom's writes)
  if (t < 32)
    *reinterpret_cast<uint4*>(sf + (tx * (rows / 128) + ty) * 512 + t * 16) = *reinterpret_cast<const uint4*>(atom + t * 16);
  if (st.counters != nullptr) block_add_counters(ov, un, st.counters, red);
  if (st.amax_cur != nullptr) {
    const uint32_t b = block_max_u32(mall, red);
    if (threadIdx.x == 0) atomic_max_amax(st.amax_cur, b);
  }
}

__global__ void history_commit_kernel(QuantStates sts) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < sts.n) {
    const QuantState& st = sts.s[threadIdx.x];
    const int n = *st.hist_count;
    st.hist[n % st.hist_len] = *st.amax_cur;
    *st.hist_count = n + 1;
    *st.amax_cur = 0.0f;  // the next step's delayed casts start a new running maximum
  }
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

// Grid of a cooperative launch: every CTA must be resident at once. The resident count per
// SM is queried once per kernel and device.
template <typename K>
int coop_grid(K kernel, int64_t work_items, int smem = 0) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  int nb = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    auto it = cache.find(key);
    if (it != cache.end()) {
      nb = it->second;
    } else {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, smem) != cudaSuccess || nb < 1) nb = 1;
      cache[key] = nb;
    }
  }
  int64_t g = static_cast<int64_t>(nb) * num_sms();
  if (work_items < g) g = work_items;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_coop_smem(void (*kernel)(KArgs...), int grid, cudaStream_t stream, int smem, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // cooperative (grid-wide syncs), without programmatic dependent launch: measured on GB300,
  // letting these grids start behind the previous kernel made the training step ~4 %
  // slower (their waiting blocks hold the SMs the previous kernel's tail would use)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_coop(void (*kernel)(KArgs...), int grid, cudaStream_t stream, Args&&... args) {
  return launch_coop_smem(kernel, grid, stream, 0, std::forward<Args>(args)...);
}


}  // namespace

cudaError_t launch_quant_tensor(int fmt, bool delayed, bool tiled, const void* x, int64_t rows, int64_t cols,
                                int64_t ld, void* q, void* qT, const QuantState& st, cudaStream_t stream) {
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  auto* tp = static_cast<uint8_t*>(qT);
  const int dl = delayed ? 1 : 0;
  auto go = [&](auto k, int grid, auto... args) { return launch_coop(k, grid, stream, args...); };
  if (tiled) {
    auto k = fmt == 0 ? quant_tensor_tiles_kernel<0, false> : quant_tensor_tiles_kernel<1, false>;
    const int64_t ntiles = ((cols + 127) / 128) * ((rows + 127) / 128);
    return go(k, coop_grid(k, ntiles), const_cast<uint16_t*>(xp), rows, cols, ld, qp, tp, st, dl,
              static_cast<const float*>(nullptr));
  }
  auto k = fmt == 0 ? quant_tensor_flat_kernel<0> : quant_tensor_flat_kernel<1>;
  return go(k, coop_grid(k, (rows * cols + 4095) / 4096), xp, rows, cols, ld, qp, st, dl,
            static_cast<const int32_t*>(nullptr));
}

cudaError_t launch_quant_many(int fmt, const TileJobs& jobs, cudaStream_t stream) {
  auto k = fmt == 0 ? quant_tiles_many_kernel<0> : quant_tiles_many_kernel<1>;
  int64_t total = 0;
  for (int j = 0; j < jobs.n; ++j) total += jobs.j[j].ntiles;
  return launch_coop(k, coop_grid(k, total), stream, jobs);
}

cudaError_t launch_quant_tensor_if_empty_history(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld,
                                                 void* q, const QuantState& st, cudaStream_t stream) {
  auto k = fmt == 0 ? quant_tensor_flat_kernel<0> : quant_tensor_flat_kernel<1>;
  return launch_coop(k, coop_grid(k, (rows * cols + 4095) / 4096), stream, static_cast<const uint16_t*>(x), rows,
                     cols, ld, static_cast<uint8_t*>(q), st, 1, static_cast<const int32_t*>(st.hist_count));
}

cudaError_t launch_update_quant_tensor(bool delayed, void* w, const float* delta, int64_t rows, int64_t cols,
                                       void* q, void* qT, const QuantState& st, cudaStream_t stream) {
  auto k = quant_tensor_tiles_kernel<0, true>;
  const int64_t ntiles = ((cols + 127) / 128) * ((rows + 127) / 128);
  return launch_coop(k, coop_grid(k, ntiles), stream, static_cast<uint16_t*>(w), rows, cols, cols,
                     static_cast<uint8_t*>(q), static_cast<uint8_t*>(qT), st, delayed ? 1 : 0, delta);
}

cudaError_t launch_cast_blocks(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q, void* qT,
                               float* unit_scale_inv, const QuantState& st, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>((rows + 127) / 128));
  return launch_pdl(fmt == 0 ? cast_block_kernel<0> : cast_block_kernel<1>, grid, dim3(kThreads), 0, stream,
                    static_cast<const uint16_t*>(x), rows, cols, ld, static_cast<uint8_t*>(q),
                    static_cast<uint8_t*>(qT), unit_scale_inv, st);
}

cudaError_t launch_cast_1x128(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                              float* unit_scale_inv, const QuantState& st, cudaStream_t stream) {
  const int sms = num_sms();
  const int64_t ntiles = rows * (cols / 128);
  const int g = grid_for(ntiles, kThreads / 4, sms, 8);
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  return launch_pdl(fmt == 0 ? cast_1x128_kernel<0> : cast_1x128_kernel<1>, dim3(g), dim3(kThreads), 0, stream, xp,
                    rows, cols, ld, qp, unit_scale_inv, st);
}

cudaError_t launch_cast_mx(int fmt, bool along_rows, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                           void* sf, const QuantState& st, cudaStream_t stream) {
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  auto* sp = static_cast<uint8_t*>(sf);
  if (along_rows) {
    const dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>(rows / 128));
    return launch_pdl(fmt == 0 ? cast_mx_cols_kernel<0> : cast_mx_cols_kernel<1>, grid, dim3(kThreads), 0, stream, xp,
                      rows, cols, ld, qp, sp, st);
  }
  const int64_t ntiles = ((rows + 127) / 128) * 128 * (cols / 128);
  const int g = grid_for(ntiles, kThreads / 4, num_sms(), 8);
  return launch_pdl(fmt == 0 ? cast_mx_rows_kernel<0> : cast_mx_rows_kernel<1>, dim3(g), dim3(kThreads), 0, stream, xp,
                    rows, cols, ld, qp, sp, st);
}

cudaError_t launch_history_commit(const QuantStates& sts, cudaStream_t stream) {
  return launch_pdl(history_commit_kernel, dim3(1), dim3(32), 0, stream, sts);
}

cudaError_t launch_selftest_wait(const WaitCtl& w, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(w);
  return cudaGetLastError();
}

}  // namespace fp8gb
