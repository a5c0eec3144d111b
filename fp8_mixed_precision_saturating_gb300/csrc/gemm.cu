// gemm.cu -- FP8 x FP8 -> bf16 GEMM on the sm_103a tensor cores (tcgen05, kind::f8f6f4).
//
// Source: "#84 FP8 Precision" page, "Explanation": the scaled FP8 matmul of the forward
// pass, with one scale per operand and both operands contiguous along the contraction
// dimension; "Hardware precision": FP8 tensor cores. "FP8 stability guardrails" page,
// "Real products, models, and research": fine-grained 1x128 tile / 128x128 block scaling.
//
//   C[m, n] = bf16( d_a * d_b * sum_k A[m, k] B[n, k] )                    (per tensor)
//   C[m, n] = bf16( sum_kb d_a[m, kb] d_b[kb, n/128] sum_{k in kb} A B )  (block scaled)
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      one thread issues TMA loads of A [128 x 128] and B [256 x 128] (K-major,
//               128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma (M=128, N=256,
//               K=32) into a TMEM accumulator and frees ring slots with tcgen05.commit;
//   warps 2..   epilogue: tcgen05.ld of the accumulator (each warp owns the 32 TMEM lanes
//               its warp index selects), multiply by the scales, convert to bf16, stage
//               128-byte rows through swizzled shared memory and write them with TMA.
// Per tensor: two 256-column accumulators, so the epilogue of one tile overlaps the
// mainloop of the next. Block scaled: every 128-deep K block gets a fresh accumulator
// buffer (two, alternating), and 8 epilogue warps fold each block into fp32 registers
// with its scale product before the next block lands.
// Every mbarrier wait is bounded (see ptx.cuh); on a timeout the CTA stops issuing work,
// drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cast.cuh"
#include "kernels.h"
#include "ptx.cuh"

#ifdef FP8GB_TRACE  // tuning builds only: per-CTA %globaltimer stamps of the GEMM's phases
__device__ unsigned long long g_gemm_trace[1024 * 8];
#define FP8GB_STAMP(k) (g_gemm_trace[blockIdx.x * 8 + (k)] = fp8gb::globaltimer_ns())
extern "C" int fp8_trace_read(void* host, int n) {
  return cudaMemcpyFromSymbol(host, g_gemm_trace, sizeof(unsigned long long) * n) == cudaSuccess ? 0 : 1;
}
#else
#define FP8GB_STAMP(k) ((void)0)
#endif

namespace fp8gb {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int A_BYTES = BM * BK;
constexpr int STG_BYTES = 32 * 128;  // one staging buffer: 32 rows x 64 bf16
constexpr int QSTG_BYTES = 32 * 64;  // one staging buffer of FP8 output: 32 rows x 64 codes
constexpr int GROUP_M = 16;          // tile raster: 16 M-blocks share each B tile

// Tile 128 x BN (BN = 256, 192 or 128); the ring depth fills ~192 KB of shared memory, less
// when the epilogue also stages FP8 output (QF >= 0: 0 = E4M3, 1 = E5M2).
template <bool BLOCK, int BN, int QF>
struct Cfg {
  static_assert(BN == 128 || BN == 192 || BN == 256, "tile width");
  static_assert(QF < 0 || !BLOCK, "FP8 output with per-tensor scales only");
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS_ = BLOCK ? 4 * (BN / 64) : 8;
  static constexpr int QSTG_PER_WARP = QF >= 0 ? QSTG_BYTES : 0;
  static constexpr int STAGES_FIT = (230000 - EPI_WARPS_ * (STG_BYTES + QSTG_PER_WARP)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < (192 * 1024) / STAGE_BYTES ? STAGES_FIT : (192 * 1024) / STAGE_BYTES;
  static constexpr int ACC = 512 / BN;                   // accumulator buffers in TMEM
  static constexpr uint32_t TMEM_COLS = 512;
  // per tensor: two warps per TMEM lane quarter, each draining half of the tile's columns;
  // block scaled: one warp per lane quarter and 64 columns
  static constexpr int EPI_WARPS = BLOCK ? 4 * (BN / 64) : 8;
  static constexpr int STG_PER_WARP = 1;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr int OFF_QSTG = OFF_STG + EPI_WARPS * STG_PER_WARP * STG_BYTES;
  static constexpr int OFF_BAR = OFF_QSTG + EPI_WARPS * QSTG_PER_WARP;
  // full[S], empty[S], tfull[ACC], tempty[ACC], final
  static constexpr int NBAR = 2 * STAGES + 2 * ACC + 1;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_TMEM_SLOT + 16 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory");
};

struct KParams {
  int M, N, K;
  int num_m, num_n, num_kb, num_tiles;
  uint32_t idesc;
  const float* sa;
  const float* sb;
  int sa_ld, sb_ld;
  WaitCtl w;
  QuantState cst;  // scaling state of the FP8 output (QF >= 0)
};

__device__ __forceinline__ void tile_coords(int t, const KParams& p, int& mb, int& nb) {
  const int per_group = GROUP_M * p.num_n;
  const int g = t / per_group;
  const int first_m = g * GROUP_M;
  const int gsize = min(GROUP_M, p.num_m - first_m);
  const int local = t - g * per_group;
  mb = first_m + local % gsize;
  nb = local / gsize;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Wait that ignores the error word (used only to drain work already issued).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Stage 32 rows x 64 bf16 (this lane's row = 32 packed words) into a 128-byte-swizzled
// buffer and store it with TMA at (c0, r0). Called by all 32 lanes of the warp.
__device__ __forceinline__ void stage_and_store(uint8_t* stg, const uint32_t (&pk)[32], int lane,
                                                const CUtensorMap* tmC, int c0, int r0) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) * 16)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, smem_u32(stg), c0, r0);
    bulk_commit_group();
  }
}

template <bool BLOCK, int BN, int QF>
__global__ void __launch_bounds__(Cfg<BLOCK, BN, QF>::THREADS, 1)
    gemm_f8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmQ,
                   const KParams p) {
  using C = Cfg<BLOCK, BN, QF>;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = C::TMEM_COLS;
  constexpr int ACC = C::ACC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;
  const uint32_t bar_tempty = bar_tfull + 8 * ACC;
  const uint32_t bar_final = bar_tempty + 8 * ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  if (threadIdx.x == 0) FP8GB_STAMP(0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, C::EPI_WARPS);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above overlaps the previous kernel; operands and scales are read after it
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) FP8GB_STAMP(1);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;  // per stage: issued?, parity of last issue
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.w, DEV_ERR_WAIT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
#ifdef FP8GB_TRACE
          if (t == (int)blockIdx.x && kb == 0) FP8GB_STAMP(7);
#endif
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          tma_load_2d(sa, &tmA, fb, kb * BK, mb * BM);
          tma_load_2d(sa + A_BYTES, &tmB, fb, kb * BK, nb * BN);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every load already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) mbar_wait_drain(bar_full + 8 * s, (issued_phase >> s) & 1u, 1000000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!BLOCK) {
          if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, p.w, DEV_ERR_WAIT_MMA)) break;
          tc_fence_after();
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (BLOCK) {
            if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, p.w, DEV_ERR_WAIT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(bar_full + 8 * stage, phase, p.w, DEV_ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
#ifdef FP8GB_TRACE
          if (t == (int)blockIdx.x && kb == 0) FP8GB_STAMP(2);
#endif
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            const uint32_t accumulate = BLOCK ? (k != 0) : ((kb | k) != 0);
            mma_f8(d, adesc + 2 * k, bdesc + 2 * k, p.idesc, accumulate);
          }
          mma_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (BLOCK) {
            mma_commit(bar_tfull + 8 * acc);
            acc = (acc + 1 == ACC) ? 0 : acc + 1;
            if (acc == 0) acc_phase ^= 1u;
          }
        }
        if (!BLOCK && ok) {
          mma_commit(bar_tfull + 8 * acc);
          acc = (acc + 1 == ACC) ? 0 : acc + 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      FP8GB_STAMP(3);
      // every MMA this thread issued has completed once this barrier flips
      mma_commit(bar_final);
      if (!mbar_wait_drain(bar_final, 0, 1000000000ull)) atomicOr(p.w.err, DEV_ERR_WAIT_TEARDOWN);
      FP8GB_STAMP(4);
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp - 2;             // 0 .. EPI_WARPS-1
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* stg = smem + C::OFF_STG + ew * C::STG_PER_WARP * STG_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    if constexpr (!BLOCK) {
      const float dd = __fmul_rn(__ldg(p.sa), __ldg(p.sb));
      // FP8 output: with a non-empty history the epilogue casts the bf16 result with the
      // delayed scale (the empty-history call is cast afterwards from its own amax)
      bool fused = false;
      castops::Scaler qsc{};
      uint32_t qov = 0, qun = 0, qam = 0;
      uint8_t* qstg = smem + C::OFF_QSTG + ew * C::QSTG_PER_WARP;
      if constexpr (QF >= 0) {
        fused = *p.cst.hist_count > 0;
        if (fused) {
          float s, d;
          castops::scales_from_amax(castops::effective_amax(p.cst, true), castops::Fmt<QF>::kMax, s, d);
          qsc = castops::make_scaler<QF>(s, d);
          if (blockIdx.x == 0 && ew == 0 && lane == 0) {
            *p.cst.scale = s;
            *p.cst.scale_inv = d;
          }
        }
      }
      // the tile's 64-column chunks alternate between the two warps of a lane quarter
      const int hc = ew >> 2;
      constexpr int NCH = BN / 64;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, p.w, DEV_ERR_WAIT_EPILOGUE)) break;
        __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the spin
        tc_fence_after();
#pragma unroll 1
        for (int ch = hc; ch < NCH; ch += 2) {
          __syncwarp();
          uint32_t r0[32], r1[32];
          const int col = ch * 64;
          const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + col);
          tmem_ld32(taddr, r0);
          tmem_ld32(taddr + 32, r1);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          if (ch + 2 >= NCH) {  // this warp's part of the accumulator is read: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
          }
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            pk[j] = pack_bf16x2(__fmul_rn(__uint_as_float(r0[2 * j]), dd), __fmul_rn(__uint_as_float(r0[2 * j + 1]), dd));
            pk[16 + j] =
                pack_bf16x2(__fmul_rn(__uint_as_float(r1[2 * j]), dd), __fmul_rn(__uint_as_float(r1[2 * j + 1]), dd));
          }
          if (lane == 0) bulk_wait_group_read<0>();  // the previous stores have read the staging buffers
          __syncwarp();
          if constexpr (QF >= 0) {
            if (fused) {
              // 64 codes of this lane's row, staged with the 64-byte swizzle: 16-byte chunk j
              // of row r sits at chunk j ^ ((r / 2) % 4)
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint2 c0 = castops::cast8<QF, true>(make_uint4(pk[8 * j], pk[8 * j + 1], pk[8 * j + 2], pk[8 * j + 3]),
                                                          qsc, qov, qun, qam);
                const uint2 c1 = castops::cast8<QF, true>(
                    make_uint4(pk[8 * j + 4], pk[8 * j + 5], pk[8 * j + 6], pk[8 * j + 7]), qsc, qov, qun, qam);
                *reinterpret_cast<uint4*>(qstg + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) =
                    make_uint4(c0.x, c0.y, c1.x, c1.y);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, smem_u32(stg), nb * BN + col, mb * BM + q * 32);
            if (fused) tma_store_2d(&tmQ, smem_u32(qstg), nb * BN + col, mb * BM + q * 32);
            bulk_commit_group();
          }
        }
        acc = (acc + 1 == ACC) ? 0 : acc + 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (fused) {  // this warp's share of the output's counters and amax
        qov = __reduce_add_sync(0xFFFFFFFFu, qov);
        qun = __reduce_add_sync(0xFFFFFFFFu, qun);
        qam = __reduce_max_sync(0xFFFFFFFFu, castops::fold2(qam));
        if (lane == 0) {
          if (qov) atomicAdd(p.cst.counters + 0, static_cast<unsigned long long>(qov));
          if (qun) atomicAdd(p.cst.counters + 1, static_cast<unsigned long long>(qun));
          castops::atomic_max_amax(p.cst.amax_cur, qam);
        }
      }
    } else {
      // each warp folds 64 columns (one 128-column scale block = BN / 128 ... of them) of its
      // TMEM lane quarter: two x32 loads issued back to back, one wait, 64 FMAs
      const int col0 = (ew >> 2) * 64;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        const int row = mb * BM + q * 32 + lane;
        const int nblk = (nb * BN + col0) / 128;
        const bool row_ok = row < p.M;
        const bool col_ok = nblk * 128 < p.N;
        float accum[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) accum[j] = 0.0f;
        float sa_next = row_ok ? __ldg(p.sa + (int64_t)row * p.sa_ld) : 0.0f;
        float sb_next = col_ok ? __ldg(p.sb + nblk) : 0.0f;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          const float sc = __fmul_rn(sa_next, sb_next);
          if (kb + 1 < p.num_kb) {
            sa_next = row_ok ? __ldg(p.sa + (int64_t)row * p.sa_ld + kb + 1) : 0.0f;
            sb_next = col_ok ? __ldg(p.sb + (int64_t)(kb + 1) * p.sb_ld + nblk) : 0.0f;
          }
          if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, p.w, DEV_ERR_WAIT_EPILOGUE)) {
            ok = false;
            break;
          }
          __syncwarp();
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + col0);
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr, r0);
          tmem_ld32(taddr + 32, r1);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);  // registers hold the block now
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            accum[j] = fmaf(__uint_as_float(r0[j]), sc, accum[j]);
            accum[32 + j] = fmaf(__uint_as_float(r1[j]), sc, accum[32 + j]);
          }
          acc = (acc + 1 == ACC) ? 0 : acc + 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) break;
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(accum[2 * j], accum[2 * j + 1]);
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        stage_and_store(stg, pk, lane, &tmC, nb * BN + col0, mb * BM + q * 32);
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    if (warp == 2 && lane == 0) FP8GB_STAMP(5);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) FP8GB_STAMP(6);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_tmap_2d(m, base, dt, inner, outer, row_bytes, box_inner, box_outer, 128);
}

template <bool BLOCK, int BN, int QF>
cudaError_t prepare_kernel() {
  // the attribute is per device; remember which devices were configured
  static bool done[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_f8_kernel<BLOCK, BN, QF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<BLOCK, BN, QF>::SMEM);
  if (e == cudaSuccess && dev < 64) done[dev] = true;
  return e;
}

// Tile width: cost = rounds of tiles over the SMs x time of one tile (width / mainloop
// efficiency). Narrower tiles move more operand bytes per FLOP: measured on GB300 the
// mainloop runs at ~94 % of the tensor peak with 256-wide tiles, ~80 % with 192-wide and
// ~60 % with 128-wide ones. Narrower tiles win only when they save rounds.
int choose_bn(int64_t M, int64_t N, int sms) {
  const int64_t tm = (M + BM - 1) / BM;
  const int widths[3] = {256, 192, 128};
  const int per_round[3] = {272, 240, 213};  // width / efficiency
  int best = 256;
  int64_t best_cost = -1;
  for (int i = 0; i < 3; ++i) {
    const int64_t rounds = (tm * ((N + widths[i] - 1) / widths[i]) + sms - 1) / sms;
    const int64_t cost = rounds * per_round[i];
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = widths[i];
    }
  }
  return best;
}

template <bool BLOCK, int BN, int QF>
cudaError_t launch_variant(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tq,
                           KParams p, cudaStream_t stream) {
  cudaError_t e = prepare_kernel<BLOCK, BN, QF>();
  if (e != cudaSuccess) return e;
  p.num_n = (p.N + BN - 1) / BN;
  p.num_tiles = p.num_m * p.num_n;
  p.idesc = idesc_f8(p.idesc & 7u, (p.idesc >> 3) & 7u, BM, BN);
  const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
  return launch_pdl(gemm_f8_kernel<BLOCK, BN, QF>, dim3(grid), dim3(Cfg<BLOCK, BN, QF>::THREADS),
                    Cfg<BLOCK, BN, QF>::SMEM, stream, ta, tb, tc, tq, p);
}

template <int QF>
cudaError_t launch_width(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const CUtensorMap& tq, const KParams& p, cudaStream_t stream) {
  if (bn == 256) return launch_variant<false, 256, QF>(ta, tb, tc, tq, p, stream);
  if (bn == 192) return launch_variant<false, 192, QF>(ta, tb, tc, tq, p, stream);
  return launch_variant<false, 128, QF>(ta, tb, tc, tq, p, stream);
}

}  // namespace

bool encode_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream, const char** why) {
  // block scaling folds every 128-deep K block out of TMEM: 128-wide tiles keep the fold's
  // registers (64 fp32 per thread) and its four accumulator buffers within budget
#ifdef FP8GB_FORCE_BN  // compile-time override of the tile-width heuristic, for tuning builds
  const int bn = g.block_scaled ? 128 : FP8GB_FORCE_BN;
#else
  const int bn = g.block_scaled ? 128 : choose_bn(g.M, g.N, num_sms());
#endif
  CUtensorMap ta, tb, tc;
  if (!make_map(&ta, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K, g.M, g.lda, BK, BM) ||
      !make_map(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K, g.N, g.ldb, BK, bn) ||
      !make_map(&tc, g.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.N, g.M, g.ldc * 2, 64, 32)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point missing or tensor map rejected)";
    return cudaErrorInvalidValue;
  }
  KParams p{};
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.num_m = static_cast<int>((g.M + BM - 1) / BM);
  p.num_kb = static_cast<int>((g.K + BK - 1) / BK);
  p.idesc = static_cast<uint32_t>(g.fa) | (static_cast<uint32_t>(g.fb) << 3);  // formats; finished per variant
  p.sa = g.sa;
  p.sb = g.sb;
  p.sa_ld = static_cast<int>(g.K / 128);
  p.sb_ld = static_cast<int>(g.N / 128);
  p.w = wait_ctl();
  if (p.w.err == nullptr) {
    *why = "device error word unavailable";
    return cudaErrorInvalidDevice;
  }
  CUtensorMap tq = tc;  // unused unless the epilogue also writes FP8 codes
  if (g.qf >= 0) {
    if (!encode_tmap_2d(&tq, g.Cq, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.N, g.M, g.ldcq, 64, 32, 64)) {
      *why = "cuTensorMapEncodeTiled failed for the FP8 output";
      return cudaErrorInvalidValue;
    }
    p.cst = g.cst;
  }
  if (g.block_scaled) return launch_variant<true, 128, -1>(ta, tb, tc, tq, p, stream);
  if (g.qf == 0) return launch_width<0>(bn, ta, tb, tc, tq, p, stream);
  if (g.qf == 1) return launch_width<1>(bn, ta, tb, tc, tq, p, stream);
  return launch_width<-1>(bn, ta, tb, tc, tq, p, stream);
}

}  // namespace fp8gb
