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
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      one thread issues TMA loads of A [128 x 128] and B [BN x 128] (K-major,
//               128-byte swizzle) into a shared-memory ring;
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma (M=128, N=BN,
//               K=32) into a TMEM accumulator and frees ring slots with tcgen05.commit;
//   warps 2..   epilogue: tcgen05.ld of the accumulator (each warp owns the 32 TMEM lanes
//               its warp index selects), multiply by the scales, convert to bf16, stage
//               128-byte rows through swizzled shared memory and write them with TMA.
// Per tensor: two 256-column accumulators, so the epilogue of one tile overlaps the
// mainloop of the next; each epilogue warp reads all of its columns before handing the
// accumulator back. A CTA takes in operands at ~140 GB/s on GB300, which caps a
// 128 x 256 tile at ~80 % of the tensor peak; with more than 128 rows the per-tensor GEMM
// therefore runs on CTA pairs (clusters of two, tcgen05 cta_group::2): the pair computes a
// 256 x BN tile, each CTA loads its own 128 rows of A and half of B's BN rows, the even
// CTA issues the MMAs, and both CTAs drain their half of the accumulator.
// Block scaled (gemm_blk_kernel): every 128-deep K block gets a fresh accumulator buffer
// (two of 256 columns, alternating), and 8 fold warps multiply it by its scale product and
// add it into fp32 registers.
// Every mbarrier wait is bounded (see ptx.cuh); on a timeout the CTA stops issuing work,
// drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <array>
#include <map>
#include <mutex>
#include <vector>

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
// Tile raster: groups of `group_m` row blocks sweep the column blocks together, so a B tile
// is read by the group's CTAs from L2 and B is read from DRAM once per group.

// Tile 128 x BN per CTA (BN = 256, 192 or 128); the ring depth fills ~192 KB of shared
// memory, less when the epilogue also stages FP8 output (QF >= 0: 0 = E4M3, 1 = E5M2).
// PAIR: two CTAs of a cluster share one 256 x BN tile through the CTA-pair MMA; each holds
// its 128 rows of A and half of B's BN rows, so a CTA loads 16 KB + BN * 64 bytes per
// 128-deep K block instead of 16 KB + BN * 128 for the same tensor work.
// MX: block-scaled MMAs (kind::mxf8f6f4) with UE8M0 scales per 32 K of every row of A and B;
// each stage also holds the K block's scale atoms (512 bytes per 128 rows of A or of B),
// which the MMA issuer copies into TMEM columns after the accumulators.
template <int BN, int QF, bool PAIR = false, bool MX = false>
struct Cfg {
  static_assert(BN == 128 || BN == 192 || BN == 256, "tile width");
  static_assert(!MX || (QF < 0 && BN != 192 && (!PAIR || BN == 256)), "MX: tiles of whole scale atoms, bf16 out");
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // B rows this CTA loads per stage
  static constexpr int B_BYTES = B_ROWS * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SFB_ATOMS = MX ? (BN + 127) / 128 : 0;
  static constexpr int SF_BYTES = MX ? 512 * (1 + SFB_ATOMS) : 0;  // scale atoms of A and B per stage
  // two warps per TMEM lane quarter, each draining half of the tile's columns
  static constexpr int EPI_WARPS = 8;
  static constexpr int QSTG_PER_WARP = QF >= 0 ? QSTG_BYTES : 0;
  // bf16 staging per epilogue warp: 32 rows x 64 columns (128-byte swizzle), or with MX
  // 32 x 32 (64-byte swizzle), which leaves shared memory for a fourth 256-wide stage
  static constexpr int STG = MX ? STG_BYTES / 2 : STG_BYTES;
  static constexpr int STAGES_FIT = (230000 - EPI_WARPS * (STG + QSTG_PER_WARP)) / (STAGE_BYTES + SF_BYTES);
  static constexpr int STAGES = STAGES_FIT < (192 * 1024) / STAGE_BYTES ? STAGES_FIT : (192 * 1024) / STAGE_BYTES;
  // TMEM: ACC accumulator buffers, then (MX) the K block's scale columns: 4 of A's scales and
  // 4 per atom of B's
  static constexpr int SF_COLS = MX ? 4 * (1 + SFB_ATOMS) : 0;
  static constexpr int ACC = (512 - SF_COLS) / BN;
  static constexpr int SFA_COL = ACC * BN;
  static_assert(!MX || SFA_COL + SF_COLS <= 512, "TMEM columns");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int STG_PER_WARP = 1;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int OFF_SF = STAGES * STAGE_BYTES;
  // the staging buffers start on a 1024-byte boundary: the TMA store applies the swizzle from
  // the shared-memory address bits, so a buffer 512 bytes off would have its 16-byte chunks
  // read from the wrong positions (columns 0-31 and 32-63 of a 64-column store exchanged)
  static constexpr int OFF_STG = (OFF_SF + STAGES * SF_BYTES + 1023) & ~1023;
  static constexpr int OFF_QSTG = OFF_STG + EPI_WARPS * STG_PER_WARP * STG;
  static constexpr int OFF_BAR = OFF_QSTG + EPI_WARPS * QSTG_PER_WARP;
  // full[S], empty[S], tfull[ACC], tempty[ACC], final
  static constexpr int NBAR = 2 * STAGES + 2 * ACC + 1;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_TMEM_SLOT + 16 + 1024;  // + alignment slack
  // arrivals that free an accumulator: every epilogue warp of the tile's CTAs
  static constexpr int TEMPTY_COUNT = (PAIR ? 2 : 1) * EPI_WARPS;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert((A_BYTES % 1024) == 0 && (B_BYTES % 1024) == 0, "stage halves on 1024-byte swizzle atoms");
  static_assert(OFF_STG % 1024 == 0 && STG % 1024 == 0 && OFF_QSTG % 512 == 0, "staging on swizzle atoms");
};

// floor(n / d) for 0 <= n < 2^31 and 1 <= d < 2^31 as (n * m) >> (32 + s), with
// s = ceil(log2 d) and m = floor(2^(32+s) / d) + 1 (division by invariant integers using
// multiplication, Granlund and Montgomery, 1994): m = (2^(32+s) + e) / d with 0 < e <= d, so
// n m / 2^(32+s) exceeds n / d by less than n / 2^(32+s) < 1 / (2 d), which never reaches the
// next integer. The work-unit mapping runs at every tile and first at each CTA's start, where
// five integer divisions (a long dependent sequence each) cost ~0.5 us before the first load.
struct DivBy {
  uint64_t m;
  uint32_t s;
};

inline DivBy make_div(uint32_t d) {
  DivBy r{0, 0};
  if (d == 0) return r;
  while ((uint64_t(1) << r.s) < d) ++r.s;
  r.m = ((uint64_t(1) << (32 + r.s)) / d) + 1;
  return r;
}

__host__ __device__ __forceinline__ uint32_t div_by(uint32_t n, const DivBy& d) {
  return static_cast<uint32_t>((static_cast<uint64_t>(n) * d.m) >> (32 + d.s));
}

// One GEMM problem of a launch. A launch runs one problem, or two independent ones (the
// backward pass's dgrad and wgrad) whose work units share the persistent grid.
struct KProb {
  int M, N, K;
  int num_m, num_n, num_kb, num_tiles;  // num_m counts 256-row tiles on CTA pairs
  uint32_t idesc;
  const float* sa;
  const float* sb;
  int sa_ld, sb_ld;
  // split K: each output tile is `splits` (1 or 2) work units over the two halves of its
  // K blocks; the last unit of a tile to finish adds the other's fp32 partial (ws) to its own.
  // ws_cnt holds one arrival counter per (tile, CTA rank, epilogue warp), zero between calls.
  int splits;
  float4* ws;
  int* ws_cnt;
  int unit0;  // first work unit of this problem in the launch
  // MX: UE8M0 scale atoms of A ([num 128-row blocks][K / 128] x 512 bytes) and of B
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sf_nkb, sfb_atoms;  // K / 128, atoms along N (ceil(N / 128))
  // operands stored contraction-major (A as [K, M], B as [K, N], row-major) and read MN-major
  // by the tensor cores: tiles arrive as boxes of 128 MN x 128 K
  int mn;
  // K blocks of a tile's first split unit (num_kb / 2; unused without split K)
  int kb_half;
  // the tile raster's divisors as multipliers (see DivBy): tiles per raster group, rows of a
  // group, rows of the last (shorter) group
  DivBy div_group, div_gm, div_glast;
};

constexpr int kMaxSlots = 160;         // CTAs (or CTA pairs) of a persistent grid
constexpr int kMaxSchedUnits = 1024;   // units of an explicit schedule

struct KParams {
  KProb pr[2];
  int nprob;  // 1 or 2
  int group_m;  // row blocks per raster group
  int units;  // work units of all problems
  WaitCtl w;
  QuantState cst;  // scaling state of the FP8 output (QF >= 0, one problem)
  // Units of CTA (pair) slot s: sched_unit[sched_off[s] .. sched_off[s + 1]) when sched_len
  // > 0 (units of unequal length, placed longest first on the least-loaded slot); otherwise
  // slot s takes units s, s + slots, s + 2 slots, ...
  int sched_len;
  uint16_t sched_off[kMaxSlots + 1];
  uint16_t sched_unit[kMaxSchedUnits];
  DivBy div_slots;  // the grid's CTA (pair) slots
};

__device__ __forceinline__ int slot_units(const KParams& p, int slot, int slots) {
  if (p.sched_len > 0) return p.sched_off[slot + 1] - p.sched_off[slot];
  return slot < p.units ? static_cast<int>(div_by(static_cast<uint32_t>(p.units - slot + slots - 1), p.div_slots)) : 0;
}

__device__ __forceinline__ int slot_unit(const KParams& p, int slot, int slots, int i) {
  return p.sched_len > 0 ? p.sched_unit[p.sched_off[slot] + i] : slot + i * slots;
}

// Problem pi's fields, selected field by field (no dynamic indexing of kernel parameters).
__device__ __forceinline__ KProb prob_of(const KParams& p, int pi) {
  const KProb& a = p.pr[0];
  const KProb& b = p.pr[1];
  KProb q;
  q.M = pi ? b.M : a.M;
  q.N = pi ? b.N : a.N;
  q.K = pi ? b.K : a.K;
  q.num_m = pi ? b.num_m : a.num_m;
  q.num_n = pi ? b.num_n : a.num_n;
  q.num_kb = pi ? b.num_kb : a.num_kb;
  q.num_tiles = pi ? b.num_tiles : a.num_tiles;
  q.idesc = pi ? b.idesc : a.idesc;
  q.sa = pi ? b.sa : a.sa;
  q.sb = pi ? b.sb : a.sb;
  q.sa_ld = pi ? b.sa_ld : a.sa_ld;
  q.sb_ld = pi ? b.sb_ld : a.sb_ld;
  q.splits = pi ? b.splits : a.splits;
  q.ws = pi ? b.ws : a.ws;
  q.ws_cnt = pi ? b.ws_cnt : a.ws_cnt;
  q.unit0 = pi ? b.unit0 : a.unit0;
  q.sfa = pi ? b.sfa : a.sfa;
  q.sfb = pi ? b.sfb : a.sfb;
  q.sf_nkb = pi ? b.sf_nkb : a.sf_nkb;
  q.sfb_atoms = pi ? b.sfb_atoms : a.sfb_atoms;
  q.mn = pi ? b.mn : a.mn;
  q.kb_half = pi ? b.kb_half : a.kb_half;
  q.div_group = pi ? b.div_group : a.div_group;
  q.div_gm = pi ? b.div_gm : a.div_gm;
  q.div_glast = pi ? b.div_glast : a.div_glast;
  return q;
}

__device__ __forceinline__ void tile_coords(int t, const KProb& q, int group_m, int& mb, int& nb) {
  const int g = static_cast<int>(div_by(static_cast<uint32_t>(t), q.div_group));
  const int first_m = g * group_m;
  const bool last = q.num_m - first_m < group_m;  // the last group may hold fewer row blocks
  const int gsize = last ? q.num_m - first_m : group_m;
  const int local = t - g * group_m * q.num_n;
  nb = static_cast<int>(div_by(static_cast<uint32_t>(local), last ? q.div_glast : q.div_gm));
  mb = first_m + (local - nb * gsize);
}

// Work unit u of the launch -> its problem, output tile (row and column block), split and
// K-block range [kb0, kb1).
struct Unit {
  int pi, t, split, kb0, kb1, mb, nb;
};

__device__ __forceinline__ Unit unit_at(int u, const KParams& p, KProb& q) {
  Unit r;
  r.pi = (p.nprob > 1 && u >= p.pr[1].unit0) ? 1 : 0;
  q = prob_of(p, r.pi);
  const int v = u - q.unit0;
  // one or two units per tile; with two, the first takes K blocks [0, num_kb / 2)
  r.t = q.splits > 1 ? v >> 1 : v;
  r.split = v - r.t * q.splits;
  r.kb0 = r.split ? q.kb_half : 0;
  r.kb1 = (q.splits > 1 && r.split == 0) ? q.kb_half : q.num_kb;
  tile_coords(r.t, q, p.group_m, r.mb, r.nb);
  return r;
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

template <int BN, int QF, bool PAIR, bool MX>
__global__ void __launch_bounds__(Cfg<BN, QF, PAIR, MX>::THREADS, 1)
    gemm_f8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ KParams p) {
  using C = Cfg<BN, QF, PAIR, MX>;
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
  // CTA pairs: rank 0 issues the MMAs and owns the stage-full and accumulator-empty
  // barriers both CTAs signal; tiles are 256 rows (rank r holds rows 128 r .. 128 r + 127)
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  constexpr int TILE_M = PAIR ? 2 * BM : BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, C::TEMPTY_COUNT);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (p.nprob > 1 || (MX && PAIR)) {  // (MX pairs: A's and B's scale maps)
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
      tma_prefetch_desc(&tmC1);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers are initialised
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
      const uint32_t full_lead = PAIR ? mapa_shared(bar_full, 0) : bar_full;
      const int nmine = slot_units(p, tile0, tile_step);
      for (int i = 0; ok && i < nmine; ++i) {
        const int u = slot_unit(p, tile0, tile_step, i);
        KProb q;
        const Unit un = unit_at(u, p, q);
        const CUtensorMap* tA = un.pi ? &tmA1 : &tmA;
        const CUtensorMap* tB = un.pi ? &tmB1 : &tmB;
        const int arow = un.mb * TILE_M + static_cast<int>(rank) * BM;
        const int brow = un.nb * BN + static_cast<int>(rank) * C::B_ROWS;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.w, DEV_ERR_WAIT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
#ifdef FP8GB_TRACE
          if (i == 0 && kb == un.kb0) FP8GB_STAMP(7);
#endif
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          if constexpr (PAIR && MX) {
            // both CTAs' operand and scale bytes land on rank 0's barrier; each CTA holds its
            // own 128 rows of A's scales and the scales of all the tile's columns of B (its
            // tensor core computes every column of the tile); the scale atoms come through
            // tensor maps (tmA1: A's atoms as rows of 512 bytes; tmB1: B's, [atom][kb][512 B])
            const uint32_t sfs = sbase + C::OFF_SF + stage * C::SF_BYTES;
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (STAGE_BYTES + C::SF_BYTES));
            tma_load_2d_pair(sa, tA, full_lead + 8 * stage, kb * BK, arow);
            tma_load_2d_pair(sa + A_BYTES, tB, full_lead + 8 * stage, kb * BK, brow);
            tma_load_2d_pair(sfs, &tmA1, full_lead + 8 * stage, 0, (arow / BM) * p.pr[0].sf_nkb + kb);
            tma_load_3d_pair(sfs + 512, &tmB1, full_lead + 8 * stage, 0, kb, un.nb * C::SFB_ATOMS);
          } else if constexpr (PAIR) {
            // both CTAs' bytes land on rank 0's barrier, which alone expects them
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * STAGE_BYTES);
            if (q.mn) {  // (a CTA's half of B is one 128-column box)
              tma_load_2d_pair(sa, tA, full_lead + 8 * stage, arow, kb * BK);
              tma_load_2d_pair(sa + A_BYTES, tB, full_lead + 8 * stage, brow, kb * BK);
            } else {
              tma_load_2d_pair(sa, tA, full_lead + 8 * stage, kb * BK, arow);
              tma_load_2d_pair(sa + A_BYTES, tB, full_lead + 8 * stage, kb * BK, brow);
            }
          } else if constexpr (MX) {
            // the K block's scale atoms: A's for this tile's 128 rows, B's for its BN columns
            // (atoms past the last column of B are not loaded; their columns are not stored)
            const int a0 = un.nb * (BN / 128);
            const int nba = min(C::SFB_ATOMS, q.sfb_atoms - a0);
            const uint32_t sfs = sbase + C::OFF_SF + stage * C::SF_BYTES;
            mbar_arrive_expect_tx(fb, STAGE_BYTES + 512u * static_cast<uint32_t>(1 + nba));
            tma_load_2d(sa, tA, fb, kb * BK, arow);
            tma_load_2d(sa + A_BYTES, tB, fb, kb * BK, brow);
            bulk_load(sfs, q.sfa + (static_cast<int64_t>(un.mb) * q.sf_nkb + kb) * 512, 512, fb);
            for (int a = 0; a < nba; ++a)
              bulk_load(sfs + 512 * (1 + a), q.sfb + (static_cast<int64_t>(a0 + a) * q.sf_nkb + kb) * 512, 512, fb);
          } else {
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            if (q.mn) {
              tma_load_2d(sa, tA, fb, arow, kb * BK);
#pragma unroll
              for (int h = 0; h < C::B_ROWS / 128; ++h)
                tma_load_2d(sa + A_BYTES + h * (128 * BK), tB, fb, brow + 128 * h, kb * BK);
            } else {
              tma_load_2d(sa, tA, fb, kb * BK, arow);
              tma_load_2d(sa + A_BYTES, tB, fb, kb * BK, brow);
            }
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every load already issued land before the CTA exits
        if constexpr (PAIR) {
          // the loads signal rank 0's barriers, which may also wait for the peer's bytes:
          // give them a fixed 200 us (a TMA load lands in microseconds)
          const unsigned long long t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        } else {
          for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s)) mbar_wait_drain(bar_full + 8 * s, (issued_phase >> s) & 1u, 1000000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer ----------------
      auto wait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, p.w, DEV_ERR_WAIT_MMA); };
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const int nmine = slot_units(p, tile0, tile_step);
      // MX: a stage's scale atoms into TMEM (a CTA pair's copy moves each CTA's shared memory
      // into its own tensor memory). The copies and the MMAs after them execute in issue order;
      // measured, they cost ~80 ns of tensor-pipe time per K block (the MMAs alone ran the
      // 16384 x 14336 x 4096 GEMM in 0.48 ms), and issuing them one block ahead into a second
      // slot, or from a second thread, made it slower
      auto copy_scales = [&](int st) {
        const uint32_t sfs = sbase + C::OFF_SF + st * C::SF_BYTES;
        const uint32_t col = tmem_base + C::SFA_COL;
        if constexpr (PAIR) {
          tmem_cp_32x128b_x4_pair(col, smem_desc_plain128(sfs));
#pragma unroll
          for (int a = 0; a < C::SFB_ATOMS; ++a) tmem_cp_32x128b_x4_pair(col + 4 + 4 * a, smem_desc_plain128(sfs + 512 * (1 + a)));
        } else {
          tmem_cp_32x128b_x4(col, smem_desc_plain128(sfs));
#pragma unroll
          for (int a = 0; a < C::SFB_ATOMS; ++a) tmem_cp_32x128b_x4(col + 4 + 4 * a, smem_desc_plain128(sfs + 512 * (1 + a)));
        }
      };
      for (int i = 0; ok && i < nmine; ++i) {
        const int u = slot_unit(p, tile0, tile_step, i);
        KProb q;
        const Unit un = unit_at(u, p, q);
        const int kb0 = un.kb0, kb1 = un.kb1;
        if (!wait(bar_tempty + 8 * acc, acc_phase ^ 1u)) break;
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait(bar_full + 8 * stage, phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
#ifdef FP8GB_TRACE
          if (i == 0 && kb == kb0) FP8GB_STAMP(2);
#endif
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          // K-major: a 32-deep step is 32 bytes along each row; MN-major: 32 rows of 128 bytes
          const uint64_t adesc = q.mn ? smem_desc_sw128_mn(sa) : smem_desc_sw128(sa);
          const uint64_t bdesc = q.mn ? smem_desc_sw128_mn(sa + A_BYTES) : smem_desc_sw128(sa + A_BYTES);
          const uint64_t kstep = q.mn ? (32 * 128) >> 4 : 32 >> 4;
          if constexpr (MX) {
            // the block's scales, then four MMAs of 32 K, each taking byte k of every row's
            // scale word
            copy_scales(stage);
            const uint32_t sfa = tmem_base + C::SFA_COL, sfb = sfa + 4;
            if constexpr (PAIR) {
#pragma unroll
              for (int k = 0; k < BK / 32; ++k)
                mma_mxf8_pair(d, adesc + 2 * k, bdesc + 2 * k, q.idesc | idesc_sf_ids(k, k), sfa, sfb,
                              (kb != kb0 || k != 0));
              mma_commit_pair(bar_empty + 8 * stage, 0x3);
            } else {
#pragma unroll
              for (int k = 0; k < BK / 32; ++k)
                mma_mxf8(d, adesc + 2 * k, bdesc + 2 * k, q.idesc | idesc_sf_ids(k, k), sfa, sfb, (kb != kb0 || k != 0));
              mma_commit(bar_empty + 8 * stage);
            }
          } else {
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              const uint32_t accumulate = (kb != kb0 || k != 0);
              if constexpr (PAIR)
                mma_f8_pair(d, adesc + kstep * k, bdesc + kstep * k, q.idesc, accumulate);
              else
                mma_f8(d, adesc + kstep * k, bdesc + kstep * k, q.idesc, accumulate);
            }
            if constexpr (PAIR)
              mma_commit_pair(bar_empty + 8 * stage, 0x3);  // frees the stage in both CTAs
            else
              mma_commit(bar_empty + 8 * stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) {
          if constexpr (PAIR)
            mma_commit_pair(bar_tfull + 8 * acc, 0x3);  // both halves of the tile are ready
          else
            mma_commit(bar_tfull + 8 * acc);
          acc = (acc + 1 == ACC) ? 0 : acc + 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      FP8GB_STAMP(3);
      // every MMA this thread issued has completed once this barrier flips
      if constexpr (PAIR)
        mma_commit_pair(bar_final, 0x1);
      else
        mma_commit(bar_final);
      if (!mbar_wait_drain(bar_final, 0, 1000000000ull)) atomicOr(p.w.err, DEV_ERR_WAIT_TEARDOWN);
      FP8GB_STAMP(4);
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp - 2;             // 0 .. EPI_WARPS-1
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* stg = smem + C::OFF_STG + ew * C::STG_PER_WARP * C::STG;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    {
      // (MX: the MMAs applied the scales)
      const float dd0 = MX ? 1.0f : __fmul_rn(__ldg(p.pr[0].sa), __ldg(p.pr[0].sb));
      const float dd1 = (!MX && p.nprob > 1) ? __fmul_rn(__ldg(p.pr[1].sa), __ldg(p.pr[1].sb)) : dd0;
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
      const uint32_t tempty_lead = PAIR ? mapa_shared(bar_tempty, 0) : bar_tempty;
      const int nmine = slot_units(p, tile0, tile_step);
      for (int i = 0; ok && i < nmine; ++i) {
        const int u = slot_unit(p, tile0, tile_step, i);
        KProb pq;
        const Unit un = unit_at(u, p, pq);
        const int t = un.t, split = un.split, mb = un.mb, nb = un.nb;
        const float dd = un.pi ? dd1 : dd0;
        const CUtensorMap* tC = un.pi ? &tmC1 : &tmC;
        const int row0 = mb * TILE_M + static_cast<int>(rank) * BM + q * 32;  // this warp's 32 rows
        const bool rows_live = row0 < pq.M;
        if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, p.w, DEV_ERR_WAIT_EPILOGUE)) break;
        __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the spin
        tc_fence_after();
        // both of this warp's chunks (64 columns each) are read before the accumulator is
        // handed back, so the next tile's MMAs do not wait for this tile's stores
        const bool two = NCH > 2 && hc + 2 < NCH;
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + hc * 64);
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        if (two) {
          tmem_ld32(taddr + 128, r2);
          tmem_ld32(taddr + 160, r3);
        }
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        reg_fence(r2);
        reg_fence(r3);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(tempty_lead + 8 * acc);
          else
            mbar_arrive(bar_tempty + 8 * acc);
        }
        // scale, convert to bf16 (and FP8 when fused), stage and store one 64-column chunk
        auto emit = [&](const uint32_t(&ra)[32], const uint32_t(&rb)[32], int col) {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            pk[j] = pack_bf16x2(__fmul_rn(__uint_as_float(ra[2 * j]), dd), __fmul_rn(__uint_as_float(ra[2 * j + 1]), dd));
            pk[16 + j] =
                pack_bf16x2(__fmul_rn(__uint_as_float(rb[2 * j]), dd), __fmul_rn(__uint_as_float(rb[2 * j + 1]), dd));
          }
          if constexpr (MX) {
            // two stores of 32 columns through the half-size buffer: 16-byte chunk j of row r
            // sits at chunk j ^ ((r / 2) % 4) (64-byte swizzle)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) =
                    make_uint4(pk[16 * h + 4 * j], pk[16 * h + 4 * j + 1], pk[16 * h + 4 * j + 2], pk[16 * h + 4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0 && rows_live) {
                tma_store_2d(tC, smem_u32(stg), nb * BN + col + 32 * h, row0);
                bulk_commit_group();
              }
            }
            return;
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
          if (lane == 0 && rows_live) {
            tma_store_2d(tC, smem_u32(stg), nb * BN + col, row0);
            if (fused) tma_store_2d(&tmQ, smem_u32(qstg), nb * BN + col, row0);
            bulk_commit_group();
          }
        };
        bool last = true;  // this unit stores the tile
        if constexpr (QF < 0 && BN != 192) {  // split K: 256- and 128-wide bf16-output tiles
          if (pq.splits > 1) {
            // this warp's slice of the partial tile: 32 lanes x (64 or 128) fp32, stored so that
            // each float4 index is 512 contiguous bytes across the warp
            constexpr int SLOT_V = ((NCH + 1) / 2) * 16;  // float4 per lane
            const int slice = (t * (PAIR ? 2 : 1) + static_cast<int>(rank)) * C::EPI_WARPS + ew;
            float4* slot0 = pq.ws + static_cast<size_t>(slice) * pq.splits * SLOT_V * 32;
            float4* mine = slot0 + static_cast<size_t>(split) * SLOT_V * 32 + lane;
            auto put = [&](const uint32_t(&r)[32], int v0) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                __stcg(mine + (v0 + i) * 32, make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                         __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
            };
            put(r0, 0);
            put(r1, 8);
            if (two) {
              put(r2, 16);
              put(r3, 24);
            }
            __threadfence();
            __syncwarp();
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(pq.ws_cnt + slice, 1);
            ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
            last = ticket == pq.splits - 1;
            if (last) {
              __threadfence();
              // two splits: add the other unit's partial to this one's in place; fp32 addition
              // is commutative, so the sum does not depend on which unit finished last. Eight
              // loads in flight per lane, then eight adds.
              const float4* other = slot0 + static_cast<size_t>(1 - split) * SLOT_V * 32 + lane;
              auto add = [&](uint32_t(&r)[32], int v0) {
                float4 b[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) b[i] = __ldcg(other + (v0 + i) * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  r[4 * i] = __float_as_uint(__fadd_rn(__uint_as_float(r[4 * i]), b[i].x));
                  r[4 * i + 1] = __float_as_uint(__fadd_rn(__uint_as_float(r[4 * i + 1]), b[i].y));
                  r[4 * i + 2] = __float_as_uint(__fadd_rn(__uint_as_float(r[4 * i + 2]), b[i].z));
                  r[4 * i + 3] = __float_as_uint(__fadd_rn(__uint_as_float(r[4 * i + 3]), b[i].w));
                }
              };
              add(r0, 0);
              add(r1, 8);
              if (two) {
                add(r2, 16);
                add(r3, 24);
              }
              if (lane == 0) pq.ws_cnt[slice] = 0;  // zero again for the next call
            }
          }
        }
        if (last) {
          emit(r0, r1, hc * 64);
          if (two) emit(r2, r3, (hc + 2) * 64);
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
    }
    if (lane == 0) bulk_wait_group<0>();
    if (warp == 2 && lane == 0) FP8GB_STAMP(5);
  }

  tc_fence_before();
  __syncthreads();
  // a pair's CTAs leave together: no MMA, commit arrival or TMA write targets an exited CTA
  if constexpr (PAIR) cluster_sync_all();
  if (threadIdx.x == 0) FP8GB_STAMP(6);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------
// Block-scaled GEMM with 256-wide tiles: the fold keeps the whole tile in registers
// ---------------------------------------------------------------------------------------
// C[m, n] = bf16( sum_kb fl32(d_a[m, kb] d_b[kb, n/128]) P_kb[m, n] ): every 128-deep K block
// is accumulated by the tensor cores in a fresh TMEM buffer (two of BN columns, alternating),
// and eight fold warps multiply it by its scale product and add it into fp32 registers.
// Warpgroup 0 holds the TMA producer (warp 0) and the MMA issuer (warp 1; warps 2-3 idle) and
// gives registers up (setmaxnreg) to the fold warpgroups 1-2, whose threads each hold BN/2
// accumulators: the two warps of a TMEM lane quarter split the tile's columns in halves, and
// each half lies in one 128-column scale block of B. With two buffers the MMA runs one block
// ahead of the fold, so the time from a block's completion to the release of its buffer sits
// on the tensor pipe's path. Per-block clock traces (16384 x 14336 x 4096, CTA pairs) put
// that time at ~700 cycles when a thread loaded 64 columns, folded them and loaded the other
// 64 (~150 without the FMAs), and the round trip from a release to the completion of the
// block two ahead at ~1200 cycles, against ~700 per block of tensor work. A warp issues in
// order, so a load into registers that the preceding FMAs read waits for them: the fold
// therefore loads through 80 registers in three groups, each load placed ahead of FMAs on
// other registers (see the loop). 224-wide tiles with a whole block in registers (32
// accumulators per thread parked in the TMEM the narrower buffers leave free) measured slower:
// the tensor pipe takes about as long per K block at N = 224 as at 256.
// With PAIR, two CTAs of a cluster share a 256 x BN tile through the CTA-pair MMA (each holds
// its 128 rows of A and half of B's rows) and each folds its own 128 rows.
template <int BN, bool PAIR>
struct BlkCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
  static constexpr int B_BYTES = B_ROWS * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int FOLD_WARPS = 8;
  static constexpr int COLS = BN / 2;  // accumulator columns per fold thread
  static constexpr int THREADS = 384;  // three warpgroups
  static constexpr int STG = FOLD_WARPS * STG_BYTES;
  static constexpr int STAGES_FIT = (230000 - STG) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < (192 * 1024) / STAGE_BYTES ? STAGES_FIT : (192 * 1024) / STAGE_BYTES;
  static constexpr int ACC = 512 / BN;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_STG + STG;
  static constexpr int NBAR = 2 * STAGES + 2 * ACC + 1;  // full[S], empty[S], tfull[ACC], tempty[ACC], final
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int TEMPTY_COUNT = (PAIR ? 2 : 1) * FOLD_WARPS;
  // register split: a CTA is launched with THREADS x LAUNCH_REGS registers; warpgroup 0 keeps
  // CTRL_REGS per thread and the two fold warpgroups take FOLD_REGS (0: no split)
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int CTRL_REGS = BN == 256 ? 40 : 56;
  static constexpr int FOLD_REGS = BN == 256 ? 232 : 0;
  static_assert(FOLD_REGS == 0 || 128 * CTRL_REGS + 256 * FOLD_REGS <= THREADS * LAUNCH_REGS, "register split");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(STAGES >= 3, "ring depth");
  static_assert(OFF_STG % 1024 == 0, "staging buffers on 1024-byte swizzle atoms");
};

// a0, a1 += fp32(v0) * s, fp32(v1) * s: two fp32 FMAs (round to nearest each) in one packed
// instruction. The pairs are formed with mov.b64 inside the asm so that ptxas can keep each
// accumulator pair in an aligned register pair (measured 4 % faster for the whole GEMM than
// building the 64-bit operands with shifts).
__device__ __forceinline__ void fma2(float& a0, float& a1, uint32_t v0, uint32_t v1, float s) {
  asm("{\n\t.reg .b64 a, v, s;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 v, {%2, %3};\n\t"
      "mov.b64 s, {%4, %4};\n\t"
      "fma.rn.f32x2 a, v, s, a;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(v0), "r"(v1), "f"(s));
}

template <int BN, bool PAIR>
__global__ void __launch_bounds__(BlkCfg<BN, PAIR>::THREADS, 1)
    gemm_blk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ KParams p) {
  using C = BlkCfg<BN, PAIR>;
  constexpr int STAGES = C::STAGES;
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
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  constexpr int TILE_M = PAIR ? 2 * BM : BM;
  const KProb& pb = p.pr[0];  // one problem, never split

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, C::TEMPTY_COUNT);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers are initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  if (warp < 4) {
    if constexpr (C::FOLD_REGS > 0) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::CTRL_REGS));
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      const uint32_t full_lead = PAIR ? mapa_shared(bar_full, 0) : bar_full;
      for (int t = tile0; ok && t < pb.num_tiles; t += tile_step) {
        int mb, nb;
        tile_coords(t, pb, p.group_m, mb, nb);
        const int arow = mb * TILE_M + static_cast<int>(rank) * BM;
        const int brow = nb * BN + static_cast<int>(rank) * C::B_ROWS;
        for (int kb = 0; kb < pb.num_kb; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.w, DEV_ERR_WAIT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          if constexpr (PAIR) {
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
            tma_load_2d_pair(sa, &tmA, full_lead + 8 * stage, kb * BK, arow);
            tma_load_2d_pair(sa + A_BYTES, &tmB, full_lead + 8 * stage, kb * BK, brow);
          } else {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            tma_load_2d(sa, &tmA, fb, kb * BK, arow);
            tma_load_2d(sa + A_BYTES, &tmB, fb, kb * BK, brow);
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every load already issued land before the CTA exits
        if constexpr (PAIR) {
          const unsigned long long t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        } else {
          for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s)) mbar_wait_drain(bar_full + 8 * s, (issued_phase >> s) & 1u, 1000000000ull);
        }
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------- MMA issuer: one TMEM buffer per K block ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = tile0; ok && t < pb.num_tiles; t += tile_step) {
        for (int kb = 0; kb < pb.num_kb; ++kb) {
          if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, p.w, DEV_ERR_WAIT_MMA) ||
              !mbar_wait(bar_full + 8 * stage, phase, p.w, DEV_ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            if constexpr (PAIR)
              mma_f8_pair(d, adesc + 2 * k, bdesc + 2 * k, pb.idesc, k != 0);
            else
              mma_f8(d, adesc + 2 * k, bdesc + 2 * k, pb.idesc, k != 0);
          }
          if constexpr (PAIR) {
            mma_commit_pair(bar_empty + 8 * stage, 0x3);
            mma_commit_pair(bar_tfull + 8 * acc, 0x3);
          } else {
            mma_commit(bar_empty + 8 * stage);
            mma_commit(bar_tfull + 8 * acc);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          acc = (acc + 1 == ACC) ? 0 : acc + 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      if constexpr (PAIR)
        mma_commit_pair(bar_final, 0x1);
      else
        mma_commit(bar_final);
      if (!mbar_wait_drain(bar_final, 0, 1000000000ull)) atomicOr(p.w.err, DEV_ERR_WAIT_TEARDOWN);
    }
  } else {
    // ---------------- fold (warpgroups 1-2) ----------------
    if constexpr (C::FOLD_REGS > 0) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::FOLD_REGS));
    constexpr int COLS = C::COLS;
    const int fw = warp - 4;  // 0 .. 7
    const int q = warp & 3;   // TMEM lane quarter
    const int col0 = (fw >> 2) * COLS;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tempty_lead = PAIR ? mapa_shared(bar_tempty, 0) : bar_tempty;
    uint8_t* stg = smem + C::OFF_STG + fw * STG_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = tile0; ok && t < pb.num_tiles; t += tile_step) {
      int mb, nb;
      tile_coords(t, pb, p.group_m, mb, nb);
      const int row0 = mb * TILE_M + static_cast<int>(rank) * BM + q * 32;  // this warp's 32 rows
      const int row = row0 + lane;
      const int nblk = (nb * BN + col0) / 128;
      const bool row_ok = row < pb.M;
      const bool col_ok = nblk * 128 < pb.N;
      const float* sa_row = pb.sa + static_cast<int64_t>(row_ok ? row : 0) * pb.sa_ld;
      const float* sb_col = pb.sb + (col_ok ? nblk : 0);
      float accum[COLS];
#pragma unroll
      for (int j = 0; j < COLS; ++j) accum[j] = 0.0f;
      // scales two K blocks ahead: an L2 round trip is longer than one block's fold
      float sa1 = row_ok ? __ldg(sa_row) : 0.0f, sb1 = col_ok ? __ldg(sb_col) : 0.0f;
      float sa2 = (row_ok && pb.num_kb > 1) ? __ldg(sa_row + 1) : 0.0f;
      float sb2 = (col_ok && pb.num_kb > 1) ? __ldg(sb_col + pb.sb_ld) : 0.0f;
      if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, p.w, DEV_ERR_WAIT_EPILOGUE)) break;
      __syncwarp();
      tc_fence_after();
      auto release = [&]() {  // this warp's reads of the buffer are done: hand it back to the MMA
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(tempty_lead + 8 * acc);
          else
            mbar_arrive(bar_tempty + 8 * acc);
        }
        acc = (acc + 1 == ACC) ? 0 : acc + 1;
        if (acc == 0) acc_phase ^= 1u;
      };
      auto next_block = [&]() {  // wait for the next K block's buffer (the whole warp agrees)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull + 8 * acc, acc_phase, p.w, DEV_ERR_WAIT_EPILOGUE));
        tc_fence_after();
        return ok;
      };
      if constexpr (COLS == 128) {
        // 128 columns per thread through 80 buffer registers in three groups: lo = columns 0-47
        // (bA, bB), mid = 48-79 (bC, bD), hi = 80-127 (bA, bB again). Per block: lo and mid
        // land; lo is folded; hi is loaded into lo's registers while mid is folded; the TMEM
        // buffer goes back once hi has landed; the next block's mid is loaded while hi is
        // folded, then its lo. A warp issues in order, so every load is placed ahead of FMAs on
        // other registers: the loads overlap the FMAs, and only 80 columns of FMAs lie between
        // a block's completion and the release of its buffer.
        uint32_t bA[32], bB[16], bC[16], bD[16];
        auto addr = [&]() { return tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + col0); };
        auto load_lo = [&](uint32_t a) {
          tmem_ld32(a, bA);
          tmem_ld16(a + 32, bB);
        };
        auto load_mid = [&](uint32_t a) {
          tmem_ld16(a + 48, bC);
          tmem_ld16(a + 64, bD);
        };
        auto fold_ab = [&](int c, float sc) {  // columns c .. c+47 from bA, bB
#pragma unroll
          for (int j = 0; j < 32; j += 2) fma2(accum[c + j], accum[c + j + 1], bA[j], bA[j + 1], sc);
#pragma unroll
          for (int j = 0; j < 16; j += 2) fma2(accum[c + 32 + j], accum[c + 33 + j], bB[j], bB[j + 1], sc);
        };
        {
          const uint32_t a = addr();
          load_mid(a);
          load_lo(a);
        }
        for (int kb = 0; ok && kb < pb.num_kb; ++kb) {
          const float sc = __fmul_rn(sa1, sb1);
          const bool more = kb + 1 < pb.num_kb;
          sa1 = sa2;
          sb1 = sb2;
          sa2 = (row_ok && kb + 2 < pb.num_kb) ? __ldg(sa_row + kb + 2) : 0.0f;
          sb2 = (col_ok && kb + 2 < pb.num_kb) ? __ldg(sb_col + static_cast<int64_t>(kb + 2) * pb.sb_ld) : 0.0f;
          tmem_ld_wait();
          reg_fence(bA);
          reg_fence(bB);
          reg_fence(bC);
          reg_fence(bD);
          fold_ab(0, sc);
          {
            const uint32_t a = addr();
            tmem_ld32(a + 80, bA);
            tmem_ld16(a + 112, bB);
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2) fma2(accum[48 + j], accum[49 + j], bC[j], bC[j + 1], sc);
#pragma unroll
          for (int j = 0; j < 16; j += 2) fma2(accum[64 + j], accum[65 + j], bD[j], bD[j + 1], sc);
          tmem_ld_wait();
          reg_fence(bA);
          reg_fence(bB);
          release();
          if (!more) {
            fold_ab(80, sc);
          } else if (__all_sync(0xFFFFFFFFu, mbar_test_wait(bar_tfull + 8 * acc, acc_phase))) {
            // the next block is already waiting: its mid goes ahead of this block's hi FMAs;
            // otherwise the hi FMAs fill the wait
            __syncwarp();
            tc_fence_after();
            const uint32_t a = addr();
            load_mid(a);
            fold_ab(80, sc);
            load_lo(a);
          } else {
            fold_ab(80, sc);
            if (next_block()) {
              const uint32_t a = addr();
              load_mid(a);
              load_lo(a);
            }
          }
        }
      } else {
        // 64 columns per thread: one load, the buffer handed back before the FMAs
        uint32_t buf[64];
        tmem_ld64(tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + col0), buf);
        for (int kb = 0; ok && kb < pb.num_kb; ++kb) {
          const float sc = __fmul_rn(sa1, sb1);
          const bool more = kb + 1 < pb.num_kb;
          sa1 = sa2;
          sb1 = sb2;
          sa2 = (row_ok && kb + 2 < pb.num_kb) ? __ldg(sa_row + kb + 2) : 0.0f;
          sb2 = (col_ok && kb + 2 < pb.num_kb) ? __ldg(sb_col + static_cast<int64_t>(kb + 2) * pb.sb_ld) : 0.0f;
          tmem_ld_wait();
          reg_fence(buf);
          release();
#pragma unroll
          for (int j = 0; j < 64; j += 2) fma2(accum[j], accum[j + 1], buf[j], buf[j + 1], sc);
          if (more && next_block()) tmem_ld64(tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + col0), buf);
        }
      }
      if (!ok) break;
      // bf16 out, 64 columns per staged TMA store
#pragma unroll
      for (int c = 0; c < COLS / 64; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(accum[c * 64 + 2 * j], accum[c * 64 + 2 * j + 1]);
        if (lane == 0) bulk_wait_group_read<0>();  // the staging buffer's previous store has read it
        __syncwarp();
        const int cc = nb * BN + col0 + c * 64;
        if (row0 < pb.M && cc < pb.N) stage_and_store(stg, pk, lane, &tmC, cc, row0);
      }
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
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

template <int BN, int QF, bool PAIR, bool MX = false>
cudaError_t prepare_kernel(int* pair_clusters) {
  // the attribute is per device; remember which devices were configured and, for CTA-pair
  // kernels, how many pairs the device holds at once
  static bool done[64] = {};
  static int clusters[64] = {};
  static std::mutex mu;
  using C = Cfg<BN, QF, PAIR, MX>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && done[dev]) {
    *pair_clusters = clusters[dev];
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(gemm_f8_kernel<BN, QF, PAIR, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int n = 0;
  if (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(gemm_f8_kernel<BN, QF, PAIR, MX>), &cfg);
    if (e != cudaSuccess) return e;
  }
  if (dev < 64) {
    done[dev] = true;
    clusters[dev] = n;
  }
  *pair_clusters = n;
  return cudaSuccess;
}

// Tile shape: cost = rounds of tiles over the SMs (or CTA pairs) x time of one round.
// Measured on GB300 (ns per 128-deep K block of one tile, 16384 x 14336 x 4096): the tensor
// pipe takes ~280-300 ns for any N <= 256, so narrower tiles save little time per tile; a
// single CTA with 256-wide tiles is bound by its operand intake (~140 GB/s, 48 KB per K
// block) at ~360 ns, 192-wide at ~320 ns; a CTA pair loads 16 KB + BN * 64 bytes per CTA
// and K block and runs at the tensor pipe's rate. Narrower tiles win only when they save
// rounds.
struct TileChoice {
  int bn;
  bool pair;
  int splits;
};

// Split K costs each unit a write of its fp32 partial and the tile's last unit a read of all
// of them (~128 KB per CTA each at ~140 GB/s): about 3 K blocks of time per unit and round,
// plus ~900 ns per split for the last round's reads. Splits are for tiles too few to fill
// the GPU, with a workspace that stays in L2.
constexpr int kSplitCostNs = 900;
constexpr int kSplitUnitKb = 3;
constexpr int64_t kSplitMaxBytes = int64_t(64) << 20;
// The workspace starts with a fixed 16 KB of arrival counters (one per tile, CTA rank and
// epilogue warp: at most 64 MB / (2 splits x 8 KB) = 4096 of them), so the partials of one
// shape never overlap the counters of another and a reused workspace needs no clearing.
constexpr int64_t kSplitCounterBytes = 4096 * 4;

TileChoice choose_tile(int64_t M, int64_t N, int64_t K, int sms, int pair_clusters, int max_splits, bool mn = false) {
  const int widths[3] = {256, 192, 128};
  const int w_single[3] = {362, 322, 275};
  const int w_pair[3] = {300, 285, 278};
  const int64_t kb = (K + BK - 1) / BK;
  TileChoice best{256, false, 1};
  int64_t best_cost = -1;
  for (int i = 0; i < 3; ++i) {
    if (mn && widths[i] == 192) continue;  // MN-major B tiles are whole 128-column boxes
    const int64_t tn = (N + widths[i] - 1) / widths[i];
    for (int pair = 0; pair < 2; ++pair) {
      if (pair && (M <= BM || pair_clusters <= 0)) continue;  // a pair computes 256 rows
      if (pair && mn && widths[i] != 256) continue;
      const int64_t tiles = pair ? (M + 2 * BM - 1) / (2 * BM) * tn : (M + BM - 1) / BM * tn;
      const int64_t slots = pair ? pair_clusters : sms;
      for (int sp = 1; sp <= (widths[i] == 192 ? 1 : max_splits) && sp <= kb; ++sp) {
        if (sp > 1) {  // workspace: one 16 KB (8 KB at 128 wide) slice per warp, tile and split
          const int64_t bytes = tiles * (pair ? 2 : 1) * 8 * sp * (widths[i] == 128 ? 8192 : 16384);
          if (bytes > kSplitMaxBytes) break;
        }
        const int64_t rounds = (tiles * sp + slots - 1) / slots;
        const int64_t cost = rounds * ((kb + sp - 1) / sp + (sp > 1 ? kSplitUnitKb : 0)) *
                                 (pair ? w_pair[i] : w_single[i]) +
                             (sp > 1 ? static_cast<int64_t>(sp) * kSplitCostNs : 0);
        if (best_cost < 0 || cost < best_cost) {
          best_cost = cost;
          best = {widths[i], pair != 0, sp};
        }
      }
    }
  }
  return best;
}

// Workspace of a split-K launch: arrival counters, then the fp32 partials.
struct SplitLayout {
  int64_t slices, counter_bytes, total_bytes;
};

SplitLayout split_layout(int64_t M, int64_t N, const TileChoice& c) {
  SplitLayout l{0, 0, 0};
  if (c.splits <= 1) return l;
  const int64_t tn = (N + c.bn - 1) / c.bn;
  const int64_t tiles = c.pair ? (M + 2 * BM - 1) / (2 * BM) * tn : (M + BM - 1) / BM * tn;
  const int64_t slot_v = ((c.bn / 64 + 1) / 2) * 16;  // float4 per lane of one warp's slice
  l.slices = tiles * (c.pair ? 2 : 1) * 8;
  l.counter_bytes = kSplitCounterBytes;
  l.total_bytes = l.counter_bytes + l.slices * c.splits * slot_v * 32 * 16;
  return l;
}

// Tensor maps of one problem (A and B K-major codes, C bf16).
struct Maps {
  CUtensorMap a, b, c;
};

// The launch's view of one GEMM: tile counts, instruction descriptor, scales and (when the
// choice splits K) its workspace; the tensor maps with the tile's box sizes.
bool make_problem(const GemmArgs& g, const TileChoice& c, KProb& q, Maps& m, const char** why) {
  const int rows = c.pair ? 2 * BM : BM;
  q.M = static_cast<int>(g.M);
  q.N = static_cast<int>(g.N);
  q.K = static_cast<int>(g.K);
  q.num_m = static_cast<int>((g.M + rows - 1) / rows);
  q.num_n = static_cast<int>((g.N + c.bn - 1) / c.bn);
  q.num_kb = static_cast<int>((g.K + BK - 1) / BK);
  q.num_tiles = q.num_m * q.num_n;
  if (g.mn && (g.mx || g.block_scaled || g.qf >= 0 || c.bn == 192 || (c.pair && c.bn != 256))) {
    *why = "MN-major operands: per-tensor scales, bf16 output, tiles of whole 128-column boxes";
    return false;
  }
  q.mn = g.mn ? 1 : 0;
  q.idesc = g.mx ? idesc_mxf8(static_cast<uint32_t>(g.fa), static_cast<uint32_t>(g.fb), static_cast<uint32_t>(rows),
                              static_cast<uint32_t>(c.bn))
                 : idesc_f8(static_cast<uint32_t>(g.fa), static_cast<uint32_t>(g.fb), static_cast<uint32_t>(rows),
                            static_cast<uint32_t>(c.bn));
  if (g.mn) q.idesc |= idesc_mn_major();
  q.sfa = g.mx ? g.sfa8 : nullptr;
  q.sfb = g.mx ? g.sfb8 : nullptr;
  q.sf_nkb = static_cast<int>(g.K / 128);
  q.sfb_atoms = static_cast<int>((g.N + 127) / 128);
  q.sa = g.sa;
  q.sb = g.sb;
  q.sa_ld = static_cast<int>(g.K / 128);
  q.sb_ld = static_cast<int>(g.N / 128);
  q.splits = 1;
  q.ws = nullptr;
  q.ws_cnt = nullptr;
  q.unit0 = 0;
  if (c.splits > 1) {
    const SplitLayout l = split_layout(g.M, g.N, c);
    q.splits = c.splits;
    q.ws_cnt = static_cast<int*>(g.ws);
    q.ws = reinterpret_cast<float4*>(static_cast<uint8_t*>(g.ws) + l.counter_bytes);
  }
  const uint32_t b_rows = c.pair ? static_cast<uint32_t>(c.bn / 2) : static_cast<uint32_t>(c.bn);
  const bool cmap = g.mx ? encode_tmap_2d(&m.c, g.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.N, g.M, g.ldc * 2, 32, 32, 64)
                         : make_map(&m.c, g.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.N, g.M, g.ldc * 2, 64, 32);
  const bool amap = g.mn ? make_map(&m.a, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.M, g.K, g.lda, 128, BK)
                        : make_map(&m.a, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K, g.M, g.lda, BK, BM);
  const bool bmap = g.mn ? make_map(&m.b, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.N, g.K, g.ldb, 128, BK)
                        : make_map(&m.b, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K, g.N, g.ldb, BK, b_rows);
  if (!amap || !bmap || !cmap) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point missing or tensor map rejected)";
    return false;
  }
  return true;
}

// Units of unequal length (a grouped launch) are packed onto the slots by first-fit
// decreasing under a makespan bound found by bisection: the shortest bound under which every
// unit fits. Returns that makespan (in K blocks) and, when `lists` is given, the packing.
int64_t pack_units(const std::vector<std::pair<int, int>>& us_sorted, int slots,
                   std::vector<std::vector<int>>* lists) {
  int64_t total = 0, longest = 0;
  for (const auto& x : us_sorted) {
    total += x.first;
    longest = std::max<int64_t>(longest, x.first);
  }
  auto fits = [&](int64_t bound, std::vector<std::vector<int>>* out) {
    std::vector<int64_t> load(slots, 0);
    if (out) out->assign(slots, {});
    for (const auto& x : us_sorted) {
      int sl = 0;
      while (sl < slots && load[sl] + x.first > bound) ++sl;
      if (sl == slots) return false;
      load[sl] += x.first;
      if (out) (*out)[sl].push_back(x.second);
    }
    return true;
  };
  int64_t lo = std::max<int64_t>(longest, (total + slots - 1) / slots), hi = total;
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (fits(mid, nullptr))
      hi = mid;
    else
      lo = mid + 1;
  }
  if (lists) fits(lo, lists);
  return lo;
}

// Units of the launch's problems as (K blocks, unit index), longest first.
std::vector<std::pair<int, int>> launch_units(const KParams& p) {
  std::vector<std::pair<int, int>> us;
  for (int pi = 0; pi < p.nprob; ++pi) {
    const KProb& q = p.pr[pi];
    for (int v = 0; v < q.num_tiles * q.splits; ++v) {
      const int sp = v % q.splits;
      us.push_back({(sp + 1) * q.num_kb / q.splits - sp * q.num_kb / q.splits, q.unit0 + v});
    }
  }
  std::stable_sort(us.begin(), us.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
  return us;
}

// Round-robin makespan (slot s takes units s, s + slots, ...), in K blocks.
int64_t round_robin_makespan(const KParams& p, int slots) {
  std::vector<int64_t> load(slots, 0);
  for (const auto& x : launch_units(p)) load[x.second % slots] += x.first;
  return *std::max_element(load.begin(), load.end());
}

// Explicit schedule of a grouped launch when it beats round robin; cached per shape (the
// packing search is host work a repeated call should not pay again).
void make_schedule(KParams& p, int slots) {
  p.sched_len = 0;
  if (p.nprob < 2 || p.units > kMaxSchedUnits || slots > kMaxSlots) return;
  using Key = std::array<int, 7>;
  struct Sched {
    int len;
    std::vector<uint16_t> off, unit;
  };
  static std::mutex mu;
  static std::map<Key, Sched> cache;
  const Key key{p.pr[0].num_tiles, p.pr[0].splits, p.pr[0].num_kb, p.pr[1].num_tiles, p.pr[1].splits,
                p.pr[1].num_kb, slots};
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it == cache.end()) {
    Sched sc{0, {}, {}};
    std::vector<std::vector<int>> lists;
    const auto us = launch_units(p);
    if (pack_units(us, slots, &lists) < round_robin_makespan(p, slots)) {
      int off = 0;
      for (int sl = 0; sl < slots; ++sl) {
        sc.off.push_back(static_cast<uint16_t>(off));
        for (int u : lists[sl]) {
          sc.unit.push_back(static_cast<uint16_t>(u));
          ++off;
        }
      }
      sc.off.push_back(static_cast<uint16_t>(off));
      sc.len = off;
    }
    if (cache.size() >= 256) cache.clear();  // bounded: a workload uses a handful of shapes
    it = cache.emplace(key, std::move(sc)).first;
  }
  const Sched& sc = it->second;
  p.sched_len = sc.len;
  for (size_t i = 0; i < sc.off.size(); ++i) p.sched_off[i] = sc.off[i];
  for (size_t i = 0; i < sc.unit.size(); ++i) p.sched_unit[i] = sc.unit[i];
}

// The kernel's division-free work-unit mapping (DivBy): per problem the tile raster's
// divisors and the first split unit's K blocks, and the grid's slot count.
void set_divisors(KParams& p, int slots) {
  for (KProb* q : {&p.pr[0], &p.pr[1]}) {
    const int gm = p.group_m;
    q->kb_half = q->num_kb / 2;
    q->div_group = make_div(static_cast<uint32_t>(gm * q->num_n));
    q->div_gm = make_div(static_cast<uint32_t>(gm));
    const int glast = q->num_m - ((q->num_m + gm - 1) / gm - 1) * gm;  // rows of the last group
    q->div_glast = make_div(static_cast<uint32_t>(glast > 0 ? glast : gm));
  }
  p.div_slots = make_div(static_cast<uint32_t>(slots));
}

template <int BN, int QF, bool PAIR, bool MX = false>
cudaError_t launch_kernel(const Maps& m0, const Maps& m1, const CUtensorMap& tq, KParams& p, cudaStream_t stream) {
  using C = Cfg<BN, QF, PAIR, MX>;
  if (p.pr[0].splits > 2 || p.pr[1].splits > 2) return cudaErrorInvalidValue;  // (unit_at: one or two)
  int clusters = 0;
  cudaError_t e = prepare_kernel<BN, QF, PAIR, MX>(&clusters);
  if (e != cudaSuccess) return e;
  int slots = PAIR ? clusters : num_sms();
  if (slots <= 0) return cudaErrorInvalidConfiguration;
  if (slots > kMaxSlots) slots = kMaxSlots;
  if (p.units < slots) slots = p.units;
  make_schedule(p, slots);
  set_divisors(p, slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * slots : slots));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_f8_kernel<BN, QF, PAIR, MX>, m0.a, m0.b, m0.c, tq, m1.a, m1.b, m1.c, p);
}

template <int QF>
cudaError_t launch_choice(const TileChoice& c, const Maps& m0, const Maps& m1, const CUtensorMap& tq, KParams& p,
                          cudaStream_t stream) {
  if (c.pair) {
    if (c.bn == 256) return launch_kernel<256, QF, true>(m0, m1, tq, p, stream);
    if (c.bn == 192) return launch_kernel<192, QF, true>(m0, m1, tq, p, stream);
    return launch_kernel<128, QF, true>(m0, m1, tq, p, stream);
  }
  if (c.bn == 256) return launch_kernel<256, QF, false>(m0, m1, tq, p, stream);
  if (c.bn == 192) return launch_kernel<192, QF, false>(m0, m1, tq, p, stream);
  return launch_kernel<128, QF, false>(m0, m1, tq, p, stream);
}

// The block-scaled kernel's launch configuration on the current device: shared memory set,
// the register split checked (setmaxnreg.inc waits until the CTA's pool holds the registers it
// asks for, so a kernel compiled with fewer registers than the split assumes is never launched)
// and, for CTA pairs, the pairs the device holds at once.
template <int BN, bool PAIR>
cudaError_t prepare_blk(int* slots, const char** why) {
  using C = BlkCfg<BN, PAIR>;
  static bool done[64] = {};
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && done[dev]) {
    *slots = cached[dev];
    return cudaSuccess;
  }
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, gemm_blk_kernel<BN, PAIR>)) != cudaSuccess) return e;
  if (C::FOLD_REGS > 0 && fa.numRegs < C::LAUNCH_REGS) {
    *why = "block-scaled GEMM: kernel compiled with fewer registers than its register split needs";
    return cudaErrorInvalidConfiguration;
  }
  if ((e = cudaFuncSetAttribute(gemm_blk_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM)) !=
      cudaSuccess)
    return e;
  int n = num_sms();
  if (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(gemm_blk_kernel<BN, PAIR>), &cfg)) !=
        cudaSuccess)
      return e;
  }
  if (dev < 64) {
    done[dev] = true;
    cached[dev] = n;
  }
  *slots = n;
  return cudaSuccess;
}

template <int BN, bool PAIR>
cudaError_t launch_blk(const Maps& m, KParams& p, cudaStream_t stream, const char** why) {
  using C = BlkCfg<BN, PAIR>;
  int slots = 0;
  cudaError_t e = prepare_blk<BN, PAIR>(&slots, why);
  if (e != cudaSuccess) return e;
  if (slots <= 0) return cudaErrorInvalidConfiguration;
  if (slots > p.pr[0].num_tiles) slots = p.pr[0].num_tiles;
  set_divisors(p, slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * slots : slots));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_blk_kernel<BN, PAIR>, m.a, m.b, m.c, p);
}

// Pairs of the block-scaled kernel the device holds at once (0: no clusters of two).
int blk_pair_capacity() {
  int n = 0;
  const char* why = nullptr;
  if (prepare_blk<256, true>(&n, &why) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Pairs the device holds at once (0 when it cannot launch clusters of two).
int pair_capacity() {
  int n = 0;
  if (prepare_kernel<256, -1, true>(&n) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
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

bool encode_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int64_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const TileChoice c = choose_tile(M, N, K, num_sms(), pair_capacity(), 2);
  return split_layout(M, N, c).total_bytes;
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream, const char** why) {
  // block scaling folds every 128-deep K block out of TMEM into registers: 256-wide tiles
  // (two TMEM buffers) unless N is one 128-column block, on CTA pairs when M has more than
  // one row block
  TileChoice choice{g.N > 128 ? 256 : 128, false, 1};
  if (g.mx) {
    // whole scale atoms per tile: 256 wide (one accumulator, the next tile's MMAs wait for this
    // tile's TMEM loads), on CTA pairs when M has more than one row block, or 128 wide on
    // single CTAs (three accumulators)
#ifdef FP8GB_MX_FORCE_BN
    choice.bn = FP8GB_MX_FORCE_BN;
#endif
#ifdef FP8GB_MX_FORCE_PAIR  // compile-time override, for tuning builds
    choice.pair = FP8GB_MX_FORCE_PAIR != 0 && choice.bn == 256 && g.M > BM;
#else
    choice.pair = choice.bn == 256 && g.M > BM && pair_capacity() > 0;
#endif
  } else if (g.block_scaled) {
#ifdef FP8GB_BLK_FORCE_PAIR  // compile-time override, for tuning builds
    choice.pair = FP8GB_BLK_FORCE_PAIR != 0 && g.M > BM;
#else
    choice.pair = g.M > BM && blk_pair_capacity() > 0;
#endif
  } else {
#ifdef FP8GB_FORCE_BN  // compile-time override of the tile choice, for tuning builds
#ifndef FP8GB_FORCE_PAIR
#define FP8GB_FORCE_PAIR 0
#endif
    choice = {FP8GB_FORCE_BN, FP8GB_FORCE_PAIR != 0, 1};
#else
    choice = choose_tile(g.M, g.N, g.K, num_sms(), pair_capacity(), g.qf < 0 && g.ws != nullptr ? 2 : 1, g.mn);
    // a workspace too small for the best split falls back to the best unsplit shape
    if (choice.splits > 1) {
      const SplitLayout l = split_layout(g.M, g.N, choice);
      if (l.total_bytes > g.ws_bytes || l.slices * 4 > kSplitCounterBytes)
        choice = choose_tile(g.M, g.N, g.K, num_sms(), pair_capacity(), 1, g.mn);
    }
#endif
  }
  KParams p{};
  // the long fine-grained GEMMs sweep B with 8192-row groups: measured at 16384 x 14336 x 4096,
  // B is then read from DRAM twice (fold kernel on pairs: 244 MB against 306 with 16 tiles per
  // group; MX on single CTAs: 204 MB against 550, 1.5 % faster); whole-M groups (16384 rows)
  // thrash L2 on pairs (937 MB)
  p.group_m = (g.block_scaled || g.mx) ? (choice.pair ? 32 : 64) : 16;
  Maps m0;
  if (!make_problem(g, choice, p.pr[0], m0, why)) return cudaErrorInvalidValue;
  p.pr[1] = p.pr[0];
  p.nprob = 1;
  p.units = p.pr[0].num_tiles * p.pr[0].splits;
  p.w = wait_ctl();
  if (p.w.err == nullptr) {
    *why = "device error word unavailable";
    return cudaErrorInvalidDevice;
  }
  CUtensorMap tq = m0.c;  // unused unless the epilogue also writes FP8 codes
  if (g.qf >= 0) {
    if (!encode_tmap_2d(&tq, g.Cq, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.N, g.M, g.ldcq, 64, 32, 64)) {
      *why = "cuTensorMapEncodeTiled failed for the FP8 output";
      return cudaErrorInvalidValue;
    }
    p.cst = g.cst;
  }
  if (g.mx && choice.pair) {
    // the scale atoms through tensor maps (a CTA pair's loads signal the even CTA's barrier):
    // A's as rows of 512 bytes (128 words), B's as [column block][K block][512 bytes], whose
    // box takes a 256-wide tile's two column blocks
    Maps msf = m0;
    const uint64_t nkb = static_cast<uint64_t>(g.K / 128);
    const uint64_t atoms_a = static_cast<uint64_t>((g.M + 127) / 128) * nkb;
    const uint64_t blocks_b = static_cast<uint64_t>((g.N + 127) / 128);
    if (!encode_tmap_2d(&msf.a, g.sfa8, CU_TENSOR_MAP_DATA_TYPE_UINT32, 128, atoms_a, 512, 128, 1, 0) ||
        !encode_tmap_3d(&msf.b, g.sfb8, CU_TENSOR_MAP_DATA_TYPE_UINT32, 128, nkb, blocks_b, 512, nkb * 512, 128, 1,
                        2)) {
      *why = "cuTensorMapEncodeTiled failed for the MX scale atoms";
      return cudaErrorInvalidValue;
    }
    return launch_kernel<256, -1, true, true>(m0, msf, tq, p, stream);
  }
  if (g.mx) return choice.bn == 256 ? launch_kernel<256, -1, false, true>(m0, m0, tq, p, stream)
                                    : launch_kernel<128, -1, false, true>(m0, m0, tq, p, stream);
  if (g.block_scaled) {
    if (choice.bn == 256)
      return choice.pair ? launch_blk<256, true>(m0, p, stream, why) : launch_blk<256, false>(m0, p, stream, why);
    return choice.pair ? launch_blk<128, true>(m0, p, stream, why) : launch_blk<128, false>(m0, p, stream, why);
  }
  if (g.qf == 0) return launch_choice<0>(choice, m0, m0, tq, p, stream);
  if (g.qf == 1) return launch_choice<1>(choice, m0, m0, tq, p, stream);
  return launch_choice<-1>(choice, m0, m0, tq, p, stream);
}

// Split-K workspace bytes of problem g in a grouped launch with tile choice c (0: no split).
int64_t group_split_bytes(const GemmArgs& g, const TileChoice& c) {
  if (c.splits <= 1) return 0;
  return split_layout(g.M, g.N, c).total_bytes;
}

bool group_pair(const GemmArgs& g0, const GemmArgs& g1) { return g0.M > BM && g1.M > BM && pair_capacity() > 0; }

// Tile choices of a grouped launch: CTA pairs with 256-wide tiles when both problems have
// more than 128 rows (else single CTAs), and for each problem K whole or in two halves,
// whichever packs the two problems' units into the shortest makespan (a split unit carries
// ~3 K blocks of partial-sum traffic) within `ws_limit` bytes of workspace. Cached per shape.
struct GroupPlan {
  TileChoice c0, c1;
  int64_t b0, b1;
};

GroupPlan plan_group(const GemmArgs& g0, const GemmArgs& g1, int64_t ws_limit) {
  const bool pair = group_pair(g0, g1);
  int slots = pair ? pair_capacity() : num_sms();
  if (slots > kMaxSlots) slots = kMaxSlots;
  using Key = std::array<int64_t, 9>;
  static std::mutex mu;
  static std::map<Key, GroupPlan> cache;
  const Key key{g0.M, g0.N, g0.K, g1.M, g1.N, g1.K, ws_limit, slots, pair ? 1 : 0};
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  GroupPlan best{{256, pair, 1}, {256, pair, 1}, 0, 0};
  int64_t best_cost = -1;
  for (int s0 = 1; s0 <= 2; ++s0) {
    for (int s1 = 1; s1 <= 2; ++s1) {
      const TileChoice c0{256, pair, s0}, c1{256, pair, s1};
      const SplitLayout l0 = split_layout(g0.M, g0.N, c0), l1 = split_layout(g1.M, g1.N, c1);
      const int64_t b0 = group_split_bytes(g0, c0), b1 = group_split_bytes(g1, c1);
      if (b0 + b1 > ws_limit || l0.slices * 4 > kSplitCounterBytes || l1.slices * 4 > kSplitCounterBytes) continue;
      if ((s0 > 1 && b0 - l0.counter_bytes > kSplitMaxBytes) || (s1 > 1 && b1 - l1.counter_bytes > kSplitMaxBytes))
        continue;
      std::vector<std::pair<int, int>> us;
      const GemmArgs* gs[2] = {&g0, &g1};
      const TileChoice* cs[2] = {&c0, &c1};
      for (int pi = 0; pi < 2; ++pi) {
        const int rows = pair ? 2 * BM : BM;
        const int64_t tiles = (gs[pi]->M + rows - 1) / rows * ((gs[pi]->N + 255) / 256);
        const int kb = static_cast<int>((gs[pi]->K + BK - 1) / BK), sp = cs[pi]->splits;
        if (sp > kb) {
          us.clear();
          break;
        }
        for (int64_t t = 0; t < tiles; ++t)
          for (int h = 0; h < sp; ++h)
            us.push_back({(h + 1) * kb / sp - h * kb / sp + (sp > 1 ? kSplitUnitKb : 0), 0});
      }
      if (us.empty() || static_cast<int64_t>(us.size()) > kMaxSchedUnits) continue;
      std::stable_sort(us.begin(), us.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
      const int64_t cost = pack_units(us, slots, nullptr);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = {c0, c1, b0, b1};
      }
    }
  }
  if (cache.size() >= 256) cache.clear();  // bounded: a workload uses a handful of shapes
  cache.emplace(key, best);
  return best;
}

int64_t gemm_group_workspace_bytes(const GemmArgs& g0, const GemmArgs& g1) {
  const GroupPlan pl = plan_group(g0, g1, INT64_MAX);
  return pl.b0 + pl.b1;
}

cudaError_t launch_gemm_group(const GemmArgs& g0in, const GemmArgs& g1in, void* ws, int64_t ws_bytes,
                              cudaStream_t stream, const char** why) {
  GemmArgs g0 = g0in, g1 = g1in;
  const GroupPlan pl = plan_group(g0, g1, ws != nullptr ? ws_bytes : 0);
  if (pl.b0 > 0) g0.ws = ws;
  if (pl.b1 > 0) g1.ws = static_cast<uint8_t*>(ws) + pl.b0;
  KParams p{};
  p.group_m = 16;
  Maps m0, m1;
  if (!make_problem(g0, pl.c0, p.pr[0], m0, why) || !make_problem(g1, pl.c1, p.pr[1], m1, why))
    return cudaErrorInvalidValue;
  p.nprob = 2;
  p.pr[0].unit0 = 0;
  p.pr[1].unit0 = p.pr[0].num_tiles * p.pr[0].splits;
  p.units = p.pr[1].unit0 + p.pr[1].num_tiles * p.pr[1].splits;
  p.w = wait_ctl();
  if (p.w.err == nullptr) {
    *why = "device error word unavailable";
    return cudaErrorInvalidDevice;
  }
  return launch_choice<-1>(pl.c0, m0, m1, m0.c, p, stream);
}

}  // namespace fp8gb
