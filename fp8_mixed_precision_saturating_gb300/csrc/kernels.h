// kernels.h -- internal interface between the C ABI (api.cu) and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8gb {

// Launch `kernel` on `stream` with programmatic stream serialization: it may begin while the
// previous kernel on the stream finishes; it waits for that kernel (pdl_wait) before it
// reads or writes global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Device pointers of one tensor role's scaling state (see fp8_tensor_state_t).
struct QuantState {
  float* hist;
  int32_t* hist_count;
  float* scale;
  float* scale_inv;
  float* amax_cur;
  unsigned long long* counters;
  int32_t hist_len;
};

// Up to 32 states pushed by one history-commit launch (distinct states, one thread each).
constexpr int kMaxCommit = 32;
struct QuantStates {
  QuantState s[kMaxCommit];
  int n;
};

// 2-D tensor map (TMA descriptor) of a row-major matrix: inner = contiguous extent, outer =
// rows, row_bytes = leading dimension in bytes; swizzle 128 = 128-byte swizzle, 0 = none.
bool encode_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle);
// 3-D tiled tensor map (no swizzle): dims d0 (contiguous) x d1 x d2, strides of dims 1 and 2
// in bytes, box b0 x b1 x b2.
bool encode_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Device error word and wait limit for launches on the current device.
WaitCtl wait_ctl();

// One tensor of a multi-tensor per-tensor quantise (tiled layout: rows, cols, ld multiples of
// 8, rows of 16 with qT); tile0 is its first tile in the launch's tile space.
constexpr int kMaxJobs = 4;
struct TileJob {
  const uint16_t* x;
  int64_t rows, cols, ld;
  uint8_t* q;
  uint8_t* qT;
  QuantState st;
  int delayed;
  int64_t tiles_x, ntiles, tile0;
};
struct TileJobs {
  TileJob j[kMaxJobs];
  int n;
};
// Up to kMaxJobs tensors of one format (0 E4M3, 1 E5M2) in one cooperative launch.
cudaError_t launch_quant_many(int fmt, const TileJobs& jobs, cudaStream_t stream);

// Per-tensor quantise in one cooperative launch: amax (when the call needs it), scale, cast
// with counters. tiled: 128x128 tiles with q and/or the transposed copy qT (rows, cols, ld
// multiples of 8); otherwise row-major q of any shape.
cudaError_t launch_quant_tensor(int fmt, bool delayed, bool tiled, const void* x, int64_t rows, int64_t cols,
                                int64_t ld, void* q, void* qT, const QuantState& st, cudaStream_t stream);
// Current-scaling quantise of a row-major tensor into contiguous codes, run only while
// st's history is empty (decided on the device); a no-op launch otherwise.
cudaError_t launch_quant_tensor_if_empty_history(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld,
                                                 void* q, const QuantState& st, cudaStream_t stream);
// W <- bf16(fl32(W) + delta) in place, then the per-tensor E4M3 quantise of the updated W into
// q [rows, cols] and/or qT [cols, rows], in one cooperative launch (W contiguous).
cudaError_t launch_update_quant_tensor(bool delayed, void* w, const float* delta, int64_t rows, int64_t cols,
                                       void* q, void* qT, const QuantState& st, cudaStream_t stream);
// One scale per 128x128 block (full blocks), q and/or qT, inverse scales [rows/128, cols/128].
cudaError_t launch_cast_blocks(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q, void* qT,
                               float* unit_scale_inv, const QuantState& st, cudaStream_t stream);
cudaError_t launch_cast_1x128(int fmt, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                              float* unit_scale_inv, const QuantState& st, cudaStream_t stream);
// MX scales (power of two per 32 elements along the contraction, UE8M0 bytes in 512-byte
// atoms [ceil(MN / 128)][K / 128]): along_rows = false quantises x [rows, cols] with groups
// along its rows (contraction = cols) into q [rows, cols]; along_rows = true quantises W
// [rows, cols] with groups along its columns (contraction = rows) into q = W_q^T [cols, rows].
cudaError_t launch_cast_mx(int fmt, bool along_rows, const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                           void* sf, const QuantState& st, cudaStream_t stream);
cudaError_t launch_history_commit(const QuantStates& sts, cudaStream_t stream);
cudaError_t launch_selftest_wait(const WaitCtl& w, cudaStream_t stream);

// GEMM: C [M,N] bf16 = A [M,K] * B [N,K]^T with per-tensor (block_scaled = false: sa, sb
// point to one fp32 each), fine-grained scales (block_scaled = true: sa [M, K/128],
// sb [K/128, N/128]) or MX scales (mx = true: sfa8, sfb8 UE8M0 scale atoms, K % 128 == 0).
struct GemmArgs {
  const void* A;
  const void* B;
  void* C;
  int64_t M, N, K, lda, ldb, ldc;
  int fa, fb;
  const float* sa;
  const float* sb;
  bool block_scaled;
  // optional FP8 output of the same epilogue: qf = -1 none, 0 E4M3, 1 E5M2
  int qf = -1;
  void* Cq = nullptr;
  int64_t ldcq = 0;
  QuantState cst{};
  // optional workspace for split K (per-tensor scales, bf16 output only)
  void* ws = nullptr;
  int64_t ws_bytes = 0;
  // MX scaling (block_scaled false): UE8M0 scale atoms of A and B; sa, sb unused
  bool mx = false;
  const uint8_t* sfa8 = nullptr;
  const uint8_t* sfb8 = nullptr;
  // operands stored contraction-major: A as [K, M] (lda >= M) and B as [K, N] (ldb >= N),
  // row-major, read MN-major (per-tensor scales, bf16 output only)
  bool mn = false;
};
// Returns cudaSuccess, or an error; `why` receives a static message for host-side failures.
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream, const char** why);
// Workspace bytes a split-K launch of this per-tensor problem uses (0: it would not split).
int64_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Two independent per-tensor GEMMs (bf16 outputs) in one persistent launch; ws (optional,
// gemm_group_workspace_bytes long, zero-filled once) lets them split K.
cudaError_t launch_gemm_group(const GemmArgs& g0, const GemmArgs& g1, void* ws, int64_t ws_bytes,
                              cudaStream_t stream, const char** why);
int64_t gemm_group_workspace_bytes(const GemmArgs& g0, const GemmArgs& g1);

}  // namespace fp8gb
