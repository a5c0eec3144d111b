// api.cu -- the C ABI declared in include/fp8gb.h: argument validation, the order of
// launches of each entry point, and the device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fp8gb.h"
#include "kernels.h"

namespace fp8gb {

// Bit set by any bounded wait that ran out (one word per device that loads the library).
__device__ uint32_t g_device_error_word;

namespace {

thread_local char g_detail[512] = "";
std::atomic<unsigned long long> g_wait_limit_ns{4000000000ull};

fp8_status_t fail(fp8_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return s;
}

fp8_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(FP8_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDev = 64;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

QuantState to_qs(const fp8_tensor_state_t* st) {
  QuantState q{};
  if (st != nullptr) {
    q.hist = st->amax_history;
    q.hist_count = st->hist_count;
    q.scale = st->scale;
    q.scale_inv = st->scale_inv;
    q.amax_cur = st->amax_cur;
    q.counters = st->counters;
    q.hist_len = st->hist_len;
  }
  return q;
}

fp8_status_t check_state(const fp8_tensor_state_t* st, fp8_scaling_t mode, const char* who) {
  if (st == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: scaling state is required", who);
  if (!st->scale || !st->scale_inv || !st->amax_cur || !st->counters)
    return fail(FP8_ERR_INVALID_ARG, "%s: state has a null scale, scale_inv, amax_cur or counters", who);
  if (mode == FP8_SCALE_DELAYED && (!st->amax_history || !st->hist_count || st->hist_len <= 0))
    return fail(FP8_ERR_INVALID_ARG, "%s: delayed scaling needs amax_history, hist_count and hist_len > 0", who);
  return FP8_OK;
}

}  // namespace

int num_sms() {
  static int cache[kMaxDev] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDev) return 148;
  if (cache[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
    cache[d] = n;
  }
  return cache[d];
}

WaitCtl wait_ctl() {
  static uint32_t* ptr[kMaxDev] = {};
  static std::mutex mu;
  const int d = current_device();
  WaitCtl w{nullptr, g_wait_limit_ns.load()};
  if (d < 0 || d >= kMaxDev) return w;
  std::lock_guard<std::mutex> lk(mu);
  if (ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) == cudaSuccess) ptr[d] = static_cast<uint32_t*>(p);
  }
  w.err = ptr[d];
  return w;
}

}  // namespace fp8gb

using namespace fp8gb;

namespace {

// 128 x 128 tiles of a [rows, cols] tensor (the tiled kernels index them in 32 bits).
int64_t tile_count(int64_t rows, int64_t cols) { return ((rows + 127) / 128) * ((cols + 127) / 128); }

fp8_status_t validate_common(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, const char* who) {
  if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_INVALID_ARG, "%s: unknown format %d", who, fmt);
  if (rows * cols > 0 && x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: null input", who);
  if (ld < cols) return fail(FP8_ERR_INVALID_ARG, "%s: ld (%lld) < cols (%lld)", who, (long long)ld, (long long)cols);
  if (rows > (1ll << 31) || cols > (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: dimension beyond 2^31", who);
  return FP8_OK;
}

// MX scales: groups of 32 along the contraction dimension, which runs along x's rows (q given:
// activations [M, K]) or down its columns (qT given: a weight [K, N], written transposed).
fp8_status_t quantize_mx_impl(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format_t fmt,
                              fp8_scaling_t mode, const fp8_tensor_state_t* st, void* q, void* qT, float* sf,
                              cudaStream_t stream) {
  const char* who = "fp8_quantize (MX)";
  if (mode != FP8_SCALE_CURRENT) return fail(FP8_ERR_UNSUPPORTED, "%s: MX scales use current scaling", who);
  if ((q == nullptr) == (qT == nullptr))
    return fail(FP8_ERR_INVALID_ARG, "%s: exactly one of q_out (groups along rows) and qT_out (groups down columns)", who);
  if (sf == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: the scale buffer is required", who);
  if (!aligned16(x) || !aligned16(q) || !aligned16(qT) || !aligned16(sf))
    return fail(FP8_ERR_ALIGNMENT, "%s: x, the codes and the scale buffer must be 16-byte aligned", who);
  if (ld % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: ld %% 8 == 0", who);
  const bool down = qT != nullptr;
  const int64_t kdim = down ? rows : cols;
  if (kdim % 128 != 0)
    return fail(FP8_ERR_UNSUPPORTED, "%s: the contraction dimension (%s) must be a multiple of 128", who,
                down ? "rows" : "cols");
  if (down && cols % 8 != 0) return fail(FP8_ERR_UNSUPPORTED, "%s: with qT_out, cols %% 8 == 0", who);
  if (down && rows / 128 > 65535) return fail(FP8_ERR_UNSUPPORTED, "%s: more than 65535 row blocks", who);
  if (!down && ((rows + 127) / 128) * 128 * (cols / 128) > INT32_MAX)
    return fail(FP8_ERR_UNSUPPORTED, "%s: more than 2^31 tiles", who);
  if (rows * cols == 0) return FP8_OK;
  cudaError_t e;
  if (st != nullptr && st->amax_cur != nullptr) {
    if ((e = cudaMemsetAsync(st->amax_cur, 0, sizeof(float), stream)) != cudaSuccess) return cuda_fail(e, who);
  }
  e = launch_cast_mx(fmt, down, x, rows, cols, ld, down ? qT : q, sf, to_qs(st), stream);
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, "MX cast kernel");
}

fp8_status_t quantize_impl(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format_t fmt, fp8_gran_t gran,
                           fp8_scaling_t mode, const fp8_tensor_state_t* st, void* q, void* qT, float* unit_si,
                           cudaStream_t stream) {
  const char* who = "fp8_quantize";
  fp8_status_t s = validate_common(x, rows, cols, ld, fmt, who);
  if (s != FP8_OK) return s;
  if (gran != FP8_GRAN_TENSOR && gran != FP8_GRAN_TILE_1x128 && gran != FP8_GRAN_BLOCK_128x128 &&
      gran != FP8_GRAN_MX_1x32)
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown granularity %d", who, (int)gran);
  if (gran == FP8_GRAN_MX_1x32) return quantize_mx_impl(x, rows, cols, ld, fmt, mode, st, q, qT, unit_si, stream);
  if (mode != FP8_SCALE_CURRENT && mode != FP8_SCALE_DELAYED)
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown scaling mode %d", who, (int)mode);
  const int64_t n = rows * cols;
  if (n > 0 && q == nullptr && qT == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output", who);
  if (!aligned16(x) || !aligned16(q) || !aligned16(qT))
    return fail(FP8_ERR_ALIGNMENT, "%s: x, q_out and qT_out must be 16-byte aligned", who);
  const bool contiguous = (ld == cols);
  const bool tiled = (qT != nullptr) || gran != FP8_GRAN_TENSOR;
  if (gran == FP8_GRAN_TILE_1x128 && n > 0 && ld % 8 != 0)
    return fail(FP8_ERR_UNSUPPORTED, "%s: 1x128 tiles need ld %% 8 == 0", who);
  if (tiled && gran != FP8_GRAN_TILE_1x128 && n > 0) {
    if (cols % 8 != 0 || ld % 8 != 0 || rows % 8 != 0)
      return fail(FP8_ERR_UNSUPPORTED, "%s: this layout needs rows, cols and ld multiples of 8", who);
    if (qT != nullptr && rows % 16 != 0)
      return fail(FP8_ERR_UNSUPPORTED, "%s: the transposed output needs rows %% 16 == 0", who);
    if (tile_count(rows, cols) > INT32_MAX) return fail(FP8_ERR_UNSUPPORTED, "%s: more than 2^31 tiles", who);
  }
  const QuantState qs = to_qs(st);
  cudaError_t e = cudaSuccess;

  if (gran == FP8_GRAN_TENSOR) {
    if ((s = check_state(st, mode, who)) != FP8_OK) return s;
    if (!tiled && !contiguous && n > 0 && q == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output", who);
    e = launch_quant_tensor(fmt, mode == FP8_SCALE_DELAYED, tiled && n > 0, x, rows, cols, ld, q, qT, qs, stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantise kernel");
    return FP8_OK;
  }

  if (mode != FP8_SCALE_CURRENT)
    return fail(FP8_ERR_UNSUPPORTED, "%s: tile and block scales support current scaling only", who);
  if (unit_si == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: unit_scale_inv is required", who);
  if (st != nullptr && st->amax_cur != nullptr) {
    if ((e = cudaMemsetAsync(st->amax_cur, 0, sizeof(float), stream)) != cudaSuccess) return cuda_fail(e, who);
  }
  if (gran == FP8_GRAN_TILE_1x128) {
    if (cols % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "%s: 1x128 tiles need cols %% 128 == 0", who);
    if (rows * (cols / 128) > INT32_MAX) return fail(FP8_ERR_UNSUPPORTED, "%s: more than 2^31 tiles", who);
    if (qT != nullptr) return fail(FP8_ERR_UNSUPPORTED, "%s: 1x128 tiles write no transposed copy", who);
    if (q == nullptr && n > 0) return fail(FP8_ERR_INVALID_ARG, "%s: q_out is required", who);
    if (n == 0) return FP8_OK;
    e = launch_cast_1x128(fmt, x, rows, cols, ld, q, unit_si, qs, stream);
  } else {
    if (rows % 128 != 0 || cols % 128 != 0)
      return fail(FP8_ERR_UNSUPPORTED, "%s: 128x128 blocks need rows and cols multiples of 128", who);
    if (rows / 128 > 65535) return fail(FP8_ERR_UNSUPPORTED, "%s: 128x128 blocks: more than 65535 block rows", who);
    if (n == 0) return FP8_OK;
    e = launch_cast_blocks(fmt, x, rows, cols, ld, q, qT, unit_si, qs, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "cast kernel");
  return FP8_OK;
}

fp8_status_t scaled_mm_impl(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, fp8_gran_t gran, const float* sa, const float* sb,
                            void* C, int64_t ldc, cudaStream_t stream, void* ws = nullptr, int64_t ws_bytes = 0,
                            const char* who = "fp8_scaled_mm") {
  if (M < 0 || N < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if ((fa != FP8_E4M3 && fa != FP8_E5M2) || (fb != FP8_E4M3 && fb != FP8_E5M2))
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown format", who);
  if (gran != FP8_GRAN_TENSOR && gran != FP8_GRAN_BLOCK_128x128 && gran != FP8_GRAN_MX_1x32)
    return fail(FP8_ERR_INVALID_ARG, "%s: granularity must be TENSOR, BLOCK_128x128 or MX_1x32", who);
  if (M == 0 || N == 0) return FP8_OK;
  if (C == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: null C", who);
  if (ldc < N) return fail(FP8_ERR_INVALID_ARG, "%s: ldc < N", who);
  if (!aligned16(C) || ldc % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: C must be 16-byte aligned, ldc %% 8 == 0", who);
  if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: size >= 2^31", who);
  if (K == 0) {
    cudaError_t e = cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, stream);
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, who);
  }
  if (A == nullptr || B == nullptr || sa == nullptr || sb == nullptr)
    return fail(FP8_ERR_INVALID_ARG, "%s: null A, B or scale", who);
  if (lda < K || ldb < K) return fail(FP8_ERR_INVALID_ARG, "%s: lda or ldb < K", who);
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0)
    return fail(FP8_ERR_ALIGNMENT, "%s: A and B must be 16-byte aligned with lda, ldb multiples of 16", who);
  if (gran == FP8_GRAN_BLOCK_128x128 && (K % 128 != 0 || N % 128 != 0))
    return fail(FP8_ERR_UNSUPPORTED, "%s: block scaling needs K and N multiples of 128", who);
  if (gran == FP8_GRAN_MX_1x32) {
    if (K % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "%s: MX scaling needs K %% 128 == 0", who);
    if (!aligned16(sa) || !aligned16(sb)) return fail(FP8_ERR_ALIGNMENT, "%s: MX scale buffers 16-byte aligned", who);
  }
  GemmArgs g{A, B, C, M, N, K, lda, ldb, ldc, (int)fa, (int)fb, sa, sb, gran == FP8_GRAN_BLOCK_128x128};
  if (gran == FP8_GRAN_MX_1x32) {
    g.mx = true;
    g.sfa8 = reinterpret_cast<const uint8_t*>(sa);
    g.sfb8 = reinterpret_cast<const uint8_t*>(sb);
  }
  if (ws != nullptr && gran == FP8_GRAN_TENSOR) {
    g.ws = ws;
    g.ws_bytes = ws_bytes;
  }
  const char* why = "launch";
  cudaError_t e = launch_gemm(g, stream, &why);
  if (e != cudaSuccess) return cuda_fail(e, why);
  return FP8_OK;
}

}  // namespace

extern "C" {

fp8_status_t fp8_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, fp8_format_t fmt,
                          fp8_gran_t gran, fp8_scaling_t mode, const fp8_tensor_state_t* st, void* q_out,
                          void* qT_out, float* unit_scale_inv, void* stream) {
  return quantize_impl(x_bf16, rows, cols, ld, fmt, gran, mode, st, q_out, qT_out, unit_scale_inv,
                       static_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_quantize_many(const fp8_quant_job_t* jobs, int32_t n, void* stream) {
  const char* who = "fp8_quantize_many";
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n < 1 || n > kMaxJobs || jobs == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: 1 to %d jobs", who, kMaxJobs);
  bool fused = true;
  int64_t total_tiles = 0;
  for (int i = 0; i < n; ++i) {
    const fp8_quant_job_t& jb = jobs[i];
    if (jb.st == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: job %d: state is required", who, i);
    for (int k = 0; k < i; ++k)
      if (jobs[k].st->amax_cur == jb.st->amax_cur) return fail(FP8_ERR_INVALID_ARG, "%s: job %d: state repeated", who, i);
    fp8_status_t st = validate_common(jb.x_bf16, jb.rows, jb.cols, jb.ld, jb.fmt, who);
    if (st != FP8_OK) return st;
    if (jb.mode != FP8_SCALE_CURRENT && jb.mode != FP8_SCALE_DELAYED)
      return fail(FP8_ERR_INVALID_ARG, "%s: job %d: unknown scaling mode", who, i);
    if ((st = check_state(jb.st, jb.mode, who)) != FP8_OK) return st;
    fused = fused && jb.fmt == jobs[0].fmt && jb.qT_out != nullptr && jb.rows > 0 && jb.cols > 0 && jb.rows % 16 == 0 &&
            jb.cols % 8 == 0 && jb.ld % 8 == 0 && aligned16(jb.x_bf16) && aligned16(jb.q_out) && aligned16(jb.qT_out);
    total_tiles += tile_count(jb.rows, jb.cols);
  }
  if (!fused || n == 1 || total_tiles > INT32_MAX) {  // one launch per job (each checked alone)
    for (int i = 0; i < n; ++i) {
      const fp8_quant_job_t& jb = jobs[i];
      const fp8_status_t st = quantize_impl(jb.x_bf16, jb.rows, jb.cols, jb.ld, jb.fmt, FP8_GRAN_TENSOR, jb.mode, jb.st,
                                            jb.q_out, jb.qT_out, nullptr, s);
      if (st != FP8_OK) return st;
    }
    return FP8_OK;
  }
  TileJobs tj{};
  tj.n = n;
  int64_t t0 = 0;
  for (int i = 0; i < n; ++i) {
    const fp8_quant_job_t& jb = jobs[i];
    TileJob& t = tj.j[i];
    t.x = static_cast<const uint16_t*>(jb.x_bf16);
    t.rows = jb.rows;
    t.cols = jb.cols;
    t.ld = jb.ld;
    t.q = static_cast<uint8_t*>(jb.q_out);
    t.qT = static_cast<uint8_t*>(jb.qT_out);
    t.st = to_qs(jb.st);
    t.delayed = jb.mode == FP8_SCALE_DELAYED ? 1 : 0;
    t.tiles_x = (jb.cols + 127) / 128;
    t.ntiles = t.tiles_x * ((jb.rows + 127) / 128);
    t.tile0 = t0;
    t0 += t.ntiles;
  }
  const cudaError_t e = launch_quant_many((int)jobs[0].fmt, tj, s);
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantise kernel");
}

fp8_status_t fp8_scaled_mm(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, fp8_gran_t gran, const float* scale_inv_a,
                           const float* scale_inv_b, void* C_bf16, int64_t ldc, void* stream) {
  return scaled_mm_impl(A, fa, B, fb, M, N, K, lda, ldb, gran, scale_inv_a, scale_inv_b, C_bf16, ldc,
                        static_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_scaled_mm_ws(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, fp8_gran_t gran, const float* scale_inv_a,
                              const float* scale_inv_b, void* C_bf16, int64_t ldc, void* workspace,
                              int64_t workspace_bytes, void* stream) {
  const char* who = "fp8_scaled_mm_ws";
  if (gran != FP8_GRAN_TENSOR) return fail(FP8_ERR_UNSUPPORTED, "%s: per-tensor scales only", who);
  if (workspace_bytes < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative workspace size", who);
  if (workspace != nullptr && !aligned16(workspace))
    return fail(FP8_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", who);
  return scaled_mm_impl(A, fa, B, fb, M, N, K, lda, ldb, gran, scale_inv_a, scale_inv_b, C_bf16, ldc,
                        static_cast<cudaStream_t>(stream), workspace, workspace_bytes, who);
}

int64_t fp8_scaled_mm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (current_device() < 0) {
    fail(FP8_ERR_CUDA, "fp8_scaled_mm_workspace_bytes: no CUDA device");
    return -1;
  }
  return gemm_workspace_bytes(M, N, K);
}

fp8_status_t fp8_scaled_mm_quant(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M,
                                 int64_t N, int64_t K, int64_t lda, int64_t ldb, const float* scale_inv_a,
                                 const float* scale_inv_b, void* C_bf16, int64_t ldc, fp8_format_t fc,
                                 const fp8_tensor_state_t* c_st, void* Cq, void* stream) {
  const char* who = "fp8_scaled_mm_quant";
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fc != FP8_E4M3 && fc != FP8_E5M2) return fail(FP8_ERR_INVALID_ARG, "%s: unknown output format", who);
  fp8_status_t st = check_state(c_st, FP8_SCALE_DELAYED, who);
  if (st != FP8_OK) return st;
  if (M < 0 || N < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if (M == 0 || N == 0) return FP8_OK;
  if (C_bf16 == nullptr || Cq == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: C_bf16 and Cq are required", who);
  if (!aligned16(Cq) || N % 16 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: Cq 16-byte aligned, N %% 16 == 0", who);
  if (K == 0) return fail(FP8_ERR_UNSUPPORTED, "%s: K must be positive", who);
  // the same checks as fp8_scaled_mm (per-tensor scales)
  if ((fa != FP8_E4M3 && fa != FP8_E5M2) || (fb != FP8_E4M3 && fb != FP8_E5M2))
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown format", who);
  if (ldc < N) return fail(FP8_ERR_INVALID_ARG, "%s: ldc < N", who);
  if (!aligned16(C_bf16) || ldc % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: C 16-byte aligned, ldc %% 8 == 0", who);
  if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: size >= 2^31", who);
  if (A == nullptr || B == nullptr || scale_inv_a == nullptr || scale_inv_b == nullptr)
    return fail(FP8_ERR_INVALID_ARG, "%s: null A, B or scale", who);
  if (lda < K || ldb < K) return fail(FP8_ERR_INVALID_ARG, "%s: lda or ldb < K", who);
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0)
    return fail(FP8_ERR_ALIGNMENT, "%s: A and B must be 16-byte aligned with lda, ldb multiples of 16", who);
  // delayed scaling: the epilogue (or, before the history holds an entry, the bootstrap cast)
  // adds the output's amax to amax_cur, the running maximum since the last history commit
  cudaError_t e;
  GemmArgs g{A, B, C_bf16, M, N, K, lda, ldb, ldc, (int)fa, (int)fb, scale_inv_a, scale_inv_b, false};
  g.qf = (int)fc;
  g.Cq = Cq;
  g.ldcq = N;
  g.cst = to_qs(c_st);
  const char* why = "launch";
  e = launch_gemm(g, s, &why);
  if (e != cudaSuccess) return cuda_fail(e, why);
  e = launch_quant_tensor_if_empty_history((int)fc, C_bf16, M, N, ldc, Cq, g.cst, s);
  if (e != cudaSuccess) return cuda_fail(e, "bootstrap cast of the FP8 output");
  return FP8_OK;
}

fp8_status_t fp8_requantize_weights(const void* w_master_bf16, int64_t K, int64_t N, fp8_gran_t gran,
                                    fp8_scaling_t mode, const fp8_tensor_state_t* st, void* wq_kn, void* wqT_nk,
                                    float* block_scale_inv, void* stream) {
  if (gran == FP8_GRAN_TILE_1x128)
    return fail(FP8_ERR_INVALID_ARG, "fp8_requantize_weights: weights take TENSOR, BLOCK_128x128 or MX_1x32 scales");
  if (gran == FP8_GRAN_MX_1x32 && wq_kn != nullptr)
    return fail(FP8_ERR_UNSUPPORTED, "fp8_requantize_weights: MX weights are written transposed only (wqT_nk)");
  if (wq_kn == nullptr && wqT_nk == nullptr && K * N > 0)
    return fail(FP8_ERR_INVALID_ARG, "fp8_requantize_weights: no output");
  return quantize_impl(w_master_bf16, K, N, N, FP8_E4M3, gran, mode, st, wq_kn, wqT_nk, block_scale_inv,
                       static_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_update_requantize_weights(void* w_master_bf16, const float* delta, int64_t K, int64_t N,
                                           fp8_scaling_t mode, const fp8_tensor_state_t* st, void* wq_kn,
                                           void* wqT_nk, void* stream) {
  const char* who = "fp8_update_requantize_weights";
  if (K < 0 || N < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if (mode != FP8_SCALE_CURRENT && mode != FP8_SCALE_DELAYED)
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown scaling mode %d", who, (int)mode);
  fp8_status_t s = check_state(st, mode, who);
  if (s != FP8_OK) return s;
  if (K * N == 0) return quantize_impl(w_master_bf16, K, N, N, FP8_E4M3, FP8_GRAN_TENSOR, mode, st, wq_kn, wqT_nk,
                                       nullptr, static_cast<cudaStream_t>(stream));
  if (w_master_bf16 == nullptr || delta == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: null W or delta", who);
  if (wq_kn == nullptr && wqT_nk == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: no output", who);
  if (!aligned16(w_master_bf16) || !aligned16(delta) || !aligned16(wq_kn) || !aligned16(wqT_nk))
    return fail(FP8_ERR_ALIGNMENT, "%s: W, delta and the caches must be 16-byte aligned", who);
  if (K % 8 != 0 || N % 8 != 0 || (wqT_nk != nullptr && K % 16 != 0))
    return fail(FP8_ERR_UNSUPPORTED, "%s: K and N must be multiples of 8 (K of 16 with wqT)", who);
  if (K > (1ll << 31) || N > (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: dimension beyond 2^31", who);
  if (tile_count(K, N) > INT32_MAX) return fail(FP8_ERR_UNSUPPORTED, "%s: more than 2^31 tiles", who);
  cudaError_t e = launch_update_quant_tensor(mode == FP8_SCALE_DELAYED, w_master_bf16, delta, K, N, wq_kn, wqT_nk,
                                             to_qs(st), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, who);
}

fp8_status_t fp8_linear_fwd(const void* x_bf16, int64_t M, int64_t K, int64_t N, const void* wqT_nk,
                            const fp8_tensor_state_t* w_st, const float* w_block_scale_inv,
                            const fp8_tensor_state_t* x_st, fp8_gran_t gran, fp8_scaling_t mode, void* xq_save,
                            void* xqT_save, float* x_tile_scale_inv, void* y_bf16, void* stream) {
  const char* who = "fp8_linear_fwd";
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M < 0 || K < 0 || N < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  // a buffer may be null only when it holds no elements (an empty token batch)
  if ((xq_save == nullptr && M * K > 0) || (y_bf16 == nullptr && M * N > 0) || (wqT_nk == nullptr && N * K > 0))
    return fail(FP8_ERR_INVALID_ARG, "%s: xq_save, y and wqT are required", who);
  fp8_status_t st;
  if (gran == FP8_GRAN_TENSOR) {
    if (w_st == nullptr || w_st->scale_inv == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: w_st->scale_inv is required", who);
    if (x_st == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: x_st is required", who);
    st = quantize_impl(x_bf16, M, K, K, FP8_E4M3, FP8_GRAN_TENSOR, mode, x_st, xq_save, xqT_save, nullptr, s);
    if (st != FP8_OK) return st;
    return scaled_mm_impl(xq_save, FP8_E4M3, wqT_nk, FP8_E4M3, M, N, K, K, K, FP8_GRAN_TENSOR, x_st->scale_inv,
                          w_st->scale_inv, y_bf16, N, s);
  }
  if (gran == FP8_GRAN_BLOCK_128x128) {
    if (mode != FP8_SCALE_CURRENT) return fail(FP8_ERR_UNSUPPORTED, "%s: block scaling uses current scaling", who);
    if (xqT_save != nullptr) return fail(FP8_ERR_UNSUPPORTED, "%s: no transposed copy with 1x128 tiles", who);
    if (w_block_scale_inv == nullptr || x_tile_scale_inv == nullptr)
      return fail(FP8_ERR_INVALID_ARG, "%s: block scaling needs w_block_scale_inv and x_tile_scale_inv", who);
    st = quantize_impl(x_bf16, M, K, K, FP8_E4M3, FP8_GRAN_TILE_1x128, FP8_SCALE_CURRENT, x_st, xq_save, nullptr,
                       x_tile_scale_inv, s);
    if (st != FP8_OK) return st;
    return scaled_mm_impl(xq_save, FP8_E4M3, wqT_nk, FP8_E4M3, M, N, K, K, K, FP8_GRAN_BLOCK_128x128,
                          x_tile_scale_inv, w_block_scale_inv, y_bf16, N, s);
  }
  if (gran == FP8_GRAN_MX_1x32) {
    if (mode != FP8_SCALE_CURRENT) return fail(FP8_ERR_UNSUPPORTED, "%s: MX scaling uses current scaling", who);
    if (xqT_save != nullptr) return fail(FP8_ERR_UNSUPPORTED, "%s: no transposed copy with MX scales", who);
    if (w_block_scale_inv == nullptr || x_tile_scale_inv == nullptr)
      return fail(FP8_ERR_INVALID_ARG, "%s: MX scaling needs the scale buffers of W and x", who);
    st = quantize_impl(x_bf16, M, K, K, FP8_E4M3, FP8_GRAN_MX_1x32, FP8_SCALE_CURRENT, x_st, xq_save, nullptr,
                       x_tile_scale_inv, s);
    if (st != FP8_OK) return st;
    return scaled_mm_impl(xq_save, FP8_E4M3, wqT_nk, FP8_E4M3, M, N, K, K, K, FP8_GRAN_MX_1x32, x_tile_scale_inv,
                          w_block_scale_inv, y_bf16, N, s);
  }
  return fail(FP8_ERR_INVALID_ARG, "%s: granularity must be TENSOR, BLOCK_128x128 or MX_1x32", who);
}

}  // extern "C"

namespace {

// C [M,N] = A^T B with A [K, M] and B [K, N] row-major, read MN-major (per-tensor scales).
fp8_status_t scaled_mm_t_impl(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, const float* sa, const float* sb, void* C,
                              int64_t ldc, void* ws, int64_t ws_bytes, cudaStream_t stream, const char* who) {
  if (M < 0 || N < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if ((fa != FP8_E4M3 && fa != FP8_E5M2) || (fb != FP8_E4M3 && fb != FP8_E5M2))
    return fail(FP8_ERR_INVALID_ARG, "%s: unknown format", who);
  if (ws_bytes < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative workspace size", who);
  if (ws != nullptr && !aligned16(ws)) return fail(FP8_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", who);
  if (M == 0 || N == 0) return FP8_OK;
  if (C == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: null C", who);
  if (ldc < N) return fail(FP8_ERR_INVALID_ARG, "%s: ldc < N", who);
  if (!aligned16(C) || ldc % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: C must be 16-byte aligned, ldc %% 8 == 0", who);
  if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: size >= 2^31", who);
  if (K == 0) {
    cudaError_t e = cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, stream);
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, who);
  }
  if (A == nullptr || B == nullptr || sa == nullptr || sb == nullptr)
    return fail(FP8_ERR_INVALID_ARG, "%s: null A, B or scale", who);
  if (lda < M || ldb < N) return fail(FP8_ERR_INVALID_ARG, "%s: lda < M or ldb < N", who);
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0)
    return fail(FP8_ERR_ALIGNMENT, "%s: A and B must be 16-byte aligned with lda, ldb multiples of 16", who);
  GemmArgs g{A, B, C, M, N, K, lda, ldb, ldc, (int)fa, (int)fb, sa, sb, false};
  g.mn = true;
  g.ws = ws;
  g.ws_bytes = ws != nullptr ? ws_bytes : 0;
  const char* why = "launch";
  cudaError_t e = launch_gemm(g, stream, &why);
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, why);
}

// Checks of fp8_scaled_mm for one problem of a grouped call (per-tensor scales, M, N, K > 0).
fp8_status_t check_group_problem(const fp8_mm_problem_t& q, int i, const char* who) {
  if ((q.fa != FP8_E4M3 && q.fa != FP8_E5M2) || (q.fb != FP8_E4M3 && q.fb != FP8_E5M2))
    return fail(FP8_ERR_INVALID_ARG, "%s: problem %d: unknown format", who, i);
  if (q.M <= 0 || q.N <= 0 || q.K <= 0) return fail(FP8_ERR_INVALID_ARG, "%s: problem %d: M, N, K must be positive", who, i);
  if (q.M >= (1ll << 31) || q.N >= (1ll << 31) || q.K >= (1ll << 31))
    return fail(FP8_ERR_UNSUPPORTED, "%s: problem %d: size >= 2^31", who, i);
  if (q.A == nullptr || q.B == nullptr || q.C_bf16 == nullptr || q.scale_inv_a == nullptr || q.scale_inv_b == nullptr)
    return fail(FP8_ERR_INVALID_ARG, "%s: problem %d: null A, B, C or scale", who, i);
  if (q.mn_major != 0 && q.mn_major != 1) return fail(FP8_ERR_INVALID_ARG, "%s: problem %d: mn_major is 0 or 1", who, i);
  if (q.mn_major ? (q.lda < q.M || q.ldb < q.N || q.ldc < q.N) : (q.lda < q.K || q.ldb < q.K || q.ldc < q.N))
    return fail(FP8_ERR_INVALID_ARG, "%s: problem %d: leading dimension too small", who, i);
  if (!aligned16(q.A) || !aligned16(q.B) || !aligned16(q.C_bf16) || q.lda % 16 || q.ldb % 16 || q.ldc % 8)
    return fail(FP8_ERR_ALIGNMENT, "%s: problem %d: A, B, C 16-byte aligned, lda and ldb multiples of 16, ldc of 8",
                who, i);
  return FP8_OK;
}

GemmArgs group_args(const fp8_mm_problem_t& q) {
  GemmArgs g{q.A, q.B, q.C_bf16, q.M, q.N, q.K, q.lda, q.ldb, q.ldc, (int)q.fa, (int)q.fb,
             q.scale_inv_a, q.scale_inv_b, false};
  g.mn = q.mn_major == 1;
  return g;
}

fp8_status_t grouped_impl(const fp8_mm_problem_t* pr, int32_t n, void* ws, int64_t ws_bytes, cudaStream_t s,
                          const char* who) {
  if (n < 1 || n > 2 || pr == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: 1 or 2 problems", who);
  if (ws_bytes < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative workspace size", who);
  if (ws != nullptr && !aligned16(ws)) return fail(FP8_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", who);
  for (int i = 0; i < n; ++i) {
    const fp8_status_t st = check_group_problem(pr[i], i, who);
    if (st != FP8_OK) return st;
  }
  if (n == 1 && pr[0].mn_major)
    return scaled_mm_t_impl(pr[0].A, pr[0].fa, pr[0].B, pr[0].fb, pr[0].M, pr[0].N, pr[0].K, pr[0].lda, pr[0].ldb,
                            pr[0].scale_inv_a, pr[0].scale_inv_b, pr[0].C_bf16, pr[0].ldc, ws, ws_bytes, s, who);
  if (n == 1)
    return scaled_mm_impl(pr[0].A, pr[0].fa, pr[0].B, pr[0].fb, pr[0].M, pr[0].N, pr[0].K, pr[0].lda, pr[0].ldb,
                          FP8_GRAN_TENSOR, pr[0].scale_inv_a, pr[0].scale_inv_b, pr[0].C_bf16, pr[0].ldc, s, ws,
                          ws_bytes, who);
  const char* why = "launch";
  const cudaError_t e = launch_gemm_group(group_args(pr[0]), group_args(pr[1]), ws, ws_bytes, s, &why);
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, why);
}

// The backward pass. mn: wgrad reads x's codes xq [M, K] and dy's codes dyq [M, N] as they are
// (MN-major; xqT_save then holds xq and dyqT_ws is unused); otherwise xqT_save [K, M] and
// dyqT_ws [N, M] are the transposed copies.
fp8_status_t linear_bwd_impl(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xqT_save,
                             const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                             fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dyqT_ws, void* dx_bf16,
                             void* dw_bf16, void* ws, int64_t ws_bytes, cudaStream_t s, const char* who,
                             bool mn = false) {
  if (M < 0 || K < 0 || N < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if (M % 16 || K % 16 || N % 16) return fail(FP8_ERR_UNSUPPORTED, "%s: M, K and N must be multiples of 16", who);
  // a buffer may be null only when it holds no elements (an empty token batch)
  if (dyq_ws == nullptr && M * N > 0) return fail(FP8_ERR_INVALID_ARG, "%s: dyq_ws is required", who);
  if (dw_bf16 != nullptr && ((!mn && dyqT_ws == nullptr && M * N > 0) || (xqT_save == nullptr && M * K > 0) ||
                             x_st == nullptr || !x_st->scale_inv))
    return fail(FP8_ERR_INVALID_ARG, "%s: wgrad needs %s and x_st", who, mn ? "xq_save" : "dyqT_ws, xqT_save");
  if (dx_bf16 != nullptr && (wq_kn == nullptr || w_st == nullptr || !w_st->scale_inv))
    return fail(FP8_ERR_INVALID_ARG, "%s: dgrad needs wq_kn and w_st", who);
  if (ws_bytes < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative workspace size", who);
  if (ws != nullptr && !aligned16(ws)) return fail(FP8_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", who);
  fp8_status_t st = quantize_impl(dy_bf16, M, N, N, FP8_E5M2, FP8_GRAN_TENSOR, mode, dy_st, dyq_ws,
                                  (dw_bf16 != nullptr && !mn) ? dyqT_ws : nullptr, nullptr, s);
  if (st != FP8_OK) return st;
  if (mn && M > 0 && K > 0 && N > 0) {
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: size >= 2^31", who);
    if ((dw_bf16 != nullptr && (!aligned16(xqT_save) || !aligned16(dw_bf16))) ||
        (dx_bf16 != nullptr && (!aligned16(wq_kn) || !aligned16(dx_bf16))) || !aligned16(dyq_ws))
      return fail(FP8_ERR_ALIGNMENT, "%s: codes and outputs must be 16-byte aligned", who);
    // wgrad dW [K,N] = xq^T dyq: A = xq as [M, K] (contraction M, K contiguous), B = dyq as [M, N]
    GemmArgs gw{xqT_save, dyq_ws, dw_bf16, K, N, M, K, N, N, (int)FP8_E4M3, (int)FP8_E5M2,
                dw_bf16 != nullptr ? x_st->scale_inv : nullptr, dy_st->scale_inv, false};
    gw.mn = true;
    GemmArgs gd{dyq_ws, wq_kn, dx_bf16, M, K, N, N, N, K, (int)FP8_E5M2, (int)FP8_E4M3, dy_st->scale_inv,
                dx_bf16 != nullptr ? w_st->scale_inv : nullptr, false};
    const char* why = "launch";
    cudaError_t e = cudaSuccess;
    if (dx_bf16 != nullptr && dw_bf16 != nullptr) {
      e = launch_gemm_group(gw, gd, ws, ws != nullptr ? ws_bytes : 0, s, &why);
    } else if (dw_bf16 != nullptr) {
      gw.ws = ws;
      gw.ws_bytes = ws != nullptr ? ws_bytes : 0;
      e = launch_gemm(gw, s, &why);
    } else if (dx_bf16 != nullptr) {
      return scaled_mm_impl(dyq_ws, FP8_E5M2, wq_kn, FP8_E4M3, M, K, N, N, N, FP8_GRAN_TENSOR, dy_st->scale_inv,
                            w_st->scale_inv, dx_bf16, K, s, ws, ws_bytes, who);
    }
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, why);
  }
  if (M == 0 || K == 0 || N == 0) {
    // an empty contraction writes zeros; empty outputs write nothing
    if (dx_bf16 != nullptr && (st = scaled_mm_impl(dyq_ws, FP8_E5M2, wq_kn, FP8_E4M3, M, K, N, N, N, FP8_GRAN_TENSOR,
                                                   dy_st->scale_inv, w_st->scale_inv, dx_bf16, K, s)) != FP8_OK)
      return st;
    if (dw_bf16 != nullptr)
      return scaled_mm_impl(xqT_save, FP8_E4M3, dyqT_ws, FP8_E5M2, K, N, M, M, M, FP8_GRAN_TENSOR, x_st->scale_inv,
                            dy_st->scale_inv, dw_bf16, N, s);
    return FP8_OK;
  }
  if (dx_bf16 != nullptr && dw_bf16 != nullptr) {
    // dgrad and wgrad in one persistent launch: neither alone fills the GPU at training
    // shapes, and the pair share the dy codes. The checks fp8_scaled_mm would make:
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31))
      return fail(FP8_ERR_UNSUPPORTED, "%s: size >= 2^31", who);
    if (!aligned16(dyq_ws) || !aligned16(dyqT_ws) || !aligned16(xqT_save) || !aligned16(wq_kn) || !aligned16(dx_bf16) ||
        !aligned16(dw_bf16))
      return fail(FP8_ERR_ALIGNMENT, "%s: codes and outputs must be 16-byte aligned", who);
    const fp8_mm_problem_t pr[2] = {
        {xqT_save, FP8_E4M3, dyqT_ws, FP8_E5M2, K, N, M, M, M, x_st->scale_inv, dy_st->scale_inv, dw_bf16, N},
        {dyq_ws, FP8_E5M2, wq_kn, FP8_E4M3, M, K, N, N, N, dy_st->scale_inv, w_st->scale_inv, dx_bf16, K}};
    return grouped_impl(pr, 2, ws, ws_bytes, s, who);
  }
  if (dx_bf16 != nullptr)
    return scaled_mm_impl(dyq_ws, FP8_E5M2, wq_kn, FP8_E4M3, M, K, N, N, N, FP8_GRAN_TENSOR, dy_st->scale_inv,
                          w_st->scale_inv, dx_bf16, K, s, ws, ws_bytes, who);
  if (dw_bf16 != nullptr)
    return scaled_mm_impl(xqT_save, FP8_E4M3, dyqT_ws, FP8_E5M2, K, N, M, M, M, FP8_GRAN_TENSOR, x_st->scale_inv,
                          dy_st->scale_inv, dw_bf16, N, s, ws, ws_bytes, who);
  return FP8_OK;
}

}  // namespace

extern "C" {

fp8_status_t fp8_linear_bwd(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xqT_save,
                            const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                            fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dyqT_ws, void* dx_bf16,
                            void* dw_bf16, void* stream) {
  return linear_bwd_impl(dy_bf16, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, dyqT_ws, dx_bf16, dw_bf16,
                         nullptr, 0, static_cast<cudaStream_t>(stream), "fp8_linear_bwd");
}

fp8_status_t fp8_linear_bwd_ws(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xqT_save,
                               const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                               fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dyqT_ws,
                               void* dx_bf16, void* dw_bf16, void* workspace, int64_t workspace_bytes, void* stream) {
  return linear_bwd_impl(dy_bf16, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, dyqT_ws, dx_bf16, dw_bf16,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream), "fp8_linear_bwd_ws");
}

fp8_status_t fp8_linear_bwd_mn(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xq_save,
                               const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                               fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dx_bf16, void* dw_bf16,
                               void* workspace, int64_t workspace_bytes, void* stream) {
  const char* who = "fp8_linear_bwd_mn";
  if (workspace_bytes < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative workspace size", who);
  if (workspace != nullptr && !aligned16(workspace))
    return fail(FP8_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", who);
  return linear_bwd_impl(dy_bf16, M, K, N, xq_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, nullptr, dx_bf16, dw_bf16,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream), who, true);
}

fp8_status_t fp8_scaled_mm_t(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                             int64_t K, int64_t lda, int64_t ldb, const float* scale_inv_a, const float* scale_inv_b,
                             void* C_bf16, int64_t ldc, void* workspace, int64_t workspace_bytes, void* stream) {
  return scaled_mm_t_impl(A, fa, B, fb, M, N, K, lda, ldb, scale_inv_a, scale_inv_b, C_bf16, ldc, workspace,
                          workspace_bytes, static_cast<cudaStream_t>(stream), "fp8_scaled_mm_t");
}

int64_t fp8_linear_bwd_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (current_device() < 0) {
    fail(FP8_ERR_CUDA, "fp8_linear_bwd_workspace_bytes: no CUDA device");
    return -1;
  }
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  // only the shapes decide the size
  const GemmArgs gw{nullptr, nullptr, nullptr, K, N, M, M, M, N, (int)FP8_E4M3, (int)FP8_E5M2, nullptr, nullptr, false};
  const GemmArgs gd{nullptr, nullptr, nullptr, M, K, N, N, N, K, (int)FP8_E5M2, (int)FP8_E4M3, nullptr, nullptr, false};
  return gemm_group_workspace_bytes(gw, gd);
}

fp8_status_t fp8_scaled_mm_grouped(const fp8_mm_problem_t* problems, int32_t n, void* workspace,
                                   int64_t workspace_bytes, void* stream) {
  return grouped_impl(problems, n, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      "fp8_scaled_mm_grouped");
}

int64_t fp8_scaled_mm_grouped_workspace_bytes(const fp8_mm_problem_t* problems, int32_t n) {
  if (current_device() < 0) {
    fail(FP8_ERR_CUDA, "fp8_scaled_mm_grouped_workspace_bytes: no CUDA device");
    return -1;
  }
  if (n < 1 || n > 2 || problems == nullptr) {
    fail(FP8_ERR_INVALID_ARG, "fp8_scaled_mm_grouped_workspace_bytes: 1 or 2 problems");
    return -1;
  }
  if (n == 1) return gemm_workspace_bytes(problems[0].M, problems[0].N, problems[0].K);
  return gemm_group_workspace_bytes(group_args(problems[0]), group_args(problems[1]));
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free backward: fp8_linear_bwd with its dy-code scratch in a static array.
// ---------------------------------------------------------------------------------------
// The backward casts dy to E5M2 twice (row-major for dgrad, transposed for wgrad) before the
// two GEMMs read the codes. fp8_linear_bwd takes those two buffers from the caller; this
// array stands in for them. It lives in this file's device module beside the error word, so
// a device holds these 64 MiB from the first call that loads the module there (any GEMM
// launch or this entry point, under lazy loading) until the process exits.
static constexpr size_t kBwdScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_bwd_scratch[kBwdScratchBytes];

namespace {

// Device address of g_bwd_scratch on the current device. The name g_bwd_scratch in host
// code is only a host-side stand-in for the symbol, never a device pointer, so it is looked
// up once per device (with that device current) and cached.
uint8_t* bwd_scratch_address(fp8_status_t* status) {
  static uint8_t* addr[kMaxDev] = {};
  static std::mutex mu;
  const int d = current_device();
  if (d < 0 || d >= kMaxDev) {
    *status = fail(FP8_ERR_CUDA, "fp8_linear_bwd_noalloc: no usable current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (addr[d] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      *status = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                          "fp8_linear_bwd_noalloc: cudaGetSymbolAddress of the static scratch");
      return nullptr;
    }
    addr[d] = static_cast<uint8_t*>(ptr);
  }
  return addr[d];
}

}  // namespace

extern "C" {

fp8_status_t fp8_linear_bwd_noalloc(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xqT_save,
                                    const fp8_tensor_state_t* x_st, const void* wq_kn,
                                    const fp8_tensor_state_t* w_st, fp8_tensor_state_t* dy_st, fp8_scaling_t mode,
                                    void* dx_bf16, void* dw_bf16, void* stream) {
  const char* who = "fp8_linear_bwd_noalloc";
  if (M < 0 || K < 0 || N < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", who);
  if (M >= (1ll << 31) || N >= (1ll << 31)) return fail(FP8_ERR_UNSUPPORTED, "%s: dimension >= 2^31", who);
  // dy codes [M,N], then (for wgrad) the transposed codes [N,M] at the next 256-byte boundary
  const uint64_t codes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  const uint64_t t_off = (codes + 255u) & ~uint64_t(255);
  const uint64_t need = dw_bf16 != nullptr ? t_off + codes : codes;
  if (need > kBwdScratchBytes)
    return fail(FP8_ERR_UNSUPPORTED,
                "%s: dy [%lld x %lld] needs %llu bytes of scratch for its FP8 codes%s, more than the %llu-byte "
                "static array; use fp8_linear_bwd with caller-provided scratch",
                who, (long long)M, (long long)N, (unsigned long long)need, dw_bf16 != nullptr ? " and their transpose" : "",
                (unsigned long long)kBwdScratchBytes);
  fp8_status_t st = FP8_OK;
  uint8_t* base = bwd_scratch_address(&st);
  if (base == nullptr) return st;
  // Both regions are written in full by the dy cast before the GEMMs read them: nothing in
  // the array has to start at zero.
  return fp8_linear_bwd(dy_bf16, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, base,
                        dw_bf16 != nullptr ? base + t_off : nullptr, dx_bf16, dw_bf16, stream);
}

fp8_status_t fp8_history_commit(const fp8_tensor_state_t* st, void* stream) {
  return fp8_history_commit_many(st, 1, stream);
}

fp8_status_t fp8_history_commit_many(const fp8_tensor_state_t* states, int32_t n, void* stream) {
  const char* who = "fp8_history_commit";
  if (n < 0 || n > kMaxCommit) return fail(FP8_ERR_INVALID_ARG, "%s: 0 <= n <= %d states per call", who, kMaxCommit);
  if (n > 0 && states == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s: null states", who);
  QuantStates sts{};
  sts.n = n;
  for (int i = 0; i < n; ++i) {
    const fp8_tensor_state_t* st = states + i;
    if (!st->amax_history || !st->hist_count || !st->amax_cur || st->hist_len <= 0)
      return fail(FP8_ERR_INVALID_ARG, "%s: state %d needs amax_history, hist_count, amax_cur, hist_len > 0", who, i);
    for (int j = 0; j < i; ++j)
      if (states[j].hist_count == st->hist_count)
        return fail(FP8_ERR_INVALID_ARG, "%s: state %d appears twice in one call", who, i);
    sts.s[i] = to_qs(st);
  }
  if (n == 0) return FP8_OK;
  cudaError_t e = launch_history_commit(sts, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8_OK : cuda_fail(e, who);
}

fp8_status_t fp8_poll_device_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "fp8_poll_device_error");
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "fp8_poll_device_error");
  if (v == 0) return FP8_OK;
  const uint32_t zero = 0;
  cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
  return fail(FP8_ERR_TIMEOUT, "a bounded wait ran out (device error bits 0x%x)", v);
}

fp8_status_t fp8_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) return fail(FP8_ERR_INVALID_ARG, "fp8_set_wait_limit_ns: limit must be > 0");
  g_wait_limit_ns.store(ns);
  return FP8_OK;
}

fp8_status_t fp8_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  WaitCtl w = wait_ctl();
  if (w.err == nullptr) return fail(FP8_ERR_CUDA, "fp8_selftest_wait_timeout: no device error word");
  w.limit_ns = limit_ns;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_selftest_wait(w, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "fp8_selftest_wait_timeout");
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "fp8_selftest_wait_timeout");
  const uint32_t zero = 0;
  cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
  if (v & DEV_ERR_WAIT_SELFTEST) return fail(FP8_ERR_TIMEOUT, "self-test wait ran out as intended");
  return fail(FP8_ERR_CUDA, "self-test wait did not report a timeout (bits 0x%x)", v);
}

fp8_status_t fp8_get_last_error_detail(char* buf, size_t n) {
  if (buf != nullptr && n > 0) {
    strncpy(buf, g_detail, n - 1);
    buf[n - 1] = '\0';
  }
  return FP8_OK;
}

const char* fp8_status_string(fp8_status_t s) {
  switch (s) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
    case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
  }
  return "FP8_ERR_UNKNOWN";
}

}  // extern "C"
