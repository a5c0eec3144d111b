/*
 * fp8gb.h -- C ABI of the GB300 (sm_103a) FP8 up-projection library.
 *
 * The library implements FP8 training's quantise-then-scaled-matmul for a transformer
 * MLP up-projection y = x W (x [M,K], W [K,N], row-major bf16):
 *   - amax reductions that produce scales (per tensor, per 1x128 row tile, per 128x128
 *     block, or from an amax history for delayed scaling),
 *   - a saturating round-to-nearest-even cast of bf16 to E4M3 (max 448; forward
 *     activations and weights) or E5M2 (max 57344; gradients), with overflow and
 *     underflow counters,
 *   - FP8 x FP8 GEMMs on the tcgen05 tensor cores with fp32 accumulation and an epilogue
 *     that multiplies by the operands' inverse scales and writes bf16,
 *   - the forward, dgrad and wgrad compositions and the FP8 weight cache refresh.
 *
 * Sources (three web pages on FP8 mixed-precision training):
 *   [GUARD]  "FP8 stability guardrails" page (zenaique): section "Why FP8 is tempting and
 *            why it is fragile" (format maxima, overflow / saturation, underflow);
 *            "Real products, models, and research" (fine-grained tile / block scaling,
 *            delayed scaling with amax history); "What an interviewer would ask next"
 *            (E4M3 and E5M2 in one run).
 *   [SPEED]  "#84 FP8 Precision" speedrun page (bubblnet): "Explanation" (weights divided
 *            by a scale before the E4M3 cast; a scaled matmul with per-operand scales;
 *            operands laid out contiguous along the contraction), "Hardware precision"
 *            (bf16 master weights in the optimizer, FP8 compute copy re-quantised after
 *            every optimizer step; FP8 only for the MLP up-projection).
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library keeps no
 *     pointer after a call returns and allocates no device memory in any call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). All
 *     work is enqueued on it; no call synchronises the host except where stated.
 *   - Scales, amaxes and counters stay on the device (fp8_tensor_state_t), so a call
 *     never reads a device value back to the host.
 *   - Arguments are validated before anything is enqueued: null pointers, negative
 *     sizes, bad enums -> FP8_ERR_INVALID_ARG; shapes the kernels do not handle ->
 *     FP8_ERR_UNSUPPORTED; pointers or leading dimensions that break the 16-byte rule of
 *     the tensor-memory-accelerator copies -> FP8_ERR_ALIGNMENT. A CUDA error reported
 *     after a launch -> FP8_ERR_CUDA. fp8_get_last_error_detail() gives a message.
 *   - Matrices are row-major with a leading dimension `ld` (elements between rows).
 *   - Codes are stored one byte per element (uint8), as the formats' bit patterns.
 *   - No C++ exception crosses the boundary. There is no CPU fallback: without a
 *     suitable GPU every compute entry point returns FP8_ERR_CUDA or FP8_ERR_UNSUPPORTED.
 *   - Thread safety: calls are stateless apart from the caller's state structs and the
 *     per-thread error message; concurrent calls on different streams are safe when they
 *     touch disjoint caller buffers.
 */
#ifndef FP8GB_H
#define FP8GB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1,
  FP8_ERR_UNSUPPORTED = 2,
  FP8_ERR_ALIGNMENT = 3,
  FP8_ERR_CUDA = 4,
  FP8_ERR_TIMEOUT = 5
} fp8_status_t;

/* [GUARD] "Why FP8 is tempting...": E4M3 (4 exponent, 3 mantissa bits, max 448) and
 * E5M2 (5 exponent, 2 mantissa bits, max 57344). */
typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format_t;

/* [GUARD] "Real products...": per-tensor, fine-grained 1x128 tiles (one scale per row
 * and 128 consecutive columns) and 128x128 blocks, with fp32 scales; and MX units, the same
 * fine-grained idea on the tensor cores' own block scaling: one power-of-two scale per 32
 * consecutive elements along the contraction dimension, stored as a UE8M0 byte.
 *
 * MX scale layout (FP8_GRAN_MX_1x32). For an operand with MN rows (M for the GEMM's A, N
 * for its B) and contraction K (K % 128 == 0), the scale of MN index m and contraction
 * group g (elements 32 g .. 32 g + 31) is 2^e with e the smallest integer such that
 * FP8_MAX * 2^e >= the group's amax (so no element saturates; e = 0 for a zero or non-finite
 * amax; e >= -127), stored as the byte e + 127. The bytes form ceil(MN / 128) x (K / 128)
 * atoms of 512 bytes, atom (m / 128, g / 4) at byte offset ((m / 128) * (K / 128) + g / 4) * 512;
 * inside it the byte of (m, g) sits at 16 (m % 32) + 4 ((m / 32) % 4) + g % 4. Rows past the
 * last MN index up to a multiple of 128 hold e = 0. The buffer (ceil(MN/128) * K/128 * 512
 * bytes) is caller-owned and 16-byte aligned; it is passed through the `float*` scale
 * arguments of the entry points below, which then point to these bytes. */
typedef enum {
  FP8_GRAN_TENSOR = 0,
  FP8_GRAN_TILE_1x128 = 1,
  FP8_GRAN_BLOCK_128x128 = 2,
  FP8_GRAN_MX_1x32 = 3
} fp8_gran_t;

/* Current scaling takes the scale from this tensor's own amax; delayed scaling takes it
 * from the maximum of an amax history ([GUARD] "Real products...": delayed scaling with
 * amax history tracking). */
typedef enum { FP8_SCALE_CURRENT = 0, FP8_SCALE_DELAYED = 1 } fp8_scaling_t;

/* Scaling state of one tensor role (x, W or dy of one layer). Every pointer is caller-
 * owned device memory; zero-initialise amax_history, hist_count and counters once.
 *   amax_history [hist_len] fp32  ring of past amaxes (delayed scaling)
 *   hist_count   int32            number of amaxes pushed so far; the next push goes to
 *                                 amax_history[hist_count % hist_len]
 *   scale        fp32             s = FP8_MAX / amax_eff of the most recent cast
 *   scale_inv    fp32             d = amax_eff / FP8_MAX (what the GEMM multiplies by)
 *   amax_cur     fp32             delayed scaling: the running maximum of max |x| over the
 *                                 casts since the last history commit (which resets it to
 *                                 0); current scaling: max |x| of the most recent cast
 *   counters     uint64 [2]       [0] saturated elements, [1] non-zero elements flushed to
 *                                 zero; both accumulate until the caller clears them
 * If amax_eff is zero or not finite, s = d = 1. */
typedef struct {
  float* amax_history;
  int32_t* hist_count;
  float* scale;
  float* scale_inv;
  float* amax_cur;
  unsigned long long* counters;
  int32_t hist_len;
} fp8_tensor_state_t;

/* Quantise a bf16 matrix x [rows, cols] (leading dimension ld) to FP8 codes.
 *  [GUARD] "Why FP8 is tempting...": cast with saturation at +-FP8_MAX, round to nearest
 *  even, NaN -> 0x7F, sign of zero kept; [SPEED] "Explanation": the tensor is divided by
 *  its scale (multiplied by s = FP8_MAX / amax) before the cast.
 *  gran = FP8_GRAN_TENSOR: one scale for the whole tensor, from x's own amax (mode
 *    CURRENT; two passes over x) or from st's history (mode DELAYED; bootstrap with the
 *    current amax while hist_count == 0). `st` is required; the call writes st->scale and
 *    st->scale_inv, adds to st->counters, and sets st->amax_cur to x's amax (CURRENT) or
 *    raises it to x's amax when below (DELAYED; the bootstrap scale then comes from that
 *    running maximum). `unit_scale_inv` is ignored.
 *  gran = FP8_GRAN_TILE_1x128: cols % 128 == 0; one scale per (row, 128 columns), the
 *    inverse scales written to unit_scale_inv [rows, cols/128] (fp32, row-major). Mode
 *    must be CURRENT. `st` may be NULL; if given, st->amax_cur receives the tensor amax and
 *    the counters accumulate.
 *  gran = FP8_GRAN_BLOCK_128x128: rows % 128 == 0 and cols % 128 == 0; one scale per
 *    128x128 block, inverse scales in unit_scale_inv [rows/128, cols/128]. Mode CURRENT;
 *    `st` as for tiles.
 *  gran = FP8_GRAN_MX_1x32: mode CURRENT; unit_scale_inv receives the MX scale bytes (layout
 *    above). Exactly one of q_out and qT_out: with q_out the groups run along x's rows
 *    (activations: contraction = cols, cols % 128 == 0; codes [rows, cols], scales with
 *    MN = rows); with qT_out they run down its columns (a weight [K, N]: contraction = rows,
 *    rows % 128 == 0, cols % 8 == 0; codes written transposed [cols, rows], scales with
 *    MN = cols). `st` as for tiles. ld % 8 == 0.
 *  q_out [rows, cols] (leading dimension cols) receives the codes; may be NULL when
 *    qT_out is given. qT_out [cols, rows] (leading dimension rows) receives the transposed
 *    codes, or is NULL. With qT_out, rows % 16 == 0. With q_out and a GEMM consumer,
 *    cols % 16 == 0 is needed by the GEMM, not by this call.
 *  Alignment: x, q_out and qT_out 16-byte aligned; ld % 8 == 0 unless ld == cols.
 *  Size: rows, cols <= 2^31; with qT_out, tile or block scales, fewer than 2^31 units of
 *  128 x 128 (1 x 128 for tile scales); block scales at most 65535 block rows. Beyond these,
 *  FP8_ERR_UNSUPPORTED. */
fp8_status_t fp8_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                          fp8_format_t fmt, fp8_gran_t gran, fp8_scaling_t mode,
                          const fp8_tensor_state_t* st, void* q_out, void* qT_out,
                          float* unit_scale_inv, void* stream);

/* One tensor of fp8_quantize_many: the arguments of fp8_quantize with gran = FP8_GRAN_TENSOR. */
typedef struct {
  const void* x_bf16;
  int64_t rows, cols, ld;
  fp8_format_t fmt;
  fp8_scaling_t mode;
  const fp8_tensor_state_t* st;
  void* q_out;
  void* qT_out;
} fp8_quant_job_t;

/* n (1..4) per-tensor quantises, each exactly fp8_quantize(job, FP8_GRAN_TENSOR): when all
 * share one format, each writes its transposed copy (qT_out non-null) and rows, cols, ld are
 * multiples of 8 (rows of 16), they run as one cooperative launch whose grid shares their
 * tiles, so small tensors (a weight cache refresh next to an activation cast) pay one
 * launch's latency; otherwise one after the other. The pages have no such entry point: it is
 * [GUARD] "Real products..." per-tensor scaling applied to several tensors at once. Every job
 * obeys fp8_quantize's rules; the states must be distinct. */
fp8_status_t fp8_quantize_many(const fp8_quant_job_t* jobs, int32_t n, void* stream);

/* C [M,N] (bf16, leading dimension ldc) = dequantised A [M,K] times B [N,K] transposed:
 *   C_ij = bf16_rne( d_a * d_b * sum_k a_ik b_jk ),  fp32 accumulation.
 *  [SPEED] "Explanation": the scaled FP8 matmul with one scale per operand, both operands
 *  contiguous along the contraction dimension K (A row-major [M,K] with lda, B row-major
 *  [N,K] with ldb). fa / fb: the codes' formats (any combination).
 *  gran = FP8_GRAN_TENSOR: scale_inv_a and scale_inv_b point to one fp32 each (device).
 *  gran = FP8_GRAN_BLOCK_128x128: [GUARD] "Real products...": fine-grained scaling; A has
 *    1x128 tile scales scale_inv_a [M, K/128], B has 128x128 block scales
 *    scale_inv_b [K/128, N/128] (indexed [k/128][n/128]); each 128-deep K block is
 *    accumulated separately and added as C_ij += d_a[i,kb] * d_b[kb, j/128] * P_ij,kb.
 *    Requires K % 128 == 0 and N % 128 == 0.
 *  gran = FP8_GRAN_MX_1x32: MX scales on the tensor cores' block scaling: scale_inv_a and
 *    scale_inv_b point to the MX scale bytes of A (MN = M) and of B (MN = N), and
 *    C_ij = bf16( sum_g 2^(e_a[i,g] + e_b[j,g]) * sum_{k in group g} a_ik b_jk ). K % 128 == 0.
 *  Any M, N >= 0 and K >= 0 (K == 0 writes zeros). A, B, C 16-byte aligned; lda and ldb
 *  multiples of 16, ldc a multiple of 8. */
fp8_status_t fp8_scaled_mm(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb,
                           int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           fp8_gran_t gran, const float* scale_inv_a, const float* scale_inv_b,
                           void* C_bf16, int64_t ldc, void* stream);

/* fp8_scaled_mm with a caller-owned workspace that lets the library split the contraction:
 * when the output has too few 256 x 256 tiles to occupy every SM (for example a weight
 * gradient, [K_model, N] with a long token contraction), each tile is computed as two units
 * over the two halves of its K range; each unit writes its fp32 partial product to the
 * workspace and the tile's second unit to finish adds the other's to its own, scales and
 * stores.
 *  The pages have no such entry point: it restates "Explanation"'s scaled FP8 matmul
 *  ([SPEED]) with the same result definition as fp8_scaled_mm. The two partial sums change
 *  the fp32 summation order, so C can differ from fp8_scaled_mm's by fp32 rounding (always
 *  within the same error bound); fp32 addition being commutative, it is the same for every
 *  call with the same inputs.
 *  gran must be FP8_GRAN_TENSOR (block scaling never splits). workspace: device, 16-byte
 *  aligned, workspace_bytes long, owned by the caller and zero-filled before its first use;
 *  its head holds arrival counters that every successful call leaves at zero, so later
 *  calls of any shape need no clearing (after an error, zero-fill it again). A workspace
 *  smaller than fp8_scaled_mm_workspace_bytes(M, N, K), or null, runs the unsplit GEMM.
 *  Two calls must not use one workspace concurrently (different streams without ordering).
 *  Other rules as fp8_scaled_mm. */
fp8_status_t fp8_scaled_mm_ws(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb,
                              int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              fp8_gran_t gran, const float* scale_inv_a, const float* scale_inv_b,
                              void* C_bf16, int64_t ldc, void* workspace, int64_t workspace_bytes,
                              void* stream);

/* Workspace bytes fp8_scaled_mm_ws uses for this per-tensor problem on the current device:
 * 0 when it would not split (a null workspace then costs nothing). Negative on a CUDA error. */
int64_t fp8_scaled_mm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* One per-tensor-scaled GEMM of a grouped call: the arguments of fp8_scaled_mm with
 * gran = FP8_GRAN_TENSOR (C_bf16 [M,N] = bf16(d_a d_b sum_k a_ik b_jk)) when mn_major is 0
 * (A [M,K], B [N,K], contiguous along K); with mn_major 1 the arguments of fp8_scaled_mm_t
 * (A [K,M] with lda >= M, B [K,N] with ldb >= N, C = A^T B). */
typedef struct {
  const void* A;
  fp8_format_t fa;
  const void* B;
  fp8_format_t fb;
  int64_t M, N, K, lda, ldb;
  const float* scale_inv_a;
  const float* scale_inv_b;
  void* C_bf16;
  int64_t ldc;
  int32_t mn_major;
} fp8_mm_problem_t;

/* n (1 or 2) independent GEMMs in one persistent launch: their tiles share the GPU (longest
 * work units first, each on the least-loaded SM pair), so two problems that each leave SMs idle
 * (the backward pass's dgrad and wgrad) finish together instead of one after the other. The
 * pages have no such entry point: each problem is "Explanation"'s scaled FP8 matmul ([SPEED]),
 * computed as fp8_scaled_mm computes it. workspace (optional) follows fp8_scaled_mm_ws's rules
 * and lets a problem split K; size from fp8_scaled_mm_grouped_workspace_bytes. Each problem
 * obeys fp8_scaled_mm's rules with M, N, K > 0; the outputs must not overlap the inputs or
 * each other. */
fp8_status_t fp8_scaled_mm_grouped(const fp8_mm_problem_t* problems, int32_t n, void* workspace,
                                   int64_t workspace_bytes, void* stream);

/* Workspace bytes fp8_scaled_mm_grouped uses for these problems (0: nothing splits); negative
 * on a CUDA error or bad arguments. */
int64_t fp8_scaled_mm_grouped_workspace_bytes(const fp8_mm_problem_t* problems, int32_t n);

/* fp8_scaled_mm (per-tensor scales) whose epilogue also emits the FP8 codes of its output for
 * a following FP8 consumer (for example dgrad's dx, cast to E5M2 for the previous layer's
 * backward), so the bf16 result is not read back by a separate cast.
 *  [GUARD] "Real products...": delayed scaling with amax history. The codes use the output's
 *  delayed scale: Cq = cast_fc( fl32( bf16(C) * s_c ) ), s_c from c_st's history (required,
 *  delayed mode); the call raises c_st->amax_cur to max |bf16(C)|, records scale and
 *  scale_inv and adds to the counters, exactly as fp8_quantize of the bf16 output with
 *  FP8_SCALE_DELAYED would.
 *  While the history is empty (the bootstrap call) the scale needs the output's own amax, so
 *  the epilogue writes only C_bf16 and a second kernel, launched every call and returning at
 *  once when the history is non-empty, casts it from its current amax.
 *  C_bf16 [M,N] (leading dimension ldc) is required; Cq [M,N] contiguous codes, N % 16 == 0;
 *  K > 0. Other rules as fp8_scaled_mm. */
fp8_status_t fp8_scaled_mm_quant(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M,
                                 int64_t N, int64_t K, int64_t lda, int64_t ldb, const float* scale_inv_a,
                                 const float* scale_inv_b, void* C_bf16, int64_t ldc, fp8_format_t fc,
                                 const fp8_tensor_state_t* c_st, void* Cq, void* stream);

/* Refresh the FP8 weight cache from the bf16 master weight W [K,N] (contiguous).
 *  [SPEED] "Hardware precision": after each optimizer step the bf16 master weights are
 *  re-quantised to E4M3 and cached for the next forward. One pass over W writes
 *  wq_kn [K,N] (for dgrad) and/or wqT_nk [N,K] (for the forward); either may be NULL but
 *  not both. gran TENSOR (st required; CURRENT or DELAYED: delayed scaling uses the
 *  history before this call's amax is pushed), BLOCK_128x128 (block_scale_inv
 *  [K/128, N/128]) or MX_1x32 (groups of 32 down each column of W, i.e. along K; wq_kn must
 *  be NULL, wqT_nk [N,K] receives the codes and block_scale_inv the MX scale bytes with
 *  MN = N). Same rules as fp8_quantize. */
fp8_status_t fp8_requantize_weights(const void* w_master_bf16, int64_t K, int64_t N,
                                    fp8_gran_t gran, fp8_scaling_t mode,
                                    const fp8_tensor_state_t* st, void* wq_kn, void* wqT_nk,
                                    float* block_scale_inv, void* stream);

/* The optimizer step's update fused with the weight cache refresh.
 *  [SPEED] "Hardware precision": the bf16 master weights are updated by the optimizer and
 *  re-quantised to E4M3 after every step. In one launch:
 *    W <- bf16_rne( fl32(W) + delta )       (in place; one fp32 add per element)
 *  then the per-tensor E4M3 quantise of the updated W exactly as fp8_requantize_weights
 *  with gran TENSOR (mode CURRENT: the updated tensor's own amax; DELAYED: the history
 *  before this call's amax is pushed), writing wq_kn [K,N] and/or wqT_nk [N,K].
 *  w_master_bf16 [K,N] contiguous, read and written; delta [K,N] fp32 contiguous (the
 *  optimizer's step, e.g. -lr * m / (sqrt(v) + eps)), finite. K, N multiples of 8 (K of
 *  16 with wqT_nk); 16-byte aligned pointers. W and delta are read once: in the amax pass
 *  when the scale needs the updated tensor's amax, else in the cast pass. */
fp8_status_t fp8_update_requantize_weights(void* w_master_bf16, const float* delta, int64_t K, int64_t N,
                                           fp8_scaling_t mode, const fp8_tensor_state_t* st, void* wq_kn,
                                           void* wqT_nk, void* stream);

/* Forward of the FP8 up-projection: y [M,N] = x [M,K] W [K,N].
 *  Quantises x to E4M3 (per tensor into xq_save [M,K] with x_st, or per 1x128 tile into
 *  xq_save with x_tile_scale_inv [M, K/128]) and runs the scaled GEMM against the cached
 *  wqT_nk [N,K]. gran TENSOR uses w_st->scale_inv; gran BLOCK_128x128 (1x128 x tiles,
 *  128x128 W blocks) uses w_block_scale_inv [K/128, N/128] and requires mode CURRENT.
 *  gran MX_1x32 (mode CURRENT): x cast with MX scales (x_tile_scale_inv receives its scale
 *  bytes, MN = M), the GEMM with W's MX scale bytes in w_block_scale_inv (MN = N).
 *  xqT_save [K,M] (nullable, gran TENSOR only) keeps the transposed codes for wgrad.
 *  x contiguous; K % 16 == 0 (K % 128 == 0 for gran BLOCK); M % 16 == 0 with xqT_save.
 *  x_st is required for gran TENSOR and optional otherwise. An empty token batch (M == 0)
 *  is valid: x, xq_save and y may then be NULL, nothing is written but x_st's unit scales. */
fp8_status_t fp8_linear_fwd(const void* x_bf16, int64_t M, int64_t K, int64_t N,
                            const void* wqT_nk, const fp8_tensor_state_t* w_st,
                            const float* w_block_scale_inv, const fp8_tensor_state_t* x_st,
                            fp8_gran_t gran, fp8_scaling_t mode, void* xq_save, void* xqT_save,
                            float* x_tile_scale_inv, void* y_bf16, void* stream);

/* Backward of the FP8 up-projection (per-tensor scales).
 *  [GUARD] "What an interviewer would ask next": the backward signal dy [M,N] is cast to
 *  E5M2 for its range (per tensor, with dy_st, mode CURRENT or DELAYED) into the caller's
 *  scratch dyq_ws [M,N] and dyqT_ws [N,M], then
 *    dgrad  dx [M,K] = d_dy d_w  dyq  wq_kn^T      (contraction over N; wq_kn [K,N])
 *    wgrad  dW [K,N] = d_x  d_dy xqT_save dyqT_ws^T (contraction over M; xqT_save [K,M])
 *  dx and dw may each be NULL (that GEMM is skipped; dyqT_ws may then be NULL when dw is).
 *  Needs M, N, K multiples of 16. dy contiguous. An empty token batch (M == 0) is valid:
 *  dy, the scratch, xqT_save and dx may then be NULL, and dW is written as zeros. */
fp8_status_t fp8_linear_bwd(const void* dy_bf16, int64_t M, int64_t K, int64_t N,
                            const void* xqT_save, const fp8_tensor_state_t* x_st,
                            const void* wq_kn, const fp8_tensor_state_t* w_st,
                            fp8_tensor_state_t* dy_st, fp8_scaling_t mode,
                            void* dyq_ws, void* dyqT_ws, void* dx_bf16, void* dw_bf16,
                            void* stream);

/* fp8_linear_bwd with a caller-owned workspace: when both dx and dW are requested, the two
 * GEMMs run in one persistent launch either way (their tiles share the grid, longest first on
 * the least-loaded SMs); the workspace also lets the weight gradient split its long token
 * contraction (see fp8_scaled_mm_ws). The pages have no such entry point: it is
 * fp8_linear_bwd's computation ("FP8 stability guardrails": E5M2 gradients) with
 * fp8_scaled_mm_ws's workspace rules (16-byte aligned, zero-filled before first use, left
 * reusable, one call at a time per workspace; smaller or null runs without split K). */
fp8_status_t fp8_linear_bwd_ws(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xqT_save,
                               const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                               fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dyqT_ws,
                               void* dx_bf16, void* dw_bf16, void* workspace, int64_t workspace_bytes, void* stream);

/* fp8_linear_bwd_ws whose weight gradient reads x's saved codes xq_save [M,K] (as the forward
 * writes them, with no transposed copy) and dy's codes dyq_ws [M,N] as they are: the tensor
 * cores read both MN-major (the contraction runs over the tokens, the rows of both), so the dy
 * cast writes one copy of the codes (3 bytes per element moved instead of 4) and the forward
 * needs no xqT_save. [GUARD] "What an interviewer would ask next": E5M2 gradients; the result
 * definition is fp8_linear_bwd's (the same per-tensor scales, products and fp32 accumulation;
 * only the operands' layout in shared memory differs):
 *   dgrad  dx [M,K] = d_dy d_w  dyq wq_kn^T
 *   wgrad  dW [K,N] = d_x  d_dy xq_save^T dyq
 * dyq_ws [M,N] caller scratch (16-byte aligned); workspace as fp8_linear_bwd_ws (size from
 * fp8_linear_bwd_workspace_bytes). M, K, N multiples of 16; dx or dw may be NULL. */
fp8_status_t fp8_linear_bwd_mn(const void* dy_bf16, int64_t M, int64_t K, int64_t N, const void* xq_save,
                               const fp8_tensor_state_t* x_st, const void* wq_kn, const fp8_tensor_state_t* w_st,
                               fp8_tensor_state_t* dy_st, fp8_scaling_t mode, void* dyq_ws, void* dx_bf16,
                               void* dw_bf16, void* workspace, int64_t workspace_bytes, void* stream);

/* C [M,N] (bf16, ldc) = A^T B for operands stored contraction-major: A [K,M] row-major (lda >= M)
 * and B [K,N] row-major (ldb >= N); C_ij = bf16( d_a d_b sum_k a_ki b_kj ), fp32 accumulation,
 * per-tensor scales. The tensor cores read both operands MN-major, so a weight gradient
 * x_q^T dy_q takes the codes as the casts wrote them. [SPEED] "Explanation": the scaled FP8
 * matmul; the page lays operands out contiguous along the contraction for the library it
 * calls, which this layout does without. A, B 16-byte aligned, lda and ldb multiples of 16, ldc
 * of 8; workspace as fp8_scaled_mm_ws (split K for few-tile outputs; size from
 * fp8_scaled_mm_workspace_bytes(M, N, K)). */
fp8_status_t fp8_scaled_mm_t(const void* A, fp8_format_t fa, const void* B, fp8_format_t fb, int64_t M, int64_t N,
                             int64_t K, int64_t lda, int64_t ldb, const float* scale_inv_a, const float* scale_inv_b,
                             void* C_bf16, int64_t ldc, void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes fp8_linear_bwd_ws uses for these sizes with dx and dW both requested on the
 * current device (0: it would not split). Negative on a CUDA error. */
int64_t fp8_linear_bwd_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* fp8_linear_bwd without caller scratch. The pages have no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory at the point of the call -- for
 * example a host framework that hands the library only its input and output tensors and
 * forbids side allocations, or a plain C program that links this library and keeps no
 * device allocator of its own. Everything is as in fp8_linear_bwd (same arguments, same
 * results, same validation) except that the E5M2 codes of dy and of dy^T live in a static
 * 64 MiB device array inside the library instead of dyq_ws / dyqT_ws:
 *   - size limit: M*N bytes when dw_bf16 is NULL, else M*N rounded up to 256 plus M*N
 *     bytes, at most 64 MiB (e.g. M*N <= 32 Mi elements with wgrad); larger shapes return
 *     FP8_ERR_UNSUPPORTED before anything is enqueued;
 *   - the array is part of the library's device code, so a device holds its 64 MiB from
 *     the moment that code is loaded there until the process exits. With CUDA's lazy
 *     module loading (the default) that is the first library call on the device that needs
 *     it -- for example any call that launches a GEMM, fp8_poll_device_error, or this one --
 *     and not only a call of this entry point; with eager loading it is context creation. That load fails with a
 *     CUDA out-of-memory error (FP8_ERR_CUDA) on a device with less than 64 MiB free;
 *   - the first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current and caches it; make that first call before any stream capture;
 *   - all calls share one array, so calls whose work overlaps on the GPU (different streams,
 *     or threads without ordering) race on it and give wrong codes; order them on one stream;
 *   - the call allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine;
 *     the array's previous contents never matter because the dy cast overwrites what it uses. */
fp8_status_t fp8_linear_bwd_noalloc(const void* dy_bf16, int64_t M, int64_t K, int64_t N,
                                    const void* xqT_save, const fp8_tensor_state_t* x_st,
                                    const void* wq_kn, const fp8_tensor_state_t* w_st,
                                    fp8_tensor_state_t* dy_st, fp8_scaling_t mode,
                                    void* dx_bf16, void* dw_bf16, void* stream);

/* Push st->amax_cur into the history: amax_history[hist_count % hist_len] = amax_cur;
 * hist_count += 1; amax_cur = 0 (the next step's delayed casts start a new running maximum).
 * [GUARD] "Real products...": amax history tracking. */
fp8_status_t fp8_history_commit(const fp8_tensor_state_t* st, void* stream);

/* The same push for n distinct states (0 <= n <= 32) in one launch: states points to a
 * host array of n structs (copied by the call), e.g. the x, W and dy states of a layer at
 * the end of a training step. A state listed twice is rejected. */
fp8_status_t fp8_history_commit_many(const fp8_tensor_state_t* states, int32_t n, void* stream);

/* Device-side error word. Every wait inside a kernel is bounded; a wait that runs out
 * sets a bit in this word and its kernel returns early (its outputs are then undefined).
 * fp8_poll_device_error synchronises the current device, returns FP8_ERR_TIMEOUT if any
 * wait ran out since the last clear (and clears the word), else FP8_OK. */
fp8_status_t fp8_poll_device_error(void);

/* Limit in nanoseconds for every bounded wait in later launches (default 4e9 ns). */
fp8_status_t fp8_set_wait_limit_ns(unsigned long long ns);

/* Self-test of the bounded wait: launches one kernel whose thread waits on a barrier
 * that nothing completes, for at most limit_ns; then synchronises the stream and returns
 * FP8_ERR_TIMEOUT (the expected result) with the device word cleared again. */
fp8_status_t fp8_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* Copy the message of the last failed call on this thread into buf (at most n bytes,
 * NUL-terminated). Returns FP8_OK. */
fp8_status_t fp8_get_last_error_detail(char* buf, size_t n);

/* Static name of a status code. */
const char* fp8_status_string(fp8_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* FP8GB_H */
