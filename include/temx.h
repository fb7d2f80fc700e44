/*
 * temx — MXFP8 block-scaled quantisation and MXFP8 GEMM for GB300 (sm_103a).
 *
 * C ABI of libtemx.so.  Plain pointers and sizes only; every device buffer and
 * the stream belong to the caller.  Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL = the legacy default stream).  No call
 * allocates device memory.
 *
 * Definitions the calls implement
 * -------------------------------
 * MXFP8 ("MXFP8 1D scaling", named in "HipKittens MXFP8 GEMM Support",
 * ROCm/TransformerEngine PR #566, review thread; "E8M0 (power-of-2)" scales,
 * ROCm/TransformerEngine README, "Blockwise FP8 GEMM support on ROCm"):
 * every 32 consecutive elements along the quantised axis share one E8M0
 * scale byte s = e + 127 with e = floor(log2 amax) - 8, clamped to
 * [-127, 127] (OCP Microscaling Formats v1.0, FP32 -> MX conversion; amax = 0
 * gives s = 0x00).  Each element becomes the E4M3 byte of x * 2^-e, rounded
 * to nearest-even and saturated to +-448; a negative value that rounds to
 * zero keeps its sign (0x80).  A block holding a NaN or an infinity gives
 * s = 0xFF and every element 0x7F.
 *
 * Layouts
 * -------
 * Matrices are row-major.  A scale matrix for data [R x C] quantised along C
 * is uint8 [R x ld_s] whose first C/32 bytes per row hold the scales; ld_s
 * must be a multiple of 16 and >= C/32 (te_mx_scale_pitch gives the
 * smallest).  Bytes past C/32 in a row are never written or read.
 *
 * Errors
 * ------
 * Every call validates its arguments on the host and returns a status before
 * launching anything; te_mx_last_error() then holds a message (per thread).
 * Kernels bound every wait; a wait that runs out sets a device status word
 * that te_mx_device_status() reports (TE_MX_ERR_DEVICE_TIMEOUT).
 *
 * Per-device state
 * ----------------
 * On its first call on a device the library looks up, and then keeps for the
 * life of the process, device addresses of its own static device memory (the
 * status word; the scratch array of te_mx_quantize_dbias_noalloc).  They are
 * valid for that device's primary context only: after the context is
 * destroyed (cudaDeviceReset) no entry point may be called on that device
 * again in the same process.
 */
#ifndef TEMX_H
#define TEMX_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TEMX_API __attribute__((visibility("default")))
#else
#define TEMX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum te_mx_status {
    TE_MX_OK = 0,
    TE_MX_ERR_INVALID_ARG = 1,       /* NULL where a buffer is required, negative size, bad enum */
    TE_MX_ERR_UNSUPPORTED_SHAPE = 2, /* a size rule below is broken */
    TE_MX_ERR_MISALIGNED = 3,        /* a pointer or pitch breaks its alignment rule */
    TE_MX_ERR_WORKSPACE_TOO_SMALL = 4,
    TE_MX_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed (message has the name) */
    TE_MX_ERR_DEVICE_TIMEOUT = 6,    /* a kernel gave up a bounded wait */
    TE_MX_ERR_ARCH = 7               /* the current device is not sm_103 */
} te_mx_status;

/* GEMM epilogues ("BIAS and GELU AUX", HipKittens MXFP8 GEMM Support, PR
 * description).  With bias: pre = acc + bias[n].  Without GELU: D = bf16(pre).
 * With GELU: AUX = bf16(pre), D = bf16(0.5 pre (1 + tanh(sqrt(2/pi)(pre +
 * 0.044715 pre^3)))) computed from the fp32 pre-activation. */
typedef enum te_mx_epilogue {
    TE_MX_EPI_NONE = 0,
    TE_MX_EPI_BIAS = 1,
    TE_MX_EPI_GELU_AUX = 2,
    TE_MX_EPI_BIAS_GELU_AUX = 3,
    /* Backward of GELU (the DGELU epilogue of "Blockwise FP8 GEMM support on
     * ROCm", ROCm/TransformerEngine README): `aux` is an INPUT holding the bf16
     * pre-activation saved by the forward GELU_AUX GEMM, and
     * D = bf16(acc * gelu'(aux)), gelu' the derivative of the tanh form.
     * bias must be NULL. */
    TE_MX_EPI_DGELU = 4,
    /* Accumulation into an fp32 output (the beta epilogue and fp32 output of
     * "Blockwise FP8 GEMM support on ROCm", ROCm/TransformerEngine README,
     * with beta = 1: gradient accumulation into an fp32 main gradient):
     * D is fp32 [M x N], read and written, D = fl32(D + acc).  bias and aux
     * must be NULL.  te_mx_gemm only (and the accumulate flag of
     * te_mx_grouped_gemm_wgrad). */
    TE_MX_EPI_ACCUMULATE_F32 = 5
} te_mx_epilogue;

/* Smallest legal scale pitch for k quantised elements per row:
 * round_up(k/32, 16) bytes. */
TEMX_API size_t te_mx_scale_pitch(int64_t k);

/* te_mx_quantize — MXFP8-quantise a bf16 matrix row-wise and/or column-wise in
 * one pass over HBM (MXFP8 1D scaling; the column-wise copy is the transposed
 * operand the wgrad GEMM consumes, cf. the cast_transpose kernels of
 * ROCm/TransformerEngine README, "Experimental Triton Kernels on ROCm").
 *
 *   x       bf16 [rows x cols], row pitch ld_x elements (device).
 *   q_row   uint8 [rows x cols] (pitch cols), E4M3 codes, blocks along a row;
 *   s_row   uint8 [rows x ld_s_row] E8M0 bytes, s_row[r][j] scales
 *           q_row[r][32j .. 32j+31].  Both NULL: row-wise output skipped.
 *   q_col   uint8 [cols x rows] (pitch rows): q_col[c][r] is X[r][c], blocks of
 *           32 consecutive rows of one column, i.e. the transpose quantised
 *           along its rows;
 *   s_col   uint8 [cols x ld_s_col], s_col[c][i] scales q_col[c][32i .. 32i+31].
 *           Both NULL: column-wise output skipped.
 * Rules: cols % 32 == 0; rows % 32 == 0 when q_col is given; rows, cols >= 0
 * (0 is a no-op); x 16-byte aligned and ld_x % 8 == 0, ld_x >= cols; q_row,
 * q_col 16-byte aligned; ld_s_* multiples of 16 and >= the block count.
 * Output is bit-exact to the definition above. */
TEMX_API te_mx_status te_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                            uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                            uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                            void* stream);

/* te_mx_quantize_dbias — te_mx_quantize plus the bias gradient of the same
 * matrix (the fused cast/transpose/bias-grad of the gradient, cf. the
 * cast_transpose_bgrad kernels of ROCm/TransformerEngine README, "Experimental
 * Triton Kernels on ROCm"):
 *   dbias[c] = bf16(sum_r x[r][c])                         (dbias: bf16 [cols])
 * Sums are taken in fp32 in a fixed order (each 64-row band of a column, then
 * the bands), so the result is deterministic; accuracy |dbias - exact| <=
 * 2^-7 |exact| + 1e-5 sum_r |x[r][c]|.
 *   workspace: device scratch of te_mx_quantize_dbias_workspace_size(rows, cols)
 *              bytes owned by the caller (fp32 band partial sums); its contents
 *              on entry do not matter and it is clobbered.
 * Quantisation outputs and rules as te_mx_quantize (either orientation may be
 * NULL, or both: then only dbias is produced); dbias must be 16-byte aligned.
 * Returns TE_MX_ERR_WORKSPACE_TOO_SMALL if workspace_bytes is short. */
TEMX_API size_t te_mx_quantize_dbias_workspace_size(int64_t rows, int64_t cols);
TEMX_API te_mx_status te_mx_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                  uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                  uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                  void* dbias, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* te_mx_quantize_dbias_noalloc — te_mx_quantize_dbias for callers that cannot
 * allocate device memory.  The sources describe no such entry point; it exists
 * for host code that has no device allocator of its own or runs under a fixed,
 * pre-planned memory budget in which allocating after start-up is not allowed
 * (and where a cudaMalloc, which may synchronise the device, is unwelcome).
 * Instead of a caller workspace, the band sums go to a scratch array built
 * into the library: 32 MiB per GPU (TE_MX_NOALLOC_SCRATCH_BYTES), held by every
 * GPU that loads the library until the process exits.  Sizes whose scratch
 * (te_mx_quantize_dbias_workspace_size) exceeds it are rejected with
 * TE_MX_ERR_WORKSPACE_TOO_SMALL and a message.  The first call on a device
 * looks up the scratch address for that device (so make that first call
 * before recording work into a stream capture).  All calls share the one
 * array: calls whose kernels overlap on the GPU (different streams without
 * ordering) race on it and give wrong results.  Nothing in it needs clearing
 * between calls (every value is written before it is read).  Arguments,
 * outputs and results are those of te_mx_quantize_dbias.  Allocates nothing. */
#define TE_MX_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
TEMX_API te_mx_status te_mx_quantize_dbias_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                          uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                          uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                          void* dbias, void* stream);

/* te_mx_block_quantize — Float8BlockScaling quantisation with E8M0-cast scales
 * ("Blockwise FP8 GEMM support on ROCm", ROCm/TransformerEngine README: 1Dx1D
 * and 1Dx2D block scaling; the recipe's FP32 scale amax/448 cast to a power of
 * two, the default there).  Blocks: block_2d == 0 gives 1x128 blocks along a
 * row for q_row and 128x1 blocks down a column for q_col (activations and
 * gradients); block_2d == 1 gives 128x128 blocks shared by both copies
 * (weights).  Per block, with amax the largest |x| of the elements present
 * (edge blocks may be partial):
 *   e = ceil(log2(amax / 448)) clamped to [-127, 127] (-127 for amax 0),
 *   q = E4M3_rn_satfinite(x 2^-e)   (no element saturates),
 * and a block holding NaN/inf gets scale byte 0xFF and codes 0x7F.
 * Outputs use the te_mx_quantize layout exactly: s_row[r][j] = e + 127 of the
 * block holding q_row[r][32j], i.e. each block scale is repeated over its
 * 32-element groups, so te_mx_gemm / te_mx_grouped_gemm on these operands
 * compute the block-scaled GEMM (1Dx1D: both operands block_2d == 0; 1Dx2D:
 * the weight with block_2d == 1).
 * Arguments, rules and errors as te_mx_quantize, plus: block_2d is 0 or 1
 * (else TE_MX_ERR_INVALID_ARG).  Output is bit-exact to the definition above. */
TEMX_API te_mx_status te_mx_block_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                           int32_t block_2d,
                                           uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                           uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                           void* stream);

/* te_mx_block_quantize_fp32 — Float8BlockScaling quantisation that keeps the
 * FP32 scales (the README's second mode: "compute the GEMM with the FP32
 * scales directly"; te_mx_gemm_fp32_scales consumes the result).  Blocks as
 * te_mx_block_quantize.  Per block, with amax the largest |x| present:
 *   s = fl32(amax / 448)                 the stored fp32 scale,
 *   r = min(fl32(1 / s), FLT_MAX),       q = E4M3_rn_satfinite(fl32(x r)),
 * every operation IEEE fp32 rounded to nearest even; amax 0 gives s = r = 1;
 * a block holding NaN/inf gets s = NaN and codes 0x7F.
 *   q_row, q_col      E4M3 codes as te_mx_quantize (device, 16-byte aligned).
 *   s_row             fp32 [rows x ld_s_row]: s_row[r][j] is the scale of the
 *                     block holding q_row[r][128 j] (2D: repeated over the
 *                     block's 128 rows); ld_s_row >= ceil(cols / 128) and a
 *                     multiple of 4 (te_mx_block_scale_pitch_fp32(cols)).
 *   s_col             fp32 [cols x ld_s_col]: the scale of the block holding
 *                     q_col[c][128 j]; ld_s_col >= ceil(rows / 128), % 4 == 0.
 * Scale arrays 16-byte aligned.  Other rules and errors as te_mx_quantize;
 * block_2d 0 or 1.  Output is bit-exact to the definition above. */
TEMX_API int64_t te_mx_block_scale_pitch_fp32(int64_t n);
TEMX_API te_mx_status te_mx_block_quantize_fp32(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                                int32_t block_2d,
                                                uint8_t* q_row, float* s_row, int64_t ld_s_row,
                                                uint8_t* q_col, float* s_col, int64_t ld_s_col,
                                                void* stream);

/* te_mx_layernorm_quantize — LayerNorm fused with MXFP8 quantisation (the
 * input of LayerNormLinear / LayerNormMLP; te.LayerNorm as the drop-in of
 * torch.nn.LayerNorm, leeroopedia "FP8 Training Quickstart"; parameters
 * 'scale' and 'bias', epsilon 1e-5 on the TE "Getting Started" JAX page).
 * Per row r of x (hidden elements):
 *   mu[r] = mean(x[r]),  var = mean((x[r] - mu)^2) (biased),
 *   rsigma[r] = 1/sqrt(var + eps),  y = (x - mu) rsigma gamma + beta,
 * and y, unrounded, is MXFP8-quantised exactly as te_mx_quantize quantises
 * its input (q_row/s_row: blocks of 32 along the row; q_col/s_col: blocks of
 * 32 rows of a column, stored transposed).  The normalised tensor is never
 * written.  Arithmetic is fp32: mu = fl(S/H) with S a sum of the row in fp32
 * whose longest chain of additions is at most 64; var likewise from the
 * squares of fl(x - mu), each rounded on its own or fused into the addition
 * that accumulates it; rsigma = fl(1/fl(sqrt(fl(var + eps)))); y =
 * fma(fl(fl(x - mu) rsigma), gamma, beta) with one rounding.  Codes and scales
 * are the exact MXFP8 quantisation of that fp32 y; the sums are taken in a
 * fixed order (deterministic).  Two kernels run on `stream`: the statistics,
 * then normalisation + quantisation (reading mu / rsigma back), the second as
 * a programmatic dependent launch of the first (it waits for the first
 * grid's results; work queued after the call waits for both, as usual).
 *
 *   x       bf16 [rows x hidden], pitch ld_x (device, 16-byte aligned, ld_x % 8 == 0);
 *   gamma, beta  bf16 [hidden] (device, 4-byte aligned);  eps > 0 and finite;
 *   q_row/s_row, q_col/s_col: as te_mx_quantize (either pair may be NULL:
 *           then only the statistics are computed);
 *   mu, rsigma   fp32 [rows] (device, required): the statistics, for the backward pass.
 * Rules: hidden % 32 == 0 and hidden <= 32768; rows % 32 == 0 when q_col is
 * given; rows == 0 or hidden == 0 is a no-op. */
TEMX_API te_mx_status te_mx_layernorm_quantize(const void* x, int64_t rows, int64_t hidden, int64_t ld_x,
                                               const void* gamma, const void* beta, float eps,
                                               uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                               uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                               float* mu, float* rsigma, void* stream);

/* te_mx_gemm — MXFP8 TN GEMM with fused epilogue (HipKittens MXFP8 GEMM
 * Support, PR description: MXFP8 GEMM with BIAS and GELU AUX epilogues; the
 * review thread's TN layout and its K % 128 rule for MXFP8 scaling):
 *   acc[m][n] = sum_k (A[m][k] 2^(sA[m][k/32]-127)) (B[n][k] 2^(sB[n][k/32]-127)),
 * accumulated in fp32 on the tensor cores, then the epilogue above.
 *
 *   A  uint8 E4M3 [M x K] (pitch K), sA uint8 [M x ld_sA];
 *   B  uint8 E4M3 [N x K] (pitch K), sB uint8 [N x ld_sB]  (both K-contiguous);
 *   bias  bf16 [N] or NULL (required for the *_BIAS* epilogues);
 *   D     bf16 [M x N] (pitch N);  aux bf16 [M x N]: written by the GELU_AUX
 *         epilogues, read by DGELU, else ignored.
 *   workspace / workspace_bytes: reserved; te_mx_gemm_workspace_size() is 0
 *         and NULL/0 may be passed.
 * Rules: K % 128 == 0, K >= 128; M, N >= 1 with N % 16 == 0 (M arbitrary);
 * A, B, sA, sB, D, aux 16-byte aligned; ld_s* multiples of 16 >= K/32.
 * Accuracy: |D - exact| <= 2^-7 |exact| + 1e-5 sum_k |a_k b_k| element-wise,
 * exact = the epilogue of the fp64 product of the dequantised operands. */
TEMX_API te_mx_status te_mx_gemm(const uint8_t* A, const uint8_t* sA, int64_t ld_sA,
                        const uint8_t* B, const uint8_t* sB, int64_t ld_sB,
                        int64_t M, int64_t N, int64_t K,
                        const void* bias, int32_t epilogue,
                        void* D, void* aux,
                        void* workspace, size_t workspace_bytes,
                        void* stream);

/* te_mx_gemm_fp32_scales — the Float8BlockScaling TN GEMM computed with the
 * FP32 scales directly (ROCm/TransformerEngine README, "Blockwise FP8 GEMM
 * support on ROCm", second mode), on te_mx_block_quantize_fp32 output:
 *   pre[m][n] = sum_kb sA[m][kb] sB[n][kb] sum_{k in block kb} A[m][k] B[n][k]
 *   (+ bias[n]),  D = the epilogue of pre as in te_mx_gemm,
 * with 128-long K blocks kb.  A: E4M3 [M x K], B: E4M3 [N x K] (K-contiguous);
 * sA fp32 [M x ld_sA], sB fp32 [N x ld_sB] (one scale per row and K block;
 * pitches multiples of 4, >= K/128; 16-byte aligned).  b_blocks_2d = 1 tells
 * the GEMM that sB is constant over 128-row blocks (128x128 weight blocks,
 * 1Dx2D scaling), so it reads one scale per block; 0 for 1x128 B blocks
 * (1Dx1D).  Epilogues: NONE, BIAS, GELU_AUX, BIAS_GELU_AUX, DGELU (not
 * ACCUMULATE_F32).  Each K block's fp32 product (tensor cores, no block
 * scaling) is scaled and accumulated in fp32.  Shapes, alignment, errors and
 * the accuracy bound as te_mx_gemm; asynchronous on `stream`. */
TEMX_API te_mx_status te_mx_gemm_fp32_scales(const uint8_t* A, const float* sA, int64_t ld_sA,
                                             const uint8_t* B, const float* sB, int64_t ld_sB,
                                             int32_t b_blocks_2d, int64_t M, int64_t N, int64_t K,
                                             const void* bias, int32_t epilogue,
                                             void* D, void* aux, void* stream);

/* te_mx_grouped_gemm — one launch over G groups (MoE experts) of the same
 * GEMM ("Single-Launch Grouped GEMM Backends on ROCm", ROCm/TransformerEngine
 * README; MXFP8 grouped GEMM), with ragged and possibly empty groups:
 *   for g with m_g > 0: D[rows of g] = epilogue(X[rows of g] . W[g]^T + bias[g]).
 *
 *   group_m  int32 [G] on the DEVICE (as routing produces it), m_g >= 0;
 *            group g owns rows [sum_{h<g} m_h, sum_{h<=g} m_h) of X, D, aux.
 *   total_m  host upper bound on sum m_g: the row count of X, sX, D, aux.
 *   X  uint8 [total_m x K], sX uint8 [total_m x ld_sX];
 *   W  uint8 [G x N x K], sW uint8 [G*N x ld_sW] (group g's scales are rows
 *      g*N .. g*N+N-1);  bias bf16 [G x N] or NULL.
 * Rows past sum m_g are not written.  If sum m_g > total_m the call writes
 * nothing past total_m and te_mx_device_status() reports TE_MX_ERR_INVALID_ARG.
 * Rules as te_mx_gemm, plus 1 <= G <= 1024. */
TEMX_API te_mx_status te_mx_grouped_gemm(int32_t num_groups, const int32_t* group_m, int64_t total_m,
                                const uint8_t* X, const uint8_t* sX, int64_t ld_sX,
                                const uint8_t* W, const uint8_t* sW, int64_t ld_sW,
                                int64_t N, int64_t K,
                                const void* bias, int32_t epilogue,
                                void* D, void* aux,
                                void* workspace, size_t workspace_bytes,
                                void* stream);

/* Grouped wgrad for MoE experts (the single-launch grouped GEMM of
 * "Single-Launch Grouped GEMM Backends on ROCm", ROCm/TransformerEngine
 * README, applied to the weight gradient dW_e = dY_e^T X_e).
 *
 * Layout of a per-expert column-wise operand.  Expert e owns rows
 * [R_e, R_e + m_e) of a token-major matrix x [total x cols]; its copy is
 * blocked along tokens (32 per E8M0 scale) and zero-padded to
 * Kp_e = round_up(m_e, 128) tokens, so no block crosses an expert boundary:
 *   q[c][P_e + t], t < Kp_e     P_e = sum_{e'<e} Kp_e'
 *   s[c][Q_e + b], b < Kp_e/32  Q_e = sum_{e'<e} round_up(Kp_e'/32, 16)
 * (codes of padding tokens are 0, their block scales 0x00).  Expert sizes
 * live on the device, so the widths are bounded on the host:
 * te_mx_grouped_code_width / te_mx_grouped_scale_width give pitches (row
 * lengths in bytes) that always suffice for total_m tokens in num_groups
 * experts. */
TEMX_API int64_t te_mx_grouped_code_width(int64_t total_m, int32_t num_groups);
TEMX_API int64_t te_mx_grouped_scale_width(int64_t total_m, int32_t num_groups);

/* te_mx_quantize_colwise_grouped — the per-expert column-wise MXFP8 copy
 * above of x (bf16 [total_m x cols], pitch ld_x; rows grouped by expert in
 * order; group_m: device int32 [num_groups] token counts, sum <= total_m).
 *   q  uint8 [cols x ld_q]: codes;  s  uint8 [cols x ld_s]: scales.
 * Rules: 1 <= num_groups <= 1024; cols % 32 == 0; x, q 16-byte aligned;
 * ld_x % 8 == 0; ld_q, ld_s multiples of 16.  Bytes of q / s past the layout's
 * width, and scale bytes between Kp_e/32 and Q_{e+1}, are not written.
 * A negative count, counts summing above total_m or a layout wider than
 * ld_q / ld_s write nothing and make te_mx_device_status() report
 * TE_MX_ERR_INVALID_ARG.  Output is bit-exact to the definition above. */
TEMX_API te_mx_status te_mx_quantize_colwise_grouped(const void* x, int64_t total_m, int64_t cols, int64_t ld_x,
                                                     int32_t num_groups, const int32_t* group_m,
                                                     uint8_t* q, int64_t ld_q, uint8_t* s, int64_t ld_s,
                                                     void* stream);

/* te_mx_grouped_gemm_wgrad — dW_e = deq(dY_e)^T deq(X_e) for every expert in
 * one launch (fp32 accumulation on the tensor cores, bf16 output):
 *   dY, s_dY   per-expert column-wise copy of dY [total_m x M]: [M x ld_q], [M x ld_s];
 *   X,  s_X    per-expert column-wise copy of X  [total_m x N]: [N x ld_q], [N x ld_s];
 *   accumulate 0: D is bf16 [num_groups x M x N], D[e] = dW_e (zeros for an
 *              expert without tokens);  1: D is fp32 [num_groups x M x N] and
 *              D[e] = fl32(D[e] + dW_e) (unchanged for an expert without tokens).
 * group_m and total_m as for te_mx_quantize_colwise_grouped (the same device
 * array that laid the operands out).  Rules: 1 <= num_groups <= 1024;
 * N % 16 == 0; ld_q, ld_s multiples of 16 (ld_s >= 16); num_groups * M <
 * 2^31; dY, X, D 16-byte aligned.  Device-side errors as above (nothing is
 * written).  Accuracy as te_mx_gemm. */
TEMX_API te_mx_status te_mx_grouped_gemm_wgrad(int32_t num_groups, const int32_t* group_m, int64_t total_m,
                                               const uint8_t* dY, const uint8_t* s_dY,
                                               const uint8_t* X, const uint8_t* s_X,
                                               int64_t M, int64_t N, int64_t ld_q, int64_t ld_s,
                                               int32_t accumulate, void* D, void* stream);

/* Workspace bytes te_mx_gemm / te_mx_grouped_gemm need: 0 for every shape
 * (scale re-layout happens in shared memory; kept so a future layout change
 * does not break the ABI). */
TEMX_API size_t te_mx_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t num_groups);

/* Synchronises the current device, returns and clears the device status word
 * the kernels set (TE_MX_OK, TE_MX_ERR_DEVICE_TIMEOUT or
 * TE_MX_ERR_INVALID_ARG), or TE_MX_ERR_CUDA if the synchronise fails. */
TEMX_API te_mx_status te_mx_device_status(void);

/* te_mx_selftest_timeout — check of the failure-detection path (no part of the
 * computation): launches one CTA that waits on an mbarrier that nothing ever
 * arrives at, with the same bounded wait the kernels use but a limit of
 * `limit_us` microseconds (1 .. 2,000,000).  The wait gives up, records
 * TE_MX_ERR_DEVICE_TIMEOUT in the device status word and the kernel returns
 * normally, so the CUDA context stays usable; the next te_mx_device_status()
 * reports the timeout (and clears it).  Returns TE_MX_ERR_INVALID_ARG for a
 * limit outside the range. */
TEMX_API te_mx_status te_mx_selftest_timeout(uint32_t limit_us, void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
TEMX_API const char* te_mx_last_error(void);

/* Library version string. */
TEMX_API const char* te_mx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TEMX_H */
