/*
 * fq.h -- C ABI of the GB300 block-scaled FP4 fake-quantization library.
 *
 * The library quantizes FP32 or BF16 tensors to 4-bit E2M1 codes under
 * per-block scales, packs them, dequantizes them, produces the
 * straight-through-estimator mask of fake quantization, and keeps the
 * OsciReset oscillation statistics of quantization-aware training.
 *
 * Sources (web pages on FP4 quantization-aware training):
 *  [GPTOSS] "Aprimorando gpt-oss para Precisão e Desempenho com Treinamento
 *           Consciente à Quantização" -- TL;DR, "O que há de novo": MXFP4 and
 *           NVFP4, NVFP4 with FP8 E4M3 block scales.
 *  [QATREC] "Como o Treinamento com Quantização Detecta e Recupera Precisão em
 *           Inferência de Baixa Precisão" -- "Detalhes técnicos": fake
 *           quantization (quantize/dequantize in a high-precision type) with a
 *           straight-through estimator exposing rounding and clipping.
 *  [TJV2]   "Resumo Técnico: TetraJet-v2" -- §2A double-block NVFP4 (FP32 scale
 *           per 128-element outer block, 8-bit scale per 16-element inner
 *           block), stochastic rounding with E[round(x)] = x, 1x16 groups and
 *           the transposed weight; §2B OsciReset (dist_Q / dist_M); §2C
 *           OutControl (random Hadamard transform of backward operands,
 *           static retention of outlier channels in FP8).
 *  [QADP]   "Quantization-Aware Distillation for NVFP4 Inference Accuracy
 *           Recovery" -- §2 Metodologia: the NVFP4 student learns the BF16
 *           teacher's output distribution through a KL-divergence loss at
 *           softmax temperature T = 1.
 *
 * Numeric definitions (the pages leave these open; this library's readings):
 *  E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 *    magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Nearest-even rounding with
 *    saturation to +-6; the sign bit is kept for zero results.
 *  E4M3 scale: OCP "FN" byte (bias 7, max 448), nearest-even, saturating.
 *  E8M0 scale: value 2^(code - 127).
 *  NVFP4 (FQ_NVFP4): s_g = amax(tensor) / 2688 (FP32, 2688 = 6 * 448);
 *    per 1x16 block s_b = (block_amax / 6) / s_g -> E4M3 code c;
 *    s_eff = E4M3(c) * s_g; r = 1 / s_eff (0 when s_eff = 0).
 *  Double block (FQ_NVFP4_2LEVEL, [TJV2] §2A): as NVFP4 with s_g replaced by
 *    s_o = amax(1x128 block) / 2688, stored per outer block.
 *  MXFP4 (FQ_MXFP4): per 1x32 block k = floor(log2 block_amax) - 2 clamped to
 *    [-127, 127], E8M0 code k + 127, s_eff = 2^k, r = 2^-k.
 *  Element: y = x * r (FP32); code = E2M1(y) (nearest-even, or stochastic:
 *    round up iff u16 < frac * 65536); xhat = E2M1value(code) * s_eff (FP32,
 *    then nearest-even to BF16 when a BF16 output is asked for).
 *  STE mask ([QATREC] clipped straight-through estimator): bit = 1 iff
 *    |x| <= 6 * s_eff, i.e. x is inside the block's representable range.
 *  Stochastic rounding draw: Philox4x32-10 (Salmon et al., SC'11) with key =
 *    (seed low, seed high) and counter = (g low, g high, stream, offset),
 *    g = flat element index / 8 in the tensor being quantized (the transpose
 *    for the column-wise pass), stream 0 row-wise / 1 column-wise; element
 *    j = index % 8 takes 16-bit half (j % 2) of output word j / 2.
 *
 * Layouts (row-major, no padding; x of fq_quantize / fq_fakequant_ste and y of
 * fq_dequantize may have a row pitch ld >= cols, every other tensor is dense):
 *  x        [rows, cols] FP32 or BF16, row r starting at element r * ld.
 *  codes    [rows, cols/2] bytes; element 2j in the low nibble of byte j.
 *  scales   [rows, cols/B] bytes, B = 16 (NVFP4, double block) or 32 (MXFP4).
 *  tscale   NVFP4: 1 float (s_g); double block: [rows, cols/128] floats;
 *           MXFP4: not used (may be NULL).
 *  column-wise outputs describe the transpose X^T [cols, rows]:
 *           codes [cols, rows/2], scales [cols, rows/B], tscale as above.
 *  mask     ceil(rows*cols/8) bytes: bit (e % 8) of byte e / 8 holds flat
 *           element e (equivalently bit e % 32 of little-endian word e / 32).
 *
 * Conventions:
 *  - Every pointer argument to tensor data is a DEVICE pointer unless said
 *    otherwise; the caller allocates all of them.  Pointers to tensor data
 *    must be 16-byte aligned (FQ_ERR_ALIGN otherwise).  Where x, xhat, y or
 *    the GEMM's C (and its row pitch) are 32-byte aligned as well, the
 *    kernels move whole 32-byte sectors per access; the results are the same
 *    either way.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Calls are asynchronous on that stream: they never synchronise,
 *    never allocate device memory, and may return before the GPU finishes.
 *  - Argument errors are detected on the host and returned before any launch;
 *    nothing is written then.  A failed launch returns FQ_ERR_CUDA.
 *  - Inputs must be finite.  A block whose effective scale s_eff is non-zero
 *    but below 2^-128 has no finite FP32 reciprocal (x * (1 / s_eff) is
 *    infinite, and NaN for a zero element); such blocks are outside the
 *    contract.  For NVFP4 none occurs while the tensor amax (for the double
 *    block: each 1x128 block amax) is 0 or at least 2^-107.
 *  - Calls keep no state between them and may run concurrently on different
 *    streams with different workspaces.
 */
#ifndef FQ_H
#define FQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FQ_API __attribute__((visibility("default")))
#else
#define FQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FQ_OK = 0,
    FQ_ERR_INVALID_ARG = 1, /* NULL where a pointer is required, unknown enum value */
    FQ_ERR_SHAPE = 2,       /* dimension not a multiple of the block length, negative size */
    FQ_ERR_ALIGN = 3,       /* a tensor pointer is not 16-byte aligned */
    FQ_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than fq_workspace_size() */
    FQ_ERR_UNSUPPORTED = 5, /* valid but not implemented combination */
    FQ_ERR_CUDA = 6         /* a CUDA launch or memset failed */
} fq_status;

typedef enum { FQ_NVFP4 = 0, FQ_MXFP4 = 1, FQ_NVFP4_2LEVEL = 2 } fq_format;
typedef enum { FQ_RNE = 0, FQ_SR = 1 } fq_rounding;
typedef enum { FQ_ROW = 1, FQ_COL = 2, FQ_ROWCOL = 3 } fq_orient;
typedef enum { FQ_F32 = 0, FQ_BF16 = 1 } fq_dtype;

/* Quantizer configuration.  seed matters only for FQ_SR; offset for FQ_SR and
 * the Hadamard transform.
 * rht_seed != 0 turns on the random Hadamard transform of the backward
 * operands ([TJV2] §2C, OutControl): every 1x16 block along the quantization
 * direction (each 16x1 block for the column-wise output) becomes
 * z = (1/4) H16 (d . x) before it is quantized -- H16 the Sylvester Hadamard
 * matrix applied as butterflies of strides 1, 2, 4, 8 in FP32, d random signs
 * shared by all blocks: bit i of Philox4x32-10(key (rht_seed, 0), counter
 * (0, 0, 2, offset)) word 0 set means d_i = -1.  Operands quantized with the
 * same rht_seed and offset share one orthogonal transform, so their product
 * is unchanged.  Outputs (codes, scales, xhat, mask) describe z.  Supported
 * for FQ_MXFP4 and FQ_NVFP4_2LEVEL (no tensor-wide amax to transform first);
 * FQ_NVFP4 returns FQ_ERR_UNSUPPORTED. */
typedef struct {
    int32_t format;    /* fq_format */
    int32_t rounding;  /* fq_rounding */
    uint64_t seed;     /* Philox key of stochastic rounding */
    uint32_t offset;   /* Philox counter word 3, e.g. the training step */
    uint32_t rht_seed; /* 0: no Hadamard transform */
} fq_config;

/* A quantized tensor: device pointers, layouts as described above. */
typedef struct {
    uint8_t *codes;
    uint8_t *scales;
    float *tscale;
} fq_qtensor;

/* Bytes of device workspace that fq_quantize / fq_fakequant_ste need for a
 * [rows, cols] tensor in this configuration (NVFP4 keeps its tensor amax
 * there; the other formats need none and get 0).  Pure host function. */
FQ_API size_t fq_workspace_size(const fq_config *cfg, int64_t rows, int64_t cols);

/* Bytes of device workspace that fq_osci_update needs for `ntensors` tensors. */
FQ_API size_t fq_osci_workspace_size(int32_t ntensors);

/* Tensor amax ([TJV2] §2A names the per-tensor max|x| that NVFP4 needs):
 * amax_out[0] = max |x| over n elements (device float).  n must be a multiple
 * of 8.  The result is order-independent, hence identical to any sequential
 * evaluation. */
FQ_API fq_status fq_amax(const void *x, int32_t x_dtype, int64_t n, float *amax_out, void *stream);

/* Quantize x ([rows, cols]) -- [GPTOSS] NVFP4/MXFP4, [TJV2] §2A double block
 * and stochastic rounding.  orient selects the row-wise output (row_out), the
 * column-wise output on the transpose (col_out, [TJV2] §2A transposed 1x16
 * groups), or both from one read of x.  Shapes: cols % B == 0 for the row
 * pass (cols % 128 for the double block); rows % B == 0 for the column pass
 * (rows % 128 for the double block).  amax_in: optional device float holding
 * the tensor amax to use for NVFP4 (NULL: computed here into the workspace).
 * NVFP4 uses the same s_g for both orientations.
 * ld: elements between the starts of consecutive rows of x (ld == cols for a
 * dense tensor; larger for a column slice or a padded row).  ld < cols:
 * FQ_ERR_SHAPE; a row pitch (ld times the element size) that is not a
 * multiple of 16 bytes: FQ_ERR_ALIGN.  The outputs are always dense. */
FQ_API fq_status fq_quantize(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                      int64_t cols, int64_t ld, int32_t orient, const fq_qtensor *row_out,
                      const fq_qtensor *col_out, const float *amax_in, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Fake quantization with the straight-through-estimator mask ([QATREC]
 * "Detalhes técnicos"): xhat = dequant(quant(x)) in xhat_dtype, mask as
 * defined above (NULL: not written), both from the row-wise pass.  row_out
 * and col_out (NULL: not written) additionally receive the packed tensors,
 * so one call does the whole forward/backward quantization of an activation.
 * ld as for fq_quantize (the row pitch of x); xhat, mask and the packed
 * outputs are dense. */
FQ_API fq_status fq_fakequant_ste(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                           int64_t cols, int64_t ld, void *xhat, int32_t xhat_dtype, uint8_t *mask,
                           const fq_qtensor *row_out, const fq_qtensor *col_out,
                           const float *amax_in, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Dequantize a row-wise quantized [rows, cols] tensor: y = E2M1value(code) *
 * s_eff, in y_dtype.  Bit-identical to the xhat of fq_fakequant_ste.  ldy:
 * elements between the starts of consecutive rows of y (cols: dense); the
 * elements between cols and ldy of each row are not written.  ldy < cols:
 * FQ_ERR_SHAPE; a row pitch that is not a multiple of 16 bytes: FQ_ERR_ALIGN. */
FQ_API fq_status fq_dequantize(const fq_config *cfg, const fq_qtensor *q, int64_t rows, int64_t cols,
                        void *y, int32_t y_dtype, int64_t ldy, void *stream);

/* Straight-through-estimator backward ([QATREC]): dx = dy where the mask bit
 * is set, +0 elsewhere.  n elements, n % 8 == 0; dy/dx share dtype. */
FQ_API fq_status fq_ste_backward(const void *dy, int32_t dtype, const uint8_t *mask, int64_t n,
                          void *dx, void *stream);

/* One optimizer step with OsciReset statistics ([TJV2] §2B), over a group of
 * tensors (e.g. every expert matrix of an MoE layer).  Host arrays of length
 * ntensors hold the shapes and the device pointers of each tensor:
 *   master[i]   FP32 [rows, cols], updated in place: w_t = w_{t-1} + delta
 *   delta[i]    FP32 update for this step
 *   dist_m[i]   FP32, += |w_t - w_{t-1}|
 *   dist_q[i]   FP32, += |xhat_t - xhat_{t-1}|
 *   prev[i]     quantized w_{t-1} (read), next[i] quantized w_t (written);
 *               the caller swaps them between steps.  Initialise prev with
 *               fq_quantize of the initial master.
 *   xhat[i]     fake-quantized w_t in xhat_dtype (NULL array or entry: skip)
 *   mask[i]     STE mask of w_t (NULL array or entry: skip)
 * Quantization follows cfg (NVFP4 takes s_g from amax(w_t)).  cols must be a
 * multiple of the block length.  The workspace holds one float per tensor
 * (fq_osci_workspace_size): the NVFP4 step keeps amax(w_t) there between its
 * two passes over the weights; MXFP4 and the double block, whose scales are
 * block-local, make one pass and leave it untouched. */
FQ_API fq_status fq_osci_update(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                         const int64_t *cols, float *const *master, const float *const *delta,
                         float *const *dist_q, float *const *dist_m, const fq_qtensor *prev,
                         const fq_qtensor *next, void *const *xhat, int32_t xhat_dtype,
                         uint8_t *const *mask, void *workspace, size_t workspace_bytes,
                         void *stream);

/* fq_osci_update for the last step of an OsciReset window ([TJV2] §2B): the
 * update, then in the same pass over the weights the reset that
 * fq_osci_reset would apply to this step's result -- where the new
 * dist_Q > threshold * dist_M (FP32 product, strict) the master weight becomes
 * xhat_t (FP32), and dist_Q and dist_M are left at zero for every weight.
 * Bit-identical to fq_osci_update followed by fq_osci_reset(cur = next), but
 * it reads dist_M once more instead of making a separate pass over both
 * accumulators.  Outputs (next, xhat, mask) describe w_t before the reset.
 * n_reset (device uint64, may be NULL) receives the number of weights reset. */
FQ_API fq_status fq_osci_update_reset(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                                      const int64_t *cols, float *const *master,
                                      const float *const *delta, float *const *dist_q,
                                      float *const *dist_m, const fq_qtensor *prev,
                                      const fq_qtensor *next, void *const *xhat,
                                      int32_t xhat_dtype, uint8_t *const *mask, float threshold,
                                      unsigned long long *n_reset, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* fq_osci_update without a workspace argument.  The pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate device
 * memory where they run the optimizer step (a framework whose allocator owns
 * all device memory, a plugin that only receives its tensors, a process that
 * forbids cudaMalloc after start-up).  The per-tensor amax scratch lives in a
 * file-scope device array of FQ_NOALLOC_MAX_TENSORS floats (256 bytes) that
 * every GPU which loads the library keeps until the process exits; the caller
 * still passes all inputs and outputs, and nothing here allocates.
 *  - At most FQ_NOALLOC_MAX_TENSORS tensors per call; more returns
 *    FQ_ERR_WORKSPACE before anything runs.  Otherwise arguments, results and
 *    errors are those of fq_osci_update.
 *  - The first call on each device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress); make that first call before
 *    any stream capture.  The address is kept for the life of the process:
 *    it belongs to the device's primary context, so after cudaDeviceReset
 *    (which destroys that context and the array with it) this entry point
 *    must not be called again in that process.
 *  - Every call shares the one array; each call clears the slots it uses on
 *    its stream before using them, but calls that overlap on the GPU (other
 *    streams, other threads) race on it. */
#define FQ_NOALLOC_MAX_TENSORS 64
FQ_API fq_status fq_osci_update_noalloc(const fq_config *cfg, int32_t ntensors,
                                        const int64_t *rows, const int64_t *cols,
                                        float *const *master, const float *const *delta,
                                        float *const *dist_q, float *const *dist_m,
                                        const fq_qtensor *prev, const fq_qtensor *next,
                                        void *const *xhat, int32_t xhat_dtype,
                                        uint8_t *const *mask, void *stream);

/* End of an OsciReset window ([TJV2] §2B): where dist_Q > threshold * dist_M
 * (FP32 product, strict), the master weight is set to xhat_t decoded from cur
 * (the quantized value of its current bin); dist_Q and dist_M are then zeroed
 * for every weight.  n_reset (device uint64, may be NULL) receives the number
 * of weights reset.  Deciding when the learning rate is low enough to call
 * this is the caller's schedule. */
FQ_API fq_status fq_osci_reset(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                        const int64_t *cols, float *const *master, float *const *dist_q,
                        float *const *dist_m, const fq_qtensor *cur, float threshold,
                        unsigned long long *n_reset, void *stream);

/* ---- Static outlier retention ([TJV2] §2C, OutControl) -------------------
 * A few activation channels (columns of a [rows, cols] activation, the
 * reduction dimension of the GEMM that consumes it) carry values far larger
 * than the rest; inside a 1x16 block they set the block scale and crush the
 * other fifteen elements to zero.  OutControl keeps the channels with the
 * largest norm over a short calibration window in FP8 and quantizes the rest
 * of the activation to FP4 with those channels removed.  This library's
 * readings: the norm is max |x| per channel; the k channels with the largest
 * amax are kept (equal amax: lower index first); each kept channel c has the
 * static FP8 scale s_c = amax_c / 448 (FP32 division) and is stored as E4M3
 * (OCP "FN", nearest-even, saturating at 448) of y = x * (1 / s_c); the FP4
 * part is the row-wise quantization of x with the kept columns set to +0.
 * Channel counts are limited to FQ_MAX_CHANNELS (FQ_ERR_SHAPE beyond). */
#define FQ_MAX_CHANNELS 131072

/* Calibration: amax_inout[c] = max(amax_inout[c], max_r |x[r, c]|) for a
 * [rows, cols] activation, so that consecutive calls over the calibration
 * batches accumulate the window's per-channel amax (zero-fill amax_inout,
 * cols floats, before the first).  cols % 16 == 0.  amax_inout must hold
 * non-negative values (atomic max on the FP32 bit patterns). */
FQ_API fq_status fq_channel_amax(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                                 float *amax_inout, void *stream);

/* Selection: the k channels with the largest channel_amax (non-negative;
 * ties go to the lower index), 0 <= k <= cols (FQ_ERR_INVALID_ARG outside).
 * Writes idx[k] (int32, ascending channel indices), bitmap[ceil(cols/32)]
 * (bit c % 32 of word c / 32 set iff channel c is kept; unused high bits of
 * the last word are zero) and fp8_scale[k] = channel_amax[idx[j]] / 448.
 * idx and fp8_scale may be NULL when k == 0.  One CTA on the GPU. */
FQ_API fq_status fq_select_channels(const float *channel_amax, int64_t cols, int64_t k,
                                    int32_t *idx, uint32_t *bitmap, float *fp8_scale,
                                    void *stream);

/* Split quantization of a [rows, cols] activation under the kept channels
 * (bitmap and fp8_scale as fq_select_channels writes them; the bitmap must
 * have exactly k bits set -- a kept channel's rank among the set bits indexes
 * fp8_scale and the FP8 columns).  Writes, each optional (NULL: skipped):
 *   out   row-wise FP4 codes / scales / tscale of x with the kept columns
 *         zeroed (layouts as fq_quantize; NVFP4 takes s_g from the amax of
 *         that zeroed tensor);
 *   fp8   [rows, k] bytes: sign | E4M3(|x * (1 / s_j)|) of the kept elements,
 *         column j holding the j-th kept channel;
 *   xhat  the fake-quantized activation in xhat_dtype: the FP4 value for
 *         ordinary elements, E4M3value * s_j (sign applied) for kept ones;
 *   mask  STE mask: the FP4 rule for ordinary elements, |x| <= 448 * s_j for
 *         kept ones.
 * cols % B == 0 (cols % 128 for the double block).  rht_seed must be 0
 * (FQ_ERR_UNSUPPORTED: OutControl retains outliers on the forward operands
 * and transforms the backward ones).  The workspace is that of
 * fq_workspace_size (NVFP4: the masked tensor amax). */
FQ_API fq_status fq_quantize_outliers(const fq_config *cfg, const void *x, int32_t x_dtype,
                                      int64_t rows, int64_t cols, const uint32_t *bitmap,
                                      int64_t k, const float *fp8_scale, const fq_qtensor *out,
                                      uint8_t *fp8, void *xhat, int32_t xhat_dtype,
                                      uint8_t *mask, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* ---- QAD distillation loss ([QADP] §2; [QATREC] "Detalhes técnicos") ------
 * For each row r of [rows, vocab] teacher logits zt and student logits zs
 * (both FP32 or both BF16, dtype):
 *   p = softmax(zt[r] / T), q = softmax(zs[r] / T),
 *   loss_rows[r] = KL(p || q) = sum_v p_v log(p_v / q_v)      (FP32, nats)
 *   loss_mean[0] = mean over rows of loss_rows                (optional)
 *   dstudent[r, v] = grad_scale * (q_v - p_v) / T             (optional, in
 *                    dstudent_dtype; the gradient of grad_scale * loss_rows[r]
 *                    with respect to zs[r, v] -- grad_scale = 1 / rows gives
 *                    the gradient of loss_mean).
 * The pages fix T = 1; other T > 0 divide the logits.  Computed in FP32 from
 * one read of each tensor (row maxima, sums of exponentials, then the terms):
 * results differ from exact arithmetic by rounding only (a few units of 1e-6
 * relative in p and q; KL to about 1e-6 absolute for vocabularies of 1e5).
 * vocab % 8 == 0 (FQ_ERR_SHAPE), vocab <= about 450000 BF16 or 225000 FP32
 * logits (FQ_ERR_UNSUPPORTED beyond: a row must fit the shared memory of one
 * 8-CTA cluster).  Logits must be finite; temperature finite and > 0.
 * err (device int32, may be NULL) is OR-ed with 1 if a copy into shared
 * memory did not complete within 2 s (results then undefined); the caller
 * zeroes it and reads it after synchronising.  rows == 0 writes only
 * loss_mean (0); the tensor pointers may then be NULL. */
FQ_API fq_status fq_qad_kl(const void *teacher, const void *student, int32_t dtype, int64_t rows,
                           int64_t vocab, float temperature, float grad_scale, float *loss_rows,
                           float *loss_mean, void *dstudent, int32_t dstudent_dtype,
                           int32_t *err, void *stream);

/* ---- Block-scaled FP4 GEMM ([GPTOSS] "O que há de novo"; [TJV2] §2A) ------
 * C[m, n] = alpha sum_k (v(a_mk) e(sa_m,k/B)) (v(b_nk) e(sb_n,k/B)) for
 * operands quantized row-wise along the shared reduction dimension k (A is
 * [m, k], e.g. an activation; B is [n, k], e.g. a weight; both exactly as
 * fq_quantize / fq_fakequant_ste write them): the GEMM of the dequantized
 * operands, computed on the tensor cores (FP4 products with their block
 * scales, FP32 accumulation).  cfg->format selects FQ_NVFP4 (E4M3 scales per
 * 1x16, alpha = s_A s_B, the two tensor scales, applied in FP32) or FQ_MXFP4
 * (E8M0 scales per 1x32, alpha = 1); the double block returns
 * FQ_ERR_UNSUPPORTED.  C is dense row-major [m, n] in c_dtype.
 * n % 32 == 0 and k % 32 == 0 (FQ_ERR_SHAPE); m is free.  Tiles are 128 x
 * 128 x 256: the parts of a tile past m, n or k are zero-filled, so any such
 * shape runs (for example gpt-oss's 2880 and 5760).  Results equal
 * the exact product up to FP32 accumulation (and the BF16 rounding of C).
 * The workspace (fq_gemm_workspace_size bytes, 16-byte aligned) receives
 * both operands' block scales rearranged into the tensor cores' layout; it
 * is scratch, owned by the caller.  err (device int32, may be NULL) is OR-ed
 * with 1 if an internal pipeline wait timed out (C is then undefined). */
FQ_API size_t fq_gemm_workspace_size(int64_t m, int64_t n, int64_t k);
FQ_API fq_status fq_gemm(const fq_config *cfg, const fq_qtensor *a, const fq_qtensor *b,
                         int64_t m, int64_t n, int64_t k, void *c, int32_t c_dtype,
                         void *workspace, size_t workspace_bytes, int32_t *err, void *stream);

/* Static description of a status code. */
FQ_API const char *fq_status_string(fq_status status);

#ifdef __cplusplus
}
#endif

#endif /* FQ_H */
