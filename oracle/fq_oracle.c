/*
 * fq_oracle.c -- reference implementation of block-scaled FP4 fake-quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load it; the library itself never calls it, and it
 * shares no code, header, table or constant generator with the CUDA sources.
 *
 * Style: plain scalar C, one element at a time, in the order the definitions
 * state.  Every floating-point step that decides a stored bit is a single
 * IEEE-754 binary32 operation rounded to nearest-even (built with
 * -ffp-contract=off, so no fused multiply-add), because the formats fix FP32
 * for the tensor scale, the outer-block scale and the dequantized output.
 * Grid searches (nearest E2M1 / E4M3 value) are brute force over every code,
 * with distances taken in binary64, which is exact for the values involved.
 *
 * Sources (web pages on FP4 quantization-aware training):
 *  - "Aprimorando gpt-oss para Precisão e Desempenho com Treinamento Consciente
 *    à Quantização", TL;DR and "O que há de novo": MXFP4 and NVFP4 are the two
 *    FP4 formats; NVFP4 uses FP8 E4M3 block scales.
 *  - "Resumo Técnico: TetraJet-v2", §2A: NVFP4 groups of 16 elements with an
 *    8-bit scale; double-block quantization (128-element outer block scaled
 *    "globally", 16-element inner blocks scaled "locally"); stochastic rounding
 *    with E[round(x)] = x in the backward pass; 1x16 groups whose transpose
 *    needs its own alignment.  §2B: OsciReset (risk = dist_Q / dist_M, reset
 *    the master weight to the centre of its current bin).
 *  - "Como o Treinamento com Quantização Detecta e Recupera Precisão em
 *    Inferência de Baixa Precisão", "Detalhes técnicos": fake quantization
 *    (quantize/dequantize held in a high-precision type) with a
 *    straight-through estimator that exposes rounding and clipping.
 * The pages do not print the E2M1 grid, the E4M3/E8M0 layouts, the MXFP4 block
 * size, the NVFP4 tensor scale, the packing order or the random-number
 * recipe; the readings used here are the ones listed beside each function.
 *
 * Parity status: every function below is pinned by tests that do not reuse
 * this file's arithmetic (exact-rational tables, torch's float8 and bfloat16
 * casts, cuRAND's host Philox generator, hand-worked blocks, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define FQO_NVFP4 0
#define FQO_MXFP4 1
#define FQO_NVFP4_2LEVEL 2
#define FQO_RNE 0
#define FQO_SR 1

#define FQO_OK 0
#define FQO_ERR_SHAPE 2
#define FQO_ERR_ARG 1

/* ------------------------------------------------------------------------ */
/* E2M1 element.  Reading: bit 3 sign, bits 2..1 exponent (bias 1), bit 0     */
/* mantissa, giving magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; no Inf or NaN.     */
/* ------------------------------------------------------------------------ */
static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float fqo_e2m1_value(int code)
{
    float v = E2M1_MAG[code & 7];
    return (code & 8) ? -v : v;
}

/* Round y to the nearest E2M1 value, ties to the even code, |y| >= 6 saturates
 * to 6.  The sign bit is copied from y, also when the result is zero. */
int fqo_e2m1_round_nearest(float y)
{
    int sign = signbit(y) ? 8 : 0;
    double a = fabs((double)y);
    int best = 0;
    if (a >= 6.0) {
        best = 7;
    } else {
        double bestd = a;
        for (int c = 1; c < 8; c++) {
            double d = fabs(a - (double)E2M1_MAG[c]);
            if (d < bestd || (d == bestd && (c & 1) == 0)) {
                best = c;
                bestd = d;
            }
        }
    }
    return sign | best;
}

/* Stochastic rounding ("Resumo Técnico: TetraJet-v2", §2A: E[round(x)] = x).
 * Reading: with lo the largest grid magnitude <= |y| and hi the next one,
 * round up iff the 16-bit uniform u satisfies (float)u < frac * 65536, where
 * frac = (|y| - lo) / (hi - lo) (exact: Sterbenz and a power-of-two gap).
 * |y| >= 6 saturates to 6.  The sign is copied. */
int fqo_e2m1_round_stochastic(float y, unsigned u)
{
    int sign = signbit(y) ? 8 : 0;
    float a = fabsf(y);
    if (a >= 6.0f)
        return sign | 7;
    int lo = 0;
    for (int c = 1; c < 8; c++)
        if (E2M1_MAG[c] <= a)
            lo = c;
    float gap = E2M1_MAG[lo + 1] - E2M1_MAG[lo];
    float frac = (a - E2M1_MAG[lo]) / gap;
    int up = (float)(u & 0xFFFFu) < frac * 65536.0f;
    return sign | (lo + up);
}

/* ------------------------------------------------------------------------ */
/* E4M3 scale byte.  Reading: the OCP "FN" variant -- bias 7, subnormals     */
/* (m/8)*2^-6, normals (1+m/8)*2^(e-7), no Inf, 0x7F/0xFF are NaN, max 448.   */
/* ------------------------------------------------------------------------ */
float fqo_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    float v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexpf((float)m, -9);
    else
        v = ldexpf((float)(8 + m), e - 10);
    return s ? -v : v;
}

/* Encode a non-negative finite scale: nearest E4M3 value, ties to the even
 * code, anything >= 448 saturates to 448 (code 0x7E). */
int fqo_e4m3_encode(float s)
{
    if (s >= 448.0f)
        return 0x7E;
    int best = 0;
    double bestd = fabs((double)s);
    for (int c = 1; c <= 0x7E; c++) {
        double d = fabs((double)s - (double)fqo_e4m3_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* E8M0 scale byte (MXFP4): value 2^(code-127); 0xFF is NaN.                  */
/* ------------------------------------------------------------------------ */
float fqo_e8m0_value(int code)
{
    if ((code & 0xFF) == 0xFF)
        return NAN;
    return ldexpf(1.0f, (code & 0xFF) - 127);
}

/* MXFP4 shared exponent: k = floor(log2 amax) - 2 (2 = largest E2M1 exponent),
 * clamped to [-127, 127]; amax = 0 gives the smallest code. */
int fqo_e8m0_for_amax(float amax)
{
    int k;
    if (amax == 0.0f)
        k = -127;
    else
        k = ilogbf(amax) - 2;
    if (k < -127)
        k = -127;
    if (k > 127)
        k = 127;
    return k + 127;
}

/* ------------------------------------------------------------------------ */
/* bfloat16: nearest value, ties to even (used for the dequantized output).   */
/* ------------------------------------------------------------------------ */
uint16_t fqo_bf16_from_f32(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    if (isnan(x))
        return (uint16_t)((b >> 16) | 0x40);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

void fqo_bf16_from_f32_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = fqo_bf16_from_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies per      */
/* round, the key bumped by the Weyl constants between rounds.               */
/* ------------------------------------------------------------------------ */
void fqo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* The 16-bit uniform for element `idx` of the tensor being quantized.
 * Reading: key = (seed low word, seed high word); counter = (g low, g high,
 * stream, offset) with g = idx / 8; element j = idx mod 8 takes the low (j
 * even) or high (j odd) half of output word j / 2.  stream is 0 for the
 * row-wise pass and 1 for the column-wise pass; offset is the caller's
 * per-call counter (e.g. the training step). */
unsigned fqo_sr_draw(uint64_t seed, uint64_t idx, uint32_t stream, uint32_t offset)
{
    uint64_t g = idx / 8;
    unsigned j = (unsigned)(idx % 8);
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), stream, offset};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    fqo_philox4x32_10(ctr, key, out);
    return (out[j / 2] >> (16 * (j % 2))) & 0xFFFFu;
}

/* ------------------------------------------------------------------------ */
/* Random Hadamard transform ("Resumo Técnico: TetraJet-v2", §2C: RHT on the  */
/* backward operands spreads outlier energy across channels).  Reading: a     */
/* 16-point transform along each quantization block, z = (1/4) H16 (d . x),   */
/* with the random signs d shared by every block of the call.  The butterfly  */
/* order is fixed (strides 1, 2, 4, 8; a, b -> a + b, a - b), each step one    */
/* FP32 addition, then the exact scaling by 1/4.                              */
/* ------------------------------------------------------------------------ */

/* The 16 sign bits: bit i set means d_i = -1.  Drawn from Philox with key
 * (rht_seed, 0) and counter (0, 0, 2, offset); the low 16 bits of word 0. */
unsigned fqo_rht_signs(uint32_t rht_seed, uint32_t offset)
{
    uint32_t ctr[4] = {0, 0, 2, offset};
    uint32_t key[2] = {rht_seed, 0};
    uint32_t out[4];
    fqo_philox4x32_10(ctr, key, out);
    return out[0] & 0xFFFFu;
}

void fqo_rht16(float *z, unsigned signs)
{
    for (int i = 0; i < 16; i++)
        if ((signs >> i) & 1u)
            z[i] = -z[i];
    for (int h = 1; h < 16; h *= 2) {
        for (int i = 0; i < 16; i++) {
            if (i & h)
                continue;
            float a = z[i], b = z[i + h];
            z[i] = a + b;
            z[i + h] = a - b;
        }
    }
    for (int i = 0; i < 16; i++)
        z[i] = z[i] * 0.25f;
}

/* Applies fqo_rht16 to every 1x16 block of a dense [rows, cols] array in place. */
void fqo_rht_rows(float *x, int64_t rows, int64_t cols, uint32_t rht_seed, uint32_t offset)
{
    unsigned signs = fqo_rht_signs(rht_seed, offset);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c + 16 <= cols; c += 16)
            fqo_rht16(x + r * cols + c, signs);
}

/* ------------------------------------------------------------------------ */
/* Tensor operations.                                                         */
/* ------------------------------------------------------------------------ */
float fqo_amax(const float *x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > m)
            m = a;
    }
    return m;
}

static int block_len(int fmt)
{
    return fmt == FQO_MXFP4 ? 32 : 16;
}

/* Row-wise block quantization of a dense row-major [rows, cols] FP32 tensor.
 *
 * fmt NVFP4 (1x16, E4M3 scale, FP32 tensor scale):
 *     s_g   = tensor_amax / (6 * 448)                 -> tscale[0]
 *     s_b   = (block_amax / 6) / s_g   (0 if s_g = 0)  -> E4M3, nearest-even,
 *                                                        saturating at 448
 *     s_eff = E4M3value(s_b code) * s_g;  r = 1 / s_eff (0 if s_eff = 0)
 * fmt NVFP4_2LEVEL ("Resumo Técnico: TetraJet-v2", §2A): as NVFP4 with s_g
 *     replaced by the outer-block scale s_o = amax_128 / (6 * 448), one per
 *     1x128 block                                       -> tscale[rows, cols/128]
 * fmt MXFP4 (1x32, E8M0 scale): k = floor(log2 block_amax) - 2 clamped to
 *     [-127, 127]; s_eff = 2^k, r = 2^-k.
 * Every element: y = x * r; code = nearest-even E2M1 (or stochastic with the
 * draw for its flat index); xhat = E2M1value(code) * s_eff.  STE mask bit
 * (clipped straight-through estimator): 1 iff |x| <= 6 * s_eff, i.e. x lies
 * inside the block's representable range [-6 s_eff, 6 s_eff] (FP32 product).
 *
 * Outputs: codes [rows, cols/2] (element 2j in the low nibble of byte j),
 * scales [rows, cols/B], mask bit i of word w = flat element 32w + i (optional),
 * xhat FP32 (optional).  Returns FQO_ERR_SHAPE if cols is not a multiple of
 * the block length. */
int fqo_quantize_rows(int fmt, int rounding, uint64_t seed, uint32_t offset, uint32_t stream,
                      const float *x, int64_t rows, int64_t cols, float tensor_amax,
                      uint8_t *codes, uint8_t *scales, float *tscale, float *xhat,
                      uint32_t *mask)
{
    int B = block_len(fmt);
    if (fmt != FQO_NVFP4 && fmt != FQO_MXFP4 && fmt != FQO_NVFP4_2LEVEL)
        return FQO_ERR_ARG;
    if (rounding != FQO_RNE && rounding != FQO_SR)
        return FQO_ERR_ARG;
    if (rows < 0 || cols < 0 || cols % B != 0)
        return FQO_ERR_SHAPE;
    if (fmt == FQO_NVFP4_2LEVEL && cols % 128 != 0)
        return FQO_ERR_SHAPE;
    int64_t n = rows * cols;
    memset(codes, 0, (size_t)(n / 2));
    if (mask)
        memset(mask, 0, (size_t)((n + 31) / 32) * 4);

    float s_g = 0.0f;
    if (fmt == FQO_NVFP4) {
        s_g = tensor_amax / 2688.0f;
        tscale[0] = s_g;
    }

    for (int64_t r = 0; r < rows; r++) {
        float s_outer = s_g;
        for (int64_t c0 = 0; c0 < cols; c0 += B) {
            const float *xb = x + r * cols + c0;
            int64_t e0 = r * cols + c0;

            if (fmt == FQO_NVFP4_2LEVEL && c0 % 128 == 0) {
                float amax128 = fqo_amax(xb, 128);
                s_outer = amax128 / 2688.0f;
                tscale[r * (cols / 128) + c0 / 128] = s_outer;
            }

            float amax_b = fqo_amax(xb, B);
            int sc;
            float s_eff, recip;
            if (fmt == FQO_MXFP4) {
                sc = fqo_e8m0_for_amax(amax_b);
                s_eff = ldexpf(1.0f, sc - 127);
                recip = ldexpf(1.0f, 127 - sc);
            } else {
                float s_b = 0.0f;
                if (s_outer != 0.0f)
                    s_b = (amax_b / 6.0f) / s_outer;
                sc = fqo_e4m3_encode(s_b);
                s_eff = fqo_e4m3_value(sc) * s_outer;
                recip = (s_eff == 0.0f) ? 0.0f : 1.0f / s_eff;
            }
            scales[e0 / B] = (uint8_t)sc;

            for (int i = 0; i < B; i++) {
                int64_t e = e0 + i;
                float y = xb[i] * recip;
                int code;
                if (rounding == FQO_SR)
                    code = fqo_e2m1_round_stochastic(y, fqo_sr_draw(seed, (uint64_t)e, stream, offset));
                else
                    code = fqo_e2m1_round_nearest(y);
                codes[e / 2] |= (uint8_t)(code << (4 * (e % 2)));
                if (xhat)
                    xhat[e] = fqo_e2m1_value(code) * s_eff;
                if (mask && fabsf(xb[i]) <= 6.0f * s_eff)
                    mask[e / 32] |= 1u << (e % 32);
            }
        }
    }
    return FQO_OK;
}

/* Dequantize codes + scales back to FP32 with the same s_eff as the quantizer:
 * xhat = E2M1value(code) * s_eff. */
int fqo_dequantize_rows(int fmt, const uint8_t *codes, const uint8_t *scales,
                        const float *tscale, int64_t rows, int64_t cols, float *xhat)
{
    int B = block_len(fmt);
    if (fmt != FQO_NVFP4 && fmt != FQO_MXFP4 && fmt != FQO_NVFP4_2LEVEL)
        return FQO_ERR_ARG;
    if (rows < 0 || cols < 0 || cols % B != 0)
        return FQO_ERR_SHAPE;
    if (fmt == FQO_NVFP4_2LEVEL && cols % 128 != 0)
        return FQO_ERR_SHAPE;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) {
            int64_t e = r * cols + c;
            int sc = scales[e / B];
            float s_eff;
            if (fmt == FQO_MXFP4)
                s_eff = fqo_e8m0_value(sc);
            else if (fmt == FQO_NVFP4)
                s_eff = fqo_e4m3_value(sc) * tscale[0];
            else
                s_eff = fqo_e4m3_value(sc) * tscale[r * (cols / 128) + c / 128];
            int code = (codes[e / 2] >> (4 * (e % 2))) & 0xF;
            xhat[e] = fqo_e2m1_value(code) * s_eff;
        }
    }
    return FQO_OK;
}

/* Straight-through estimator backward ("Como o Treinamento com Quantização...",
 * "Detalhes técnicos": gradients pass through the quantize/dequantize operator;
 * clipped elements are exposed through the mask): dx = dy where the mask bit
 * is set, else +0.  Works on raw element bits of width 2 or 4 bytes. */
void fqo_ste_backward(const void *dy, const uint32_t *mask, int64_t n, int elem_bytes, void *dx)
{
    for (int64_t i = 0; i < n; i++) {
        int pass = (mask[i / 32] >> (i % 32)) & 1u;
        if (elem_bytes == 2) {
            uint16_t v = ((const uint16_t *)dy)[i];
            ((uint16_t *)dx)[i] = pass ? v : 0;
        } else {
            uint32_t v = ((const uint32_t *)dy)[i];
            ((uint32_t *)dx)[i] = pass ? v : 0;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Static outlier retention ("Resumo Técnico: TetraJet-v2", §2C, OutControl:  */
/* the top p% channels by norm, found in a short calibration window, stay in  */
/* higher precision -- e.g. FP8 -- in both passes; the rest stays FP4).       */
/* Readings: channel = column of an activation [tokens, channels]; the norm   */
/* is the L-infinity norm (max |x|) over the calibration window; ties go to   */
/* the lower channel index; the retained channels use FP8 E4M3 with a static  */
/* per-channel scale s_c = amax_c / 448; the FP4 part quantizes the tensor    */
/* with the retained columns set to +0.                                       */
/* ------------------------------------------------------------------------ */

/* amax[c] = max(amax[c], max over rows |x[r, c]|): a running maximum. */
void fqo_channel_amax(const float *x, int64_t rows, int64_t cols, float *amax)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            float a = fabsf(x[r * cols + c]);
            if (a > amax[c])
                amax[c] = a;
        }
}

/* The k channels with the largest amax (ties: lower index first), returned in
 * ascending index order, plus the bitmap (bit c % 32 of word c / 32) and the
 * FP8 scale amax_c / 448 of each selected channel. */
int fqo_select_channels(const float *amax, int64_t cols, int64_t k, int32_t *idx,
                        uint32_t *bitmap, float *fp8_scale)
{
    if (k < 0 || k > cols)
        return FQO_ERR_ARG;
    memset(bitmap, 0, (size_t)((cols + 31) / 32) * 4);
    for (int64_t j = 0; j < k; j++) {
        int64_t best = -1;
        for (int64_t c = 0; c < cols; c++) {
            if ((bitmap[c / 32] >> (c % 32)) & 1u)
                continue;
            if (best < 0 || amax[c] > amax[best])
                best = c;
        }
        bitmap[best / 32] |= 1u << (best % 32);
    }
    int64_t j = 0;
    for (int64_t c = 0; c < cols; c++)
        if ((bitmap[c / 32] >> (c % 32)) & 1u) {
            idx[j] = (int32_t)c;
            fp8_scale[j] = amax[c] / 448.0f;
            j++;
        }
    return FQO_OK;
}

/* Split fake-quantization.  The FP4 part is fqo_quantize_rows of x with the
 * retained columns zeroed (NVFP4: tensor amax of that tensor).  Retained
 * column c (the j-th selected) gets y = x * r_j, r_j = 1 / s_j (0 if s_j = 0),
 * code = sign | E4M3 nearest-even saturating of |y| into fp8[r, j],
 * xhat = E4M3value(code) * s_j, mask bit = |x| <= 448 * s_j. */
int fqo_quantize_outliers(int fmt, int rounding, uint64_t seed, uint32_t offset,
                          const float *x, int64_t rows, int64_t cols, const int32_t *idx,
                          int64_t k, const float *fp8_scale, float *xz_scratch,
                          uint8_t *codes, uint8_t *scales, float *tscale, uint8_t *fp8,
                          float *xhat, uint32_t *mask)
{
    int64_t n = rows * cols;
    memcpy(xz_scratch, x, (size_t)n * 4);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < k; j++)
            xz_scratch[r * cols + idx[j]] = 0.0f;
    float amax = fqo_amax(xz_scratch, n);
    int st = fqo_quantize_rows(fmt, rounding, seed, offset, 0, xz_scratch, rows, cols, amax,
                               codes, scales, tscale, xhat, mask);
    if (st != FQO_OK)
        return st;
    for (int64_t j = 0; j < k; j++) {
        float s = fp8_scale[j];
        float rcp = (s == 0.0f) ? 0.0f : 1.0f / s;
        float lim = 448.0f * s;
        for (int64_t r = 0; r < rows; r++) {
            int64_t e = r * cols + idx[j];
            float y = x[e] * rcp;
            int code = fqo_e4m3_encode(fabsf(y)) | (signbit(y) ? 0x80 : 0);
            fp8[r * k + j] = (uint8_t)code;
            if (xhat)
                xhat[e] = fqo_e4m3_value(code) * s;
            if (mask) {
                if (fabsf(x[e]) <= lim)
                    mask[e / 32] |= 1u << (e % 32);
                else
                    mask[e / 32] &= ~(1u << (e % 32));
            }
        }
    }
    return FQO_OK;
}

/* ------------------------------------------------------------------------ */
/* OsciReset ("Resumo Técnico: TetraJet-v2", §2B).                            */
/* ------------------------------------------------------------------------ */

/* One optimizer step on one tensor, with the oscillation statistics:
 *   w_t = w_{t-1} + delta;            dist_M += |w_t - w_{t-1}|
 *   xhat_t = fake-quant(w_t) (fmt/rounding as given; NVFP4 tensor scale from
 *            amax(w_t));              dist_Q += |xhat_t - xhat_{t-1}|
 * where xhat_{t-1} is decoded from the previous codes/scales/tscale.  New
 * codes, scales and tscale go to the *_new buffers; xhat_t (FP32) and the
 * mask are returned when the pointers are non-NULL.  master, dist_q and
 * dist_m are updated in place. */
int fqo_osci_step(int fmt, int rounding, uint64_t seed, uint32_t offset,
                  float *master, const float *delta, float *dist_q, float *dist_m,
                  const uint8_t *codes_prev, const uint8_t *scales_prev, const float *tscale_prev,
                  uint8_t *codes_new, uint8_t *scales_new, float *tscale_new,
                  int64_t rows, int64_t cols, float *xhat, uint32_t *mask,
                  float *xhat_prev_scratch)
{
    int64_t n = rows * cols;
    for (int64_t i = 0; i < n; i++) {
        float w_old = master[i];
        float w_new = w_old + delta[i];
        dist_m[i] = dist_m[i] + fabsf(w_new - w_old);
        master[i] = w_new;
    }
    float amax = fqo_amax(master, n);
    int st = fqo_quantize_rows(fmt, rounding, seed, offset, 0, master, rows, cols, amax,
                               codes_new, scales_new, tscale_new, xhat, mask);
    if (st != FQO_OK)
        return st;
    st = fqo_dequantize_rows(fmt, codes_prev, scales_prev, tscale_prev, rows, cols,
                             xhat_prev_scratch);
    if (st != FQO_OK)
        return st;
    for (int64_t i = 0; i < n; i++)
        dist_q[i] = dist_q[i] + fabsf(xhat[i] - xhat_prev_scratch[i]);
    return FQO_OK;
}

/* End of an observation window: where dist_Q > threshold * dist_M (strict),
 * the master weight goes to the quantized value of its current bin (xhat_t,
 * decoded from the current codes/scales/tscale -- the plainest reading of
 * "centre of its current quantization bin"); both accumulators are then
 * cleared for every weight.  Returns the number of weights reset. */
int64_t fqo_osci_reset(int fmt, float *master, float *dist_q, float *dist_m,
                       const uint8_t *codes, const uint8_t *scales, const float *tscale,
                       int64_t rows, int64_t cols, float threshold, float *xhat_scratch)
{
    int64_t n = rows * cols, count = 0;
    if (fqo_dequantize_rows(fmt, codes, scales, tscale, rows, cols, xhat_scratch) != FQO_OK)
        return -1;
    for (int64_t i = 0; i < n; i++) {
        if (dist_q[i] > threshold * dist_m[i]) {
            master[i] = xhat_scratch[i];
            count++;
        }
        dist_q[i] = 0.0f;
        dist_m[i] = 0.0f;
    }
    return count;
}

/* ------------------------------------------------------------------------ */
/* QAD distillation loss ("Quantization-Aware Distillation for NVFP4         */
/* Inference Accuracy Recovery", §2 Metodologia: KL divergence between the   */
/* BF16 teacher's and the NVFP4 student's output distributions, softmax      */
/* temperature T = 1).  Double precision throughout.                        */
/* ------------------------------------------------------------------------ */

/* log of the sum of exp over n values, shifted by their maximum */
static double fqo_logsumexp(const double *v, int64_t n)
{
    double m = v[0];
    for (int64_t i = 1; i < n; i++)
        if (v[i] > m)
            m = v[i];
    double s = 0.0;
    for (int64_t i = 0; i < n; i++)
        s += exp(v[i] - m);
    return m + log(s);
}

/* For each row r of the [rows, vocab] teacher logits zt and student logits
 * zs: p = softmax(zt / T), q = softmax(zs / T),
 *   loss_rows[r] = KL(p || q) = sum_v p_v (log p_v - log q_v),
 *   dz[r, v]     = g * (q_v - p_v) / T   (the gradient of g * loss_rows[r]
 *                                         with respect to zs[r, v]).
 * and *loss_mean = the mean of loss_rows over the rows (0 for no rows).
 * dz may be NULL.  scratch holds 2 * vocab doubles. */
int fqo_qad_kl(const float *zt, const float *zs, int64_t rows, int64_t vocab, double temperature,
               double g, double *loss_rows, double *loss_mean, double *dz, double *scratch)
{
    if (vocab <= 0 || !(temperature > 0.0))
        return FQO_ERR_ARG;
    double *a = scratch, *b = scratch + vocab;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t v = 0; v < vocab; v++) {
            a[v] = (double)zt[r * vocab + v] / temperature;
            b[v] = (double)zs[r * vocab + v] / temperature;
        }
        double lse_t = fqo_logsumexp(a, vocab), lse_s = fqo_logsumexp(b, vocab);
        double kl = 0.0;
        for (int64_t v = 0; v < vocab; v++) {
            double log_p = a[v] - lse_t, log_q = b[v] - lse_s;
            double p = exp(log_p), q = exp(log_q);
            kl += p * (log_p - log_q);
            if (dz)
                dz[r * vocab + v] = g * (q - p) / temperature;
        }
        loss_rows[r] = kl;
    }
    double sum = 0.0;
    for (int64_t r = 0; r < rows; r++)
        sum += loss_rows[r];
    *loss_mean = rows ? sum / (double)rows : 0.0;
    return FQO_OK;
}
