// fq_device.cuh -- device-side building blocks of the FP4 fake-quantization
// kernels: E2M1 / E4M3 / E8M0 encode and decode in registers, Philox4x32-10,
// stochastic rounding and the per-block scale derivation.
//
// Definitions follow the library header (include/fq.h): NVFP4 and MXFP4 as
// named on "Aprimorando gpt-oss para Precisão e Desempenho com Treinamento
// Consciente à Quantização" ("O que há de novo"), the double block and
// stochastic rounding of "Resumo Técnico: TetraJet-v2" §2A.  Every operation
// that decides a stored bit has an explicit rounding (round-to-nearest
// intrinsics such as __fdiv_rn and __fmul_rn, or PTX with its rounding mode:
// the packed f32x2 forms, the round-up and round-toward-zero steps of
// stochastic rounding), so no FMA contraction can change one.  The one
// approximate operation, the reciprocal estimate of the scale-code search,
// works inside a guard band: near an E4M3 rounding boundary the code is taken
// from the exact divisions instead.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fq_internal.h"

namespace fqk {

enum Fmt : int { NVFP4 = 0, MXFP4 = 1, NV2L = 2 };
enum Rnd : int { RNE = 0, SR = 1 };

template <int FMT>
struct FmtInfo {
    static constexpr int B = (FMT == MXFP4) ? 32 : 16;  // inner block length
    static constexpr int BO = 128;                      // outer block (double block only)
};

// Elements carried by one 16-byte vector of the input type.
template <typename T>
struct VecInfo;
template <>
struct VecInfo<float> {
    static constexpr int E = 4;
};
template <>
struct VecInfo<__nv_bfloat16> {
    static constexpr int E = 8;
};

// ---------------------------------------------------------------- packed FP32 pairs
// Blackwell's f32x2 forms: one instruction for two lanes, each rounded exactly
// as the scalar operation with the same rounding mode would be.
#define FQK_F32X2_TERNARY(name, op)                                                         \
    __device__ __forceinline__ float2 name(float2 a, float2 b, float2 c)                    \
    {                                                                                       \
        float2 d;                                                                           \
        asm("{\n\t.reg .b64 A, B, C, D;\n\t"                                                \
            "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%6, %7};\n\t" op  \
            " D, A, B, C;\n\tmov.b64 {%0, %1}, D;\n\t}"                                     \
            : "=f"(d.x), "=f"(d.y)                                                          \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));                  \
        return d;                                                                           \
    }
#define FQK_F32X2_BINARY(name, op)                                                          \
    __device__ __forceinline__ float2 name(float2 a, float2 b)                              \
    {                                                                                       \
        float2 d;                                                                           \
        asm("{\n\t.reg .b64 A, B, D;\n\t"                                                   \
            "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t" op                           \
            " D, A, B;\n\tmov.b64 {%0, %1}, D;\n\t}"                                        \
            : "=f"(d.x), "=f"(d.y)                                                          \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                      \
        return d;                                                                           \
    }
FQK_F32X2_TERNARY(fma2, "fma.rn.f32x2")
FQK_F32X2_BINARY(add2, "add.rn.f32x2")
FQK_F32X2_BINARY(sub2, "sub.rn.f32x2")
FQK_F32X2_BINARY(mul2, "mul.rn.f32x2")
#undef FQK_F32X2_TERNARY
#undef FQK_F32X2_BINARY

// ---------------------------------------------------------------- dependent launches
// The quantizers are launched with programmatic stream serialization: their
// launch and CTA set-up may overlap the tail of the kernel before them on the
// stream (from the point where that kernel allows dependent launches, else
// from its end).  Such a kernel calls wait_prior_grid() before any global
// memory access: it returns once every earlier grid on the stream has
// completed and its writes are visible (at once when there is none).  The
// tensor amax pass before the persistent row and tile quantizers does not
// allow an early launch: their grids are sized to be resident at once, and
// CTAs held back by the amax pass's would leave a tail (measured: the NVFP4
// row + column call 123 us with an early launch against 116 us without);
// the masked amax before the split quantizer does (1 us faster).
__device__ __forceinline__ void wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld16(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *v);

template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *v)
{
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
}

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &u, float *v)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// max(|a|, |b|) lane by lane on two BF16 pairs.  The result's sign bits are
// the XOR of the operands' and carry no meaning here: callers mask them off.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Lane-wise largest BF16 magnitude over N packed pairs (N a power of two),
// reduced as a tree.  Exact: the maximum of BF16 magnitudes is one of them.
// The low half of the result holds the low lanes' maximum, the high half the
// high lanes'; read them with bf16_lo / bf16_hi.
template <int N>
__device__ __forceinline__ uint32_t bf16x2_absmax_tree(const uint32_t *w)
{
    uint32_t m[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        m[i] = w[i];
#pragma unroll
    for (int n = N; n > 1; n >>= 1)
#pragma unroll
        for (int i = 0; i < n / 2; ++i)
            m[i] = bf16x2_absmax(m[i], m[i + n / 2]);
    return m[0];
}
__device__ __forceinline__ float bf16_lo_abs(uint32_t m)
{
    return fabsf(__uint_as_float(m << 16));
}
__device__ __forceinline__ float bf16_hi_abs(uint32_t m)
{
    return fabsf(__uint_as_float(m & 0xFFFF0000u));
}

// Amax of one block of B elements of type T held as raw 16-byte vectors.
// BF16 blocks reduce the packed pairs; both forms give max |x| exactly.
template <typename T, int B>
__device__ __forceinline__ float block_amax(const uint4 *raw)
{
    uint32_t w[B * sizeof(T) / 4];
#pragma unroll
    for (int k = 0; k < B * (int)sizeof(T) / 16; ++k) {
        w[4 * k] = raw[k].x;
        w[4 * k + 1] = raw[k].y;
        w[4 * k + 2] = raw[k].z;
        w[4 * k + 3] = raw[k].w;
    }
    if constexpr (sizeof(T) == 2) {
        const uint32_t m = bf16x2_absmax_tree<B / 2>(w);
        return fmaxf(bf16_lo_abs(m), bf16_hi_abs(m));
    } else {
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < B; ++i)
            am = fmaxf(am, fabsf(__uint_as_float(w[i])));
        return am;
    }
}

// ---------------------------------------------------------------- E2M1
// Nearest-even, saturating conversion of 8 floats to 8 packed E2M1 nibbles
// (element 2j in the low nibble of byte j).  The cvt instruction takes its
// first source into the high nibble.
__device__ __forceinline__ uint32_t e2m1_rn_pack8(const float *y)
{
    uint32_t out;
    asm("{\n\t"
        ".reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t"
        "}"
        : "=r"(out)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]),
          "f"(y[7]));
    return out;
}

// E2M1 magnitude of code bits 0..2 as an FP32 bit pattern: 0, 0.5, then
// (1 + m/2) * 2^(e-1) for exponent e >= 1.
__device__ __forceinline__ float e2m1_value(uint32_t code)
{
    const uint32_t mag = code & 7u;
    uint32_t bits = (mag >= 2u) ? ((mag + 252u) << 22) : (mag ? 0x3F000000u : 0u);
    bits |= (code & 8u) << 28;
    return __uint_as_float(bits);
}

// ---------------------------------------------------------------- E4M3
__device__ __forceinline__ uint32_t e4m3_rn_sat(float s)
{
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(s));
    return out & 0xFFu;
}

// Value of a non-negative E4M3 code (never 0x7F here).  Every E4M3 value is
// exact in FP16 (normals (8 + m) 2^(e - 10), subnormals m 2^-9), so the
// hardware E4M3 -> FP16 conversion followed by the exact FP16 -> FP32 widening
// gives it in two conversions.  The code sits in both bytes of the pair, so
// either half of the result holds it.
__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    uint32_t h;
    asm("{\n\t"
        ".reg .b16 c;\n\t"
        "cvt.u16.u32 c, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c;\n\t"
        "}"
        : "=r"(h)
        : "r"(code * 0x101u));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// ---------------------------------------------------------------- block scales
struct Scale {
    float s_eff;  // effective scale of the block
    float r;      // 1 / s_eff (0 for an all-zero block)
    float lim;    // 6 * s_eff: the block's representable range (STE mask)
    uint32_t code;
};

// An approximation of 1 / (6 s_outer) (the hardware reciprocal, within 1 ulp),
// used to find block scale codes without dividing (nv_scale_code).  0 when
// s_outer is 0 or below 2^-120: there 6 s_outer or its reciprocal would leave
// the normal range, and nv_scale_code divides instead.
__device__ __forceinline__ float nv_inv6(float s_outer)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(__fmul_rn(6.0f, s_outer)));
    return (s_outer < 0x1p-120f) ? 0.0f : r;
}

// E4M3 code of the block scale s_b = (amax_b / 6) / s_outer (two IEEE
// divisions, in that order).  With every operand and quotient normal,
// amax_b * inv6 differs from s_b by at most 3 * 2^-23 relative (two roundings
// in s_b; the rounding of 6 s_outer, the reciprocal's 1 ulp and the product's
// rounding in the estimate), i.e. by at most 6 ulps, so both round to the same
// E4M3 code unless the product lies within 64 ulps of an E4M3 rounding
// boundary -- in the E4M3 normal range every boundary has FP32 mantissa bits
// 19..0 equal to 0x80000 -- or below 2^-6, where E4M3 is subnormal.  Those rare blocks take the exact divisions, and so do blocks
// whose amax_b / 6 would be subnormal (amax_b < 2^-123) or whose outer scale
// has no product form (inv6 = 0).
__device__ __forceinline__ uint32_t nv_scale_code(float amax_b, float s_outer, float inv6)
{
    float sb = __fmul_rn(amax_b, inv6);
    const uint32_t low = __float_as_uint(sb) & 0xFFFFFu;
    const bool near = amax_b != 0.0f && ((low - 0x7FFC0u) < 128u || sb < 0.0157f ||
                                         amax_b < 0x1p-123f || inv6 == 0.0f);
    if (near)
        sb = (s_outer == 0.0f) ? 0.0f : __fdiv_rn(__fdiv_rn(amax_b, 6.0f), s_outer);
    return e4m3_rn_sat(sb);
}

// NVFP4-style inner scale under an outer scale s_outer (the tensor scale s_g
// for NVFP4, the 1x128 block scale for the double block).
__device__ __forceinline__ Scale nv_scale(float amax_b, float s_outer, float inv6)
{
    Scale s;
    s.code = nv_scale_code(amax_b, s_outer, inv6);
    s.s_eff = __fmul_rn(e4m3_value(s.code), s_outer);
    s.r = (s.s_eff == 0.0f) ? 0.0f : __frcp_rn(s.s_eff);
    s.lim = __fmul_rn(6.0f, s.s_eff);
    return s;
}

// Per-code tables of one tensor scale s_g (NVFP4): the effective scale, its
// reciprocal and 6 s_eff for each of the 127 finite non-negative E4M3 codes.
// Built once per CTA in shared memory (fill with all threads, then sync).
// One 16-byte entry per code, {s_eff, r, lim, 0}, so that a block reads its
// three values with one shared-memory load.
struct NvTables {
    float4 e[128];
};

__device__ __forceinline__ void nv_tables_fill(NvTables &t, float s_g)
{
    for (int c = threadIdx.x; c < 128; c += blockDim.x) {
        const float se = (c < 0x7F) ? __fmul_rn(e4m3_value(c), s_g) : 0.0f;
        t.e[c] = make_float4(se, (se == 0.0f) ? 0.0f : __frcp_rn(se), __fmul_rn(6.0f, se), 0.0f);
    }
}

__device__ __forceinline__ Scale nv_scale_tab(float amax_b, float s_g, float inv6,
                                              const NvTables &t)
{
    Scale s;
    s.code = nv_scale_code(amax_b, s_g, inv6);
    const float4 e = t.e[s.code];
    s.s_eff = e.x;
    s.r = e.y;
    s.lim = e.z;
    return s;
}

// MXFP4 shared exponent from the FP32 exponent field of the block amax:
// k = floor(log2 amax) - 2, clamped below at -127 (zero and subnormal amax).
__device__ __forceinline__ Scale mx_scale(float amax_b)
{
    Scale s;
    const int ebits = (int)(__float_as_uint(amax_b) >> 23);
    int k = ebits - 129;
    k = k < -127 ? -127 : k;
    s.code = (uint32_t)(k + 127);
    s.s_eff = (k > -127) ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
    s.r = __uint_as_float((uint32_t)(127 - k) << 23);
    s.lim = __fmul_rn(6.0f, s.s_eff);
    return s;
}

// amax_o / 2688 rounded to nearest (IEEE division).  q0 = amax_o * R with
// R = RN(1 / 2688), then one FMA step with the exact residual amax_o - 2688 q0.
// This equals the IEEE quotient for every finite amax_o >= 2^-119 (checked
// exhaustively against division on the host); smaller amax_o, whose quotient
// is subnormal or nearly so, take the division.
__device__ __forceinline__ float outer_scale(float amax_o)
{
    if (amax_o < 0x1p-119f)
        return __fdiv_rn(amax_o, 2688.0f);
    const float R = 0x1.861862p-12f;
    const float q0 = __fmul_rn(amax_o, R);
    return __fmaf_rn(__fmaf_rn(-q0, 2688.0f, amax_o), R, q0);
}

// Effective scale of a stored block (for dequantization).
template <int FMT>
__device__ __forceinline__ float stored_s_eff(uint32_t code, float s_outer)
{
    if (FMT == MXFP4)
        return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
    return __fmul_rn(e4m3_value(code), s_outer);
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): ten rounds; each round multiplies counter words 0 and 2 by the two
// round multipliers, mixes the high halves with words 1 / 3 and the round key
// (PhiloxKey, fq_internal.h).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKey &k)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k.k0[r], (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[r], (uint32_t)p0);
    }
    return c;
}

// Eight 16-bit uniforms for elements 8g .. 8g+7 of a tensor, in element order
// (element j: half j % 2 of word j / 2).
__device__ __forceinline__ uint4 sr_bits8(const PhiloxKey &k, uint64_t g, uint32_t stream,
                                          uint32_t offset)
{
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), stream, offset), k);
}

// ---------------------------------------------------------------- Hadamard transform
// Random Hadamard transform of the backward operands ("Resumo Técnico:
// TetraJet-v2", §2C): z = (1/4) H16 (d . x) on each 16-element block, H16 the
// Sylvester Hadamard matrix as butterflies of strides 1, 2, 4, 8 (one FP32
// addition each), d the signs of bits 0..15 of Philox word 0 at counter
// (0, 0, 2, offset) under key (rht_seed, 0).
__device__ __forceinline__ uint32_t rht_signs(uint32_t rht_seed, uint32_t offset)
{
    const uint4 o = philox4x32_10(make_uint4(0u, 0u, 2u, offset), philox_key(rht_seed));
    return o.x & 0xFFFFu;
}

__device__ __forceinline__ void rht16(float *z, uint32_t signs)
{
    // Strides 1, 2 and 4 on packed pairs (z[i], z[i + 8]), two butterflies per
    // instruction; stride 8 combines the two halves of each pair; then the
    // scaling on pairs (z[2k], z[2k + 1]).  Every element sees the same FP32
    // additions in the same order as the scalar butterflies.
    float2 p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        p[i] = make_float2(
            __uint_as_float(__float_as_uint(z[i]) ^ (((signs >> i) & 1u) << 31)),
            __uint_as_float(__float_as_uint(z[i + 8]) ^ (((signs >> (i + 8)) & 1u) << 31)));
#pragma unroll
    for (int h = 1; h < 8; h *= 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & h)
                continue;
            const float2 a = p[i], b = p[i + h];
            p[i] = add2(a, b);
            p[i + h] = sub2(a, b);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        z[i] = __fadd_rn(p[i].x, p[i].y);
        z[i + 8] = __fsub_rn(p[i].x, p[i].y);
    }
    const float2 quarter = make_float2(0.25f, 0.25f);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float2 q = mul2(make_float2(z[i], z[i + 1]), quarter);
        z[i] = q.x;
        z[i + 1] = q.y;
    }
}

// The stochastic-rounding operand of element j (0..7) of a Philox draw: its
// 16-bit uniform u (half j % 2 of word j / 2) as c = (2^22 - 1 - 64 u) / 2^23,
// exactly (see e2m1_sr_value).  2^23 + u is assembled as an FP32 bit pattern
// by a byte permute, so no integer-to-float conversion is needed.
__device__ __forceinline__ float sr_operand(const uint4 &w, int j)
{
    const uint32_t word = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
    const uint32_t bits = __byte_perm(word, 0x4B000000u, (j & 1) ? 0x7632u : 0x7610u);
    const float u = __fsub_rn(__uint_as_float(bits), 8388608.0f);  // exact
    return __fmaf_rn(u, -7.62939453125e-06f, 0.49999988079071044921875f);  // exact
}

// ---------------------------------------------------------------- misc
template <int L>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = 1; o < L; o <<= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- per-block core
// Dequantize 8 packed E2M1 codes to their grid values (exact in FP16, then
// widened): element 2j comes from the low nibble of byte j.
__device__ __forceinline__ void e2m1_decode8(uint32_t q, float *out)
{
    uint32_t h[4];
    asm("{\n\t"
        ".reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t"
        "}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(q));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[i]));
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// Stochastic rounding of y to the E2M1 grid given a 16-bit uniform u, as an
// FP32 value on the grid (values at or above 6 come out >= 6 and saturate in
// the final conversion).  With lo the grid magnitude at or below a = |y|, g
// the gap above it and F = 65536 (a - lo) / g, the result rounds up iff u < F.
// The work is floating-point, with c = (2^22 - 1 - 64 u) / 2^23 from
// sr_operand, so that 2c = 1 - (u + 2^-6) / 65536:
//  a >= 1: g = 2^(e-1) for a in [2^e, 2^(e+1)), and F is a multiple of 2^-6
//    (a has 23 fraction bits), so u < F iff (a - lo) / g + 2c >= 1.  Hence
//    t = a + 2^e c, rounded toward zero (which never crosses a grid point:
//    they are representable) and cut to one mantissa bit, is lo or lo + g; a
//    sum that crosses into the next binade comes out as its first grid point,
//    2^(e+1) = lo + g.
//  a < 1: g = 1/2, as on [1, 2), so the same is done for z = 1 + a rounded
//    up, and the 1 is subtracted again.  Rounding up moves F only up to the
//    next multiple of 2^-6, which decides u < F the same way for every
//    integer u; a z of 2 rounds up, as then F > 65536 - 2^-6.
// The sign of y is copied (a zero result keeps it).
__device__ __forceinline__ float e2m1_sr_value(float y, float c)
{
    // q = 1 for |y| < 1, else 0, on the FMA pipe: 2^24 (1 - |y|) is at least 1
    // for every FP32 |y| < 1 (the largest is 1 - 2^-24) and at most 0 from 1 on,
    // so clamping it to [0, 1] gives q exactly (a NaN clamps to 0, as a compare
    // would give)
    float q;
    asm("fma.rn.sat.f32 %0, %1, 0fCB800000, 0f4B800000;" : "=f"(q) : "f"(fabsf(y)));
    const float z = __fadd_ru(fabsf(y), q);                              // |y| + 1 or |y|
    const float p = __uint_as_float(__float_as_uint(z) & 0x7F800000u);   // 2^e of z
    const float t = __fmaf_rz(c, p, z);
    const float m = __uint_as_float(__float_as_uint(t) & 0xFFC00000u);   // on the grid
    const float r = __fsub_rn(m, q);                                     // exact
    return __uint_as_float(__float_as_uint(r) | (__float_as_uint(y) & 0x80000000u));
}

// sr_operand for elements 2k and 2k + 1 (both halves of word k).
__device__ __forceinline__ float2 sr_operand2(uint32_t word)
{
    // 2^23 + u as FP32 bits for both halves: the low half by a byte permute,
    // the high half as the high word of word * 2^16 plus 2^23's bits (one
    // integer multiply-add, which runs beside the permutes and logic ops)
    uint32_t hi;
    asm("mad.hi.u32 %0, %1, 65536, 0x4B000000;" : "=r"(hi) : "r"(word));
    const float2 b = make_float2(__uint_as_float(__byte_perm(word, 0x4B000000u, 0x7610u)),
                                 __uint_as_float(hi));
    const float2 u = sub2(b, make_float2(8388608.0f, 8388608.0f));  // exact
    return fma2(u, make_float2(-7.62939453125e-06f, -7.62939453125e-06f),
                make_float2(0.49999988079071044921875f, 0.49999988079071044921875f));
}

// One 32-byte store (st.global.v8.b32): a whole sector per lane, where two
// 16-byte stores from the same lane would each fill half of it in separate
// instructions.  p must be 32-byte aligned.
__device__ __forceinline__ void st32(void *p, const uint4 &a, const uint4 &b)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
                 "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// BF16 fake-quantized values of eight codes (q: one packed word) under the
// effective scale s, as one 16-byte vector: v(code) * s in FP32, then RNE.
__device__ __forceinline__ uint4 xhat8_bf16(uint32_t q, float s)
{
    float h[8];
    e2m1_decode8(q, h);
    const float2 s2 = make_float2(s, s);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 p = mul2(make_float2(h[i], h[i + 1]), s2);
        h[i] = p.x;
        h[i + 1] = p.y;
    }
    return make_uint4(bf16x2_rn(h[0], h[1]), bf16x2_rn(h[2], h[3]), bf16x2_rn(h[4], h[5]),
                      bf16x2_rn(h[6], h[7]));
}

// Encode B values (already loaded as FP32) of one block under scale sc into
// B/8 words of packed codes, and the block's STE mask bits (bit i = element i
// inside [-6 s_eff, 6 s_eff]).  e0 is the flat index of the block's first
// element in the tensor being quantized (Philox counter for SR).
template <int B, int RND>
__device__ __forceinline__ void encode_block(const float *v, const Scale &sc, const PhiloxKey &key,
                                             uint64_t e0, uint32_t stream_id, uint32_t offset,
                                             uint32_t *q)
{
    const float2 r2 = make_float2(sc.r, sc.r);
#pragma unroll
    for (int w = 0; w < B / 8; ++w) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float2 p = mul2(make_float2(v[w * 8 + i], v[w * 8 + i + 1]), r2);
            y[i] = p.x;
            y[i + 1] = p.y;
        }
        if (RND == SR) {
            const uint4 rb = sr_bits8(key, (e0 >> 3) + w, stream_id, offset);
            const uint32_t words[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 c = sr_operand2(words[k]);
                y[2 * k] = e2m1_sr_value(y[2 * k], c.x);
                y[2 * k + 1] = e2m1_sr_value(y[2 * k + 1], c.y);
            }
        }
        q[w] = e2m1_rn_pack8(y);
    }
}

// STE mask bits of a block: bit i = element i inside [-6 s_eff, 6 s_eff].
// The clip bit is the sign of (lim - |x|): exact, since a non-zero difference
// of two floats never rounds to zero without flush-to-zero.  A funnel shift
// moves each sign bit into the accumulator, last element first, so bit i ends
// at position i: one instruction per element besides the subtraction.
template <int B>
__device__ __forceinline__ uint32_t block_mask(const float *v, float lim)
{
    uint32_t clip = 0;
#pragma unroll
    for (int i = B - 1; i >= 0; --i)
        clip = __funnelshift_l(__float_as_uint(__fsub_rn(lim, fabsf(v[i]))), clip, 1);
    return (B == 32) ? ~clip : (~clip & ((1u << B) - 1u));
}

// Block scale for one block.  NVFP4 reads the per-code tables of its tensor
// scale; the double block derives its scale from the outer scale s_o.
template <int FMT>
__device__ __forceinline__ Scale block_scale(float amax_b, float s_outer, float inv6,
                                             const NvTables *tab)
{
    if (FMT == MXFP4)
        return mx_scale(amax_b);
    if (FMT == NVFP4)
        return nv_scale_tab(amax_b, s_outer, inv6, *tab);
    return nv_scale(amax_b, s_outer, inv6);
}

template <typename T, int N>
__device__ __forceinline__ void load_block(const void *src, float *v)
{
    constexpr int E = VecInfo<T>::E;
#pragma unroll
    for (int k = 0; k < N / E; ++k)
        unpack16<T>(ld16((const char *)src + 16 * k), v + k * E);
}

// One 32-byte load (ld.global.nc.v8.b32): a whole sector per lane, where two
// 16-byte loads from the same lane each take half of it.  p must be 32-byte
// aligned.
__device__ __forceinline__ void ld32(const void *p, uint4 &a, uint4 &b)
{
    asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
        : "l"(p));
}

// NV consecutive 16-byte vectors from src, 32 bytes per load when al32 (src
// 32-byte aligned; NV even).
template <int NV>
__device__ __forceinline__ void load_vecs(const char *src, uint4 *raw, bool al32)
{
    if (NV % 2 == 0 && al32) {
#pragma unroll
        for (int k = 0; k < NV; k += 2)
            ld32(src + 16 * k, raw[k], raw[k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < NV; ++k)
            raw[k] = ld16(src + 16 * k);
    }
}

}  // namespace fqk

