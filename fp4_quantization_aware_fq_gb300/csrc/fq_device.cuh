// fq_device.cuh -- device-side building blocks of the FP4 fake-quantization
// kernels: E2M1 / E4M3 / E8M0 encode and decode in registers, Philox4x32-10,
// stochastic rounding and the per-block scale derivation.
//
// Definitions follow the library header (include/fq.h): NVFP4 and MXFP4 as
// named on "Aprimorando gpt-oss para Precisão e Desempenho com Treinamento
// Consciente à Quantização" ("O que há de novo"), the double block and
// stochastic rounding of "Resumo Técnico: TetraJet-v2" §2A.  All scale and
// product arithmetic uses explicit round-to-nearest intrinsics (__fdiv_rn,
// __fmul_rn, __frcp_rn) so that no FMA contraction or approximate division
// can change a stored bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

__device__ __forceinline__ uint32_t e2m1_rn_pack4(const float *y)
{
    uint32_t out;
    asm("{\n\t"
        ".reg .b8 q0, q1;\n\t"
        ".reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "mov.b16 h, {q0, q1};\n\t"
        "cvt.u32.u16 %0, h;\n\t"
        "}"
        : "=r"(out)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]));
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

// Stochastic rounding of one value given a 16-bit uniform u: with lo the
// largest grid magnitude <= |y|, round up iff u < frac * 65536.  In each
// binade of the grid the scaled value z = |y| * {2, 1, 1/2} has unit spacing,
// so lo and frac come from floor(z) exactly.
__device__ __forceinline__ uint32_t e2m1_sr(float y, uint32_t u)
{
    const uint32_t sign = (__float_as_uint(y) >> 28) & 8u;
    const float a = fabsf(y);
    if (!(a < 6.0f))
        return sign | 7u;
    const bool lo2 = a < 2.0f, lo4 = a < 4.0f;
    const float s = lo2 ? 2.0f : (lo4 ? 1.0f : 0.5f);
    const uint32_t base = lo2 ? 0u : (lo4 ? 2u : 4u);
    const float z = __fmul_rn(a, s);
    const float f = floorf(z);
    const float t = __fmul_rn(__fsub_rn(z, f), 65536.0f);
    const uint32_t up = (__uint2float_rn(u) < t) ? 1u : 0u;
    return sign | (base + (uint32_t)f + up);
}

// ---------------------------------------------------------------- E4M3
__device__ __forceinline__ uint32_t e4m3_rn_sat(float s)
{
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(s));
    return out & 0xFFu;
}

// Value of a non-negative E4M3 code (never 0x7F here): subnormal m * 2^-9,
// normal (8 + m) * 2^(e - 10).
__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    const uint32_t e = (code >> 3) & 15u, m = code & 7u;
    const uint32_t mant = e ? (8u | m) : m;
    const uint32_t ee = e ? e : 1u;
    // 2^(ee - 10) as an FP32 bit pattern: ee - 10 ranges over [-9, 5]
    const float p2 = __uint_as_float((ee - 10u + 127u) << 23);
    return __fmul_rn(__uint2float_rn(mant), p2);
}

// ---------------------------------------------------------------- block scales
struct Scale {
    float s_eff;  // effective scale of the block
    float r;      // 1 / s_eff (0 for an all-zero block)
    float lim;    // 6 * s_eff: the block's representable range (STE mask)
    uint32_t code;
};

// NVFP4-style inner scale under an outer scale s_outer (the tensor scale s_g
// for NVFP4, the 1x128 block scale for the double block).
__device__ __forceinline__ Scale nv_scale(float amax_b, float s_outer)
{
    Scale s;
    const float sb = (s_outer == 0.0f) ? 0.0f : __fdiv_rn(__fdiv_rn(amax_b, 6.0f), s_outer);
    s.code = e4m3_rn_sat(sb);
    s.s_eff = __fmul_rn(e4m3_value(s.code), s_outer);
    s.r = (s.s_eff == 0.0f) ? 0.0f : __frcp_rn(s.s_eff);
    s.lim = __fmul_rn(6.0f, s.s_eff);
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

__device__ __forceinline__ float outer_scale(float amax_o)
{
    return __fdiv_rn(amax_o, 2688.0f);
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
// round multipliers, mixes the high halves with words 1 / 3 and the key, and
// the key is bumped by the two Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c.x;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Eight 16-bit uniforms for elements 8g .. 8g+7 of a tensor, in element order
// (element j: half j % 2 of word j / 2).
__device__ __forceinline__ uint4 sr_bits8(uint64_t seed, uint64_t g, uint32_t stream,
                                          uint32_t offset)
{
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), stream, offset),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t u16_of(const uint4 &w, int j)
{
    const uint32_t word = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
    return (j & 1) ? (word >> 16) : (word & 0xFFFFu);
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

// ---------------------------------------------------------------- per-vector core
// Result of quantizing one 16-byte input vector (E values) of a row-wise block.
template <int E>
struct VecQ {
    float v[E];       // the input values (FP32)
    uint32_t q;       // packed codes, element i in nibble i
    uint32_t mbits;   // STE mask bits, element i in bit i
    Scale sc;         // inner block scale
    float s_o;        // outer scale (double block only)
};

// Quantize the vector `raw` whose flat vector index in the tensor is `ch`
// (flat element index ch * E).  All 32 lanes of the warp must call this
// together: the block amax is combined with shuffles over the lanes that hold
// the block.  s_g is the NVFP4 tensor scale (unused for the other formats).
template <typename T, int FMT, int RND>
__device__ __forceinline__ VecQ<VecInfo<T>::E> quant_vec(const uint4 &raw, int64_t ch, float s_g,
                                                        uint64_t seed, uint32_t offset,
                                                        uint32_t stream_id)
{
    constexpr int E = VecInfo<T>::E;
    constexpr int L = FmtInfo<FMT>::B / E;  // lanes per inner block
    constexpr int LO = 128 / E;             // lanes per outer block (double block)
    VecQ<E> r;
    unpack16<T>(raw, r.v);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < E; ++i)
        am = fmaxf(am, fabsf(r.v[i]));
    const float amb = group_max<L>(am);
    r.s_o = 0.0f;
    if (FMT == MXFP4) {
        r.sc = mx_scale(amb);
    } else if (FMT == NVFP4) {
        r.sc = nv_scale(amb, s_g);
    } else {
        r.s_o = outer_scale(group_max<LO>(amb));
        r.sc = nv_scale(amb, r.s_o);
    }
    float y[E];
    r.mbits = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        y[i] = __fmul_rn(r.v[i], r.sc.r);
        r.mbits |= (fabsf(r.v[i]) <= r.sc.lim ? 1u : 0u) << i;
    }
    if (RND == RNE) {
        r.q = (E == 8) ? e2m1_rn_pack8(y) : e2m1_rn_pack4(y);
    } else {
        const int64_t e0 = ch * E;
        const uint4 rb = sr_bits8(seed, (uint64_t)e0 >> 3, stream_id, offset);
        uint32_t q = 0;
        if (E == 8) {
#pragma unroll
            for (int i = 0; i < E; ++i)
                q |= e2m1_sr(y[i], u16_of(rb, i)) << (4 * i);
        } else {
            const bool hi = (e0 & 7) != 0;
            const uint4 h = hi ? make_uint4(rb.z, rb.w, 0, 0) : make_uint4(rb.x, rb.y, 0, 0);
#pragma unroll
            for (int i = 0; i < E; ++i)
                q |= e2m1_sr(y[i], u16_of(h, i)) << (4 * i);
        }
        r.q = q;
    }
    return r;
}

}  // namespace fqk
