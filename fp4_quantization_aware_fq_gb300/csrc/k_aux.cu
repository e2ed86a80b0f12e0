// k_aux.cu -- dequantization and the straight-through-estimator backward.
//
// Dequantization is the "dequantize" half of the quantize/dequantize operator
// of fake quantization ("Como o Treinamento com Quantização Detecta e Recupera
// Precisão em Inferência de Baixa Precisão", "Detalhes técnicos"); the STE
// backward lets the gradient through where the element was inside the
// block's representable range and zeroes it where it was clipped.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kAuxThreads = 256;

// One thread = 8 consecutive elements (4 code bytes).  STRIDED: the rows of y
// lie a.ldy elements apart (cols is a multiple of 8, so a group never spans
// two rows).
template <int FMT, bool STRIDED>
__global__ void __launch_bounds__(kAuxThreads) dequant_kernel(DequantArgs a)
{
    constexpr int B = FmtInfo<FMT>::B;
    const int64_t ng = a.n / 8;
    const int64_t stride = (int64_t)gridDim.x * kAuxThreads;
    // FP32 output in 32-byte stores when every group of 8 starts on a 32-byte
    // boundary (y aligned, and so is its row pitch)
    const bool y32 = ((reinterpret_cast<uintptr_t>(a.y) | (uintptr_t)(a.ldy * 4)) & 31u) == 0;
    for (int64_t g = (int64_t)blockIdx.x * kAuxThreads + threadIdx.x; g < ng; g += stride) {
        const uint32_t q = __ldg(reinterpret_cast<const uint32_t *>(a.codes) + g);
        const int64_t e0 = g * 8;
        const uint32_t sc = __ldg(a.scales + e0 / B);
        float s_outer = 0.0f;
        if (FMT == NVFP4)
            s_outer = __ldg(a.tscale);
        else if (FMT == NV2L)
            s_outer = __ldg(a.tscale + e0 / 128);
        const float s_eff = stored_s_eff<FMT>(sc, s_outer);
        float xh[8];
        e2m1_decode8(q, xh);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xh[i] = __fmul_rn(xh[i], s_eff);
        int64_t oe = e0;  // element offset of the group in y
        if constexpr (STRIDED) {
            const int64_t r = e0 / a.cols;
            oe = r * a.ldy + (e0 - r * a.cols);
        }
        if (a.y_bf16) {
            uint4 o = make_uint4(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]),
                                 bf16x2_rn(xh[4], xh[5]), bf16x2_rn(xh[6], xh[7]));
            *reinterpret_cast<uint4 *>((char *)a.y + oe * 2) = o;
        } else if (y32) {  // whole 32-byte sectors
            st32((char *)a.y + oe * 4,
                 make_uint4(__float_as_uint(xh[0]), __float_as_uint(xh[1]), __float_as_uint(xh[2]),
                            __float_as_uint(xh[3])),
                 make_uint4(__float_as_uint(xh[4]), __float_as_uint(xh[5]), __float_as_uint(xh[6]),
                            __float_as_uint(xh[7])));
        } else {
            float4 *dst = reinterpret_cast<float4 *>((char *)a.y + oe * 4);
            dst[0] = make_float4(xh[0], xh[1], xh[2], xh[3]);
            dst[1] = make_float4(xh[4], xh[5], xh[6], xh[7]);
        }
    }
}

// Each thread takes kSteU 16-byte vectors of dy per step (kAuxThreads apart,
// so every load is coalesced across the warp), all loads issued before any
// is used: four vectors in flight per thread keep about 32 KB of loads in
// flight per CTA.
constexpr int kSteU = 4;
template <typename T>
__global__ void __launch_bounds__(kAuxThreads) ste_kernel(const void *__restrict__ dy,
                                                          const uint8_t *__restrict__ mask,
                                                          int64_t nch, void *__restrict__ dx)
{
    constexpr int E = VecInfo<T>::E;
    const int64_t stride = (int64_t)gridDim.x * kAuxThreads * kSteU;
    for (int64_t base = (int64_t)blockIdx.x * kAuxThreads * kSteU; base < nch; base += stride) {
        uint4 v[kSteU];
        uint32_t m[kSteU];
#pragma unroll
        for (int k = 0; k < kSteU; ++k) {
            const int64_t ch = base + k * kAuxThreads + threadIdx.x;
            if (ch < nch) {
                v[k] = ld16((const char *)dy + ch * 16);
                m[k] = __ldg(mask + (ch * E) / 8);
            }
        }
#pragma unroll
        for (int k = 0; k < kSteU; ++k) {
            const int64_t ch = base + k * kAuxThreads + threadIdx.x;
            if (ch >= nch)
                continue;
            uint32_t mk = m[k];
            if (E == 4)
                mk >>= (ch & 1) * 4;
            uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            if (E == 8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t keep = ((mk >> (2 * i)) & 1u ? 0x0000FFFFu : 0u) |
                                          ((mk >> (2 * i + 1)) & 1u ? 0xFFFF0000u : 0u);
                    w[i] &= keep;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[i] = ((mk >> i) & 1u) ? w[i] : 0u;
            }
            reinterpret_cast<uint4 *>(dx)[ch] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

static int grid_for(int64_t items, int ctas_per_sm)
{
    const int64_t need = (items + kAuxThreads - 1) / kAuxThreads;
    const int64_t cap = (int64_t)sm_count() * ctas_per_sm;
    return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

cudaError_t launch_dequant(const DequantArgs &a, int fmt, cudaStream_t s)
{
    if (a.n == 0)
        return cudaSuccess;
    const int grid = grid_for(a.n / 8, 8);
    const bool st = a.ldy != a.cols;
    if (fmt == NVFP4)
        st ? dequant_kernel<NVFP4, true><<<grid, kAuxThreads, 0, s>>>(a)
           : dequant_kernel<NVFP4, false><<<grid, kAuxThreads, 0, s>>>(a);
    else if (fmt == MXFP4)
        st ? dequant_kernel<MXFP4, true><<<grid, kAuxThreads, 0, s>>>(a)
           : dequant_kernel<MXFP4, false><<<grid, kAuxThreads, 0, s>>>(a);
    else
        st ? dequant_kernel<NV2L, true><<<grid, kAuxThreads, 0, s>>>(a)
           : dequant_kernel<NV2L, false><<<grid, kAuxThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ste(const void *dy, int bf16, const uint8_t *mask, int64_t n, void *dx,
                       cudaStream_t s)
{
    if (n == 0)
        return cudaSuccess;
    const int64_t nch = n / (bf16 ? 8 : 4);
    // a grid-stride walk by 32 CTAs per SM, the later ones starting as the
    // first finish (BF16 [8192, 8192] in the step: 45.5 us against 47.2 with
    // 4 per SM and 47.5 with 8; 16 to 64 measure the same)
    const int grid = grid_for((nch + kSteU - 1) / kSteU, 32);
    if (bf16)
        ste_kernel<__nv_bfloat16><<<grid, kAuxThreads, 0, s>>>(dy, mask, nch, dx);
    else
        ste_kernel<float><<<grid, kAuxThreads, 0, s>>>(dy, mask, nch, dx);
    return cudaGetLastError();
}

}  // namespace fqk
