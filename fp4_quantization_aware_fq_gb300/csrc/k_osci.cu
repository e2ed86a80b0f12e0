// k_osci.cu -- OsciReset statistics and reset ("Resumo Técnico: TetraJet-v2"
// §2B): the oscillation risk of a weight is the distance its quantized value
// travelled (dist_Q) over the distance its master value travelled (dist_M);
// weights whose risk exceeds a threshold are moved to the quantized value of
// their current bin.
//
// One optimizer step is two passes over a group of tensors (e.g. all expert
// matrices of an MoE layer), each a persistent grid walking 16-byte chunks of
// FP32 master weights tile by tile across the whole group:
//   A: w += delta, dist_M += |w_t - w_{t-1}|, per-tensor amax of w_t (atomic);
//   B: fake-quantize w_t under the new tensor scale, decode w_{t-1}'s stored
//      codes, dist_Q += |xhat_t - xhat_{t-1}|, write codes/scales/xhat/mask.
// The tensor amax is the only dependency between the passes, hence the split.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kOsciThreads = 256;
constexpr int kOsciU = 4;

__device__ __forceinline__ float4 ldf4(const float *p)
{
    return __ldg(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ float4 ldf4_rw(const float *p)
{
    return *reinterpret_cast<const float4 *>(p);
}

__device__ __forceinline__ void stf4(float *p, float4 v)
{
    *reinterpret_cast<float4 *>(p) = v;
}

__global__ void __launch_bounds__(kOsciThreads) osci_pass_a(const __grid_constant__ OsciArgs a)
{
    const int64_t ntiles = a.tile_start[a.ntensors];
    int t = 0;
    __shared__ float wm[kOsciThreads / 32];
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        while (a.tile_start[t + 1] <= tile)
            ++t;
        const OsciTensor &T = a.t[t];
        const int64_t nch = T.n / 4;
        const int64_t cbeg = (tile - a.tile_start[t]) * kOsciTileChunks;
        float m = 0.0f;
        for (int k0 = 0; k0 < kOsciTileChunks; k0 += kOsciThreads * kOsciU) {
            float4 w[kOsciU], d[kOsciU], dm[kOsciU];
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch < nch) {
                    w[k] = ldf4_rw(T.master + ch * 4);
                    d[k] = ldf4(T.delta + ch * 4);
                    dm[k] = ldf4_rw(T.dist_m + ch * 4);
                }
            }
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch < nch) {
                    float4 wn;
                    wn.x = __fadd_rn(w[k].x, d[k].x);
                    wn.y = __fadd_rn(w[k].y, d[k].y);
                    wn.z = __fadd_rn(w[k].z, d[k].z);
                    wn.w = __fadd_rn(w[k].w, d[k].w);
                    float4 dn;
                    dn.x = __fadd_rn(dm[k].x, fabsf(__fsub_rn(wn.x, w[k].x)));
                    dn.y = __fadd_rn(dm[k].y, fabsf(__fsub_rn(wn.y, w[k].y)));
                    dn.z = __fadd_rn(dm[k].z, fabsf(__fsub_rn(wn.z, w[k].z)));
                    dn.w = __fadd_rn(dm[k].w, fabsf(__fsub_rn(wn.w, w[k].w)));
                    stf4(T.master + ch * 4, wn);
                    stf4(T.dist_m + ch * 4, dn);
                    m = fmaxf(m, fmaxf(fmaxf(fabsf(wn.x), fabsf(wn.y)),
                                       fmaxf(fabsf(wn.z), fabsf(wn.w))));
                }
            }
        }
        m = group_max<32>(m);
        if ((threadIdx.x & 31) == 0)
            wm[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float b = wm[0];
#pragma unroll
            for (int i = 1; i < kOsciThreads / 32; ++i)
                b = fmaxf(b, wm[i]);
            atomicMax(reinterpret_cast<unsigned *>(a.amax) + t, __float_as_uint(b));
        }
        __syncthreads();
    }
}

template <int FMT, int RND>
__global__ void __launch_bounds__(kOsciThreads) osci_pass_b(const __grid_constant__ OsciArgs a)
{
    constexpr int E = 4;
    constexpr int L = FmtInfo<FMT>::B / E;
    constexpr int LO = 128 / E;
    const int64_t ntiles = a.tile_start[a.ntensors];
    int t = 0;
    const int lane = threadIdx.x & 31;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        while (a.tile_start[t + 1] <= tile)
            ++t;
        const OsciTensor &T = a.t[t];
        const int64_t nch = T.n / 4;
        const int64_t cbeg = (tile - a.tile_start[t]) * kOsciTileChunks;
        float s_g = 0.0f, s_gp = 0.0f;
        if (FMT == NVFP4) {
            s_g = outer_scale(__ldg(a.amax + t));
            s_gp = __ldg(T.ptscale);
            if (cbeg == 0 && threadIdx.x == 0)
                T.ntscale[0] = s_g;
        }
        for (int k0 = 0; k0 < kOsciTileChunks; k0 += kOsciThreads * kOsciU) {
            uint4 raw[kOsciU];
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                raw[k] = ch < nch ? *reinterpret_cast<const uint4 *>(T.master + ch * 4)
                                  : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                const bool valid = ch < nch;
                const VecQ<E> r = quant_vec<float, FMT, RND>(raw[k], ch, s_g, a.seed, a.offset, 0u);
                const uint32_t mpair = __shfl_down_sync(0xFFFFFFFFu, r.mbits, 1);
                if (!valid)
                    continue;
                // previous quantized value of these 4 weights
                const uint32_t qp = __ldg(reinterpret_cast<const uint16_t *>(T.pcodes) + ch);
                const uint32_t scp = __ldg(T.pscales + ch / L);
                float so_p = s_gp;
                if (FMT == NV2L)
                    so_p = __ldg(T.ptscale + ch / LO);
                const float seff_p = stored_s_eff<FMT>(scp, so_p);
                float xh[E], xp[E];
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    xh[i] = __fmul_rn(e2m1_value(r.q >> (4 * i)), r.sc.s_eff);
                    xp[i] = __fmul_rn(e2m1_value(qp >> (4 * i)), seff_p);
                }
                float4 dq = ldf4_rw(T.dist_q + ch * 4);
                dq.x = __fadd_rn(dq.x, fabsf(__fsub_rn(xh[0], xp[0])));
                dq.y = __fadd_rn(dq.y, fabsf(__fsub_rn(xh[1], xp[1])));
                dq.z = __fadd_rn(dq.z, fabsf(__fsub_rn(xh[2], xp[2])));
                dq.w = __fadd_rn(dq.w, fabsf(__fsub_rn(xh[3], xp[3])));
                stf4(T.dist_q + ch * 4, dq);
                reinterpret_cast<uint16_t *>(T.ncodes)[ch] = (uint16_t)r.q;
                if ((lane % L) == 0)
                    T.nscales[ch / L] = (uint8_t)r.sc.code;
                if (FMT == NV2L && (lane % LO) == 0)
                    T.ntscale[ch / LO] = r.s_o;
                if (T.xhat) {
                    if (a.xhat_bf16)
                        reinterpret_cast<uint2 *>(T.xhat)[ch] =
                            make_uint2(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]));
                    else
                        reinterpret_cast<float4 *>(T.xhat)[ch] = make_float4(xh[0], xh[1], xh[2], xh[3]);
                }
                if (T.mask && (lane & 1) == 0)
                    T.mask[ch >> 1] = (uint8_t)(r.mbits | (mpair << 4));
            }
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kOsciThreads) osci_reset_kernel(const __grid_constant__ OsciArgs a)
{
    constexpr int L = FmtInfo<FMT>::B / 4;
    constexpr int LO = 128 / 4;
    const int64_t ntiles = a.tile_start[a.ntensors];
    int t = 0;
    unsigned long long cnt = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        while (a.tile_start[t + 1] <= tile)
            ++t;
        const OsciTensor &T = a.t[t];
        const int64_t nch = T.n / 4;
        const int64_t cbeg = (tile - a.tile_start[t]) * kOsciTileChunks;
        float s_g = 0.0f;
        if (FMT == NVFP4)
            s_g = __ldg(T.ptscale);
        for (int k = 0; k < kOsciTileChunks; k += kOsciThreads) {
            const int64_t ch = cbeg + k + threadIdx.x;
            if (ch >= nch)
                continue;
            const float4 dq = ldf4_rw(T.dist_q + ch * 4);
            const float4 dm = ldf4_rw(T.dist_m + ch * 4);
            const float q4[4] = {dq.x, dq.y, dq.z, dq.w};
            const float m4[4] = {dm.x, dm.y, dm.z, dm.w};
            uint32_t hit = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                hit |= (q4[i] > __fmul_rn(a.threshold, m4[i]) ? 1u : 0u) << i;
            if (hit) {
                const uint32_t q = __ldg(reinterpret_cast<const uint16_t *>(T.pcodes) + ch);
                const uint32_t sc = __ldg(T.pscales + ch / L);
                float so = s_g;
                if (FMT == NV2L)
                    so = __ldg(T.ptscale + ch / LO);
                const float s_eff = stored_s_eff<FMT>(sc, so);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((hit >> i) & 1u)
                        T.master[ch * 4 + i] = __fmul_rn(e2m1_value(q >> (4 * i)), s_eff);
                cnt += __popc(hit);
            }
            stf4(T.dist_q + ch * 4, make_float4(0.f, 0.f, 0.f, 0.f));
            stf4(T.dist_m + ch * 4, make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    if (a.n_reset) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
        if ((threadIdx.x & 31) == 0 && cnt)
            atomicAdd(a.n_reset, cnt);
    }
}

static int osci_grid(int64_t ntiles)
{
    const int64_t cap = (int64_t)sm_count() * 4;
    return (int)(ntiles < cap ? (ntiles > 0 ? ntiles : 1) : cap);
}

cudaError_t launch_osci_update(const OsciArgs &a, int fmt, int rnd, cudaStream_t s)
{
    const int64_t ntiles = a.tile_start[a.ntensors];
    cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(float) * (size_t)a.ntensors, s);
    if (e != cudaSuccess || ntiles == 0)
        return e;
    const int grid = osci_grid(ntiles);
    osci_pass_a<<<grid, kOsciThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    switch (fmt * 2 + rnd) {
    case NVFP4 * 2 + RNE: osci_pass_b<NVFP4, RNE><<<grid, kOsciThreads, 0, s>>>(a); break;
    case NVFP4 * 2 + SR: osci_pass_b<NVFP4, SR><<<grid, kOsciThreads, 0, s>>>(a); break;
    case MXFP4 * 2 + RNE: osci_pass_b<MXFP4, RNE><<<grid, kOsciThreads, 0, s>>>(a); break;
    case MXFP4 * 2 + SR: osci_pass_b<MXFP4, SR><<<grid, kOsciThreads, 0, s>>>(a); break;
    case NV2L * 2 + RNE: osci_pass_b<NV2L, RNE><<<grid, kOsciThreads, 0, s>>>(a); break;
    default: osci_pass_b<NV2L, SR><<<grid, kOsciThreads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_osci_reset(const OsciArgs &a, int fmt, cudaStream_t s)
{
    const int64_t ntiles = a.tile_start[a.ntensors];
    if (ntiles == 0)
        return cudaSuccess;
    const int grid = osci_grid(ntiles);
    if (fmt == NVFP4)
        osci_reset_kernel<NVFP4><<<grid, kOsciThreads, 0, s>>>(a);
    else if (fmt == MXFP4)
        osci_reset_kernel<MXFP4><<<grid, kOsciThreads, 0, s>>>(a);
    else
        osci_reset_kernel<NV2L><<<grid, kOsciThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace fqk
