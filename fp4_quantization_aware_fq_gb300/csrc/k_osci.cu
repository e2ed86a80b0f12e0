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

// Pass B: one thread per block of 16 (32 for MXFP4) master weights, NB blocks
// per thread per iteration with all their loads issued before any compute.
// With RESET, this step also ends the OsciReset window: where the new
// dist_Q exceeds threshold * dist_M, the master weight becomes xhat_t, and
// both accumulators are written back as zero (the same bits as the separate
// reset pass after this update).
template <int FMT, int RND, bool RESET>
__global__ void __launch_bounds__(kOsciThreads) osci_pass_b(const __grid_constant__ OsciArgs a)
{
    constexpr int B = FmtInfo<FMT>::B;
    constexpr int BPTILE = kOsciTileChunks * 4 / B;  // blocks per tile
    // two blocks in flight per thread, one when dist_M is read as well
    constexpr int NB = (!RESET && BPTILE >= 2 * kOsciThreads) ? 2 : 1;
    static_assert(BPTILE % (NB * kOsciThreads) == 0, "tile must split evenly");
    __shared__ NvTables tab, tabp;  // NVFP4: this step's and the previous step's tensor scale
    const int64_t ntiles = a.tile_start[a.ntensors];
    const PhiloxKey key = philox_key(a.seed);
    int t = 0, t_tab = -1;
    const int lane = threadIdx.x & 31;
    unsigned long long cnt = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        while (a.tile_start[t + 1] <= tile)
            ++t;
        const OsciTensor &T = a.t[t];
        const int64_t nblk = T.n / B;
        const int64_t bbeg = (tile - a.tile_start[t]) * BPTILE;
        float s_g = 0.0f, inv6 = 0.0f;
        if (FMT == NVFP4) {
            s_g = outer_scale(__ldg(a.amax + t));
            inv6 = nv_inv6(s_g);
            if (t != t_tab) {  // uniform across the CTA: rebuild the tables
                __syncthreads();
                nv_tables_fill(tab, s_g);
                nv_tables_fill(tabp, __ldg(T.ptscale));
                __syncthreads();
                t_tab = t;
            }
            if (bbeg == 0 && threadIdx.x == 0)
                T.ntscale[0] = s_g;
        }
        for (int k = 0; k < BPTILE; k += NB * kOsciThreads) {
            float v[NB][B], dq[NB][B], dm[NB][B];
            uint32_t qp[NB][B / 8];
            uint32_t scp[NB];
            float so_p[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int64_t blk = bbeg + k + j * kOsciThreads + threadIdx.x;
                if (blk < nblk) {
#pragma unroll
                    for (int i = 0; i < B / 4; ++i) {
                        const float4 w = ldf4_rw(T.master + blk * B + 4 * i);
                        v[j][4 * i] = w.x;
                        v[j][4 * i + 1] = w.y;
                        v[j][4 * i + 2] = w.z;
                        v[j][4 * i + 3] = w.w;
                        const float4 d = ldf4_rw(T.dist_q + blk * B + 4 * i);
                        dq[j][4 * i] = d.x;
                        dq[j][4 * i + 1] = d.y;
                        dq[j][4 * i + 2] = d.z;
                        dq[j][4 * i + 3] = d.w;
                        if (RESET) {
                            const float4 e = ldf4_rw(T.dist_m + blk * B + 4 * i);
                            dm[j][4 * i] = e.x;
                            dm[j][4 * i + 1] = e.y;
                            dm[j][4 * i + 2] = e.z;
                            dm[j][4 * i + 3] = e.w;
                        }
                    }
                    if (B == 16) {
                        const uint2 p2 = __ldg(reinterpret_cast<const uint2 *>(T.pcodes) + blk);
                        qp[j][0] = p2.x;
                        qp[j][1] = p2.y;
                    } else {
                        const uint4 p4 = __ldg(reinterpret_cast<const uint4 *>(T.pcodes) + blk);
                        qp[j][0] = p4.x;
                        qp[j][1] = p4.y;
                        qp[j][2] = p4.z;
                        qp[j][3] = p4.w;
                    }
                    scp[j] = __ldg(T.pscales + blk);
                    so_p[j] = (FMT == NV2L) ? __ldg(T.ptscale + (blk >> 3)) : 0.0f;
                } else {
#pragma unroll
                    for (int i = 0; i < B; ++i)
                        v[j][i] = dq[j][i] = dm[j][i] = 0.0f;
#pragma unroll
                    for (int w = 0; w < B / 8; ++w)
                        qp[j][w] = 0;
                    scp[j] = 0;
                    so_p[j] = 0.0f;
                }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int64_t blk = bbeg + k + j * kOsciThreads + threadIdx.x;
                const bool valid = blk < nblk;
                float am = 0.0f;
#pragma unroll
                for (int i = 0; i < B; ++i)
                    am = fmaxf(am, fabsf(v[j][i]));
                float s_o = s_g, inv6b = inv6;
                if (FMT == NV2L) {
                    s_o = outer_scale(group_max<8>(am));
                    inv6b = nv_inv6(s_o);
                }
                const Scale sc = block_scale<FMT>(am, s_o, inv6b, &tab);
                uint32_t q[B / 8];
                encode_block<B, RND>(v[j], sc, key, (uint64_t)blk * B, 0u, a.offset, q);
                if (!valid)
                    continue;
                const float seff_p = (FMT == NVFP4) ? tabp.s_eff[scp[j] & 127u]
                                                    : stored_s_eff<FMT>(scp[j], so_p[j]);
                uint32_t hit = 0;
#pragma unroll
                for (int w = 0; w < B / 8; ++w) {
                    float xh[8], xp[8];
                    e2m1_decode8(q[w], xh);
                    e2m1_decode8(qp[j][w], xp);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xh[i] = __fmul_rn(xh[i], sc.s_eff);
                        xp[i] = __fmul_rn(xp[i], seff_p);
                        const float dn =
                            __fadd_rn(dq[j][w * 8 + i], fabsf(__fsub_rn(xh[i], xp[i])));
                        if (RESET) {
                            const int e = w * 8 + i;
                            if (dn > __fmul_rn(a.threshold, dm[j][e])) {
                                T.master[blk * B + e] = xh[i];
                                hit |= 1u << e;
                            }
                            dq[j][e] = 0.0f;
                        } else {
                            dq[j][w * 8 + i] = dn;
                        }
                    }
                    if (T.xhat) {
                        if (a.xhat_bf16) {
                            *reinterpret_cast<uint4 *>((char *)T.xhat + (blk * B + w * 8) * 2) =
                                make_uint4(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]),
                                           bf16x2_rn(xh[4], xh[5]), bf16x2_rn(xh[6], xh[7]));
                        } else {
                            float *xo = reinterpret_cast<float *>(T.xhat) + blk * B + w * 8;
                            stf4(xo, make_float4(xh[0], xh[1], xh[2], xh[3]));
                            stf4(xo + 4, make_float4(xh[4], xh[5], xh[6], xh[7]));
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < B / 4; ++i) {
                    stf4(T.dist_q + blk * B + 4 * i,
                         make_float4(dq[j][4 * i], dq[j][4 * i + 1], dq[j][4 * i + 2],
                                     dq[j][4 * i + 3]));
                    if (RESET)
                        stf4(T.dist_m + blk * B + 4 * i, make_float4(0.f, 0.f, 0.f, 0.f));
                }
                cnt += __popc(hit);
                if (B == 16)
                    reinterpret_cast<uint2 *>(T.ncodes)[blk] = make_uint2(q[0], q[1]);
                else
                    reinterpret_cast<uint4 *>(T.ncodes)[blk] = make_uint4(q[0], q[1], q[2], q[3]);
                T.nscales[blk] = (uint8_t)sc.code;
                if (FMT == NV2L && (lane & 7) == 0)
                    T.ntscale[blk >> 3] = s_o;
                if (T.mask) {
                    const uint32_t mask = block_mask<B>(v[j], sc.lim);
                    if (B == 16)
                        reinterpret_cast<uint16_t *>(T.mask)[blk] = (uint16_t)mask;
                    else
                        reinterpret_cast<uint32_t *>(T.mask)[blk] = mask;
                }
            }
        }
    }
    if (RESET && a.n_reset) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
        if (lane == 0 && cnt)
            atomicAdd(a.n_reset, cnt);
    }
}

// Reset: one thread per 16-byte chunk, four chunks in flight per thread.
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
        for (int k0 = 0; k0 < kOsciTileChunks; k0 += kOsciThreads * kOsciU) {
            float4 dq[kOsciU], dm[kOsciU];
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch < nch) {
                    dq[k] = ldf4_rw(T.dist_q + ch * 4);
                    dm[k] = ldf4_rw(T.dist_m + ch * 4);
                }
            }
#pragma unroll
            for (int k = 0; k < kOsciU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch >= nch)
                    continue;
                const float q4[4] = {dq[k].x, dq[k].y, dq[k].z, dq[k].w};
                const float m4[4] = {dm[k].x, dm[k].y, dm[k].z, dm[k].w};
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
    const int64_t cap = (int64_t)sm_count() * 8;
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
    const int key = (fmt * 2 + rnd) * 2 + (a.reset ? 1 : 0);
    switch (key) {
    case (NVFP4 * 2 + RNE) * 2: osci_pass_b<NVFP4, RNE, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NVFP4 * 2 + RNE) * 2 + 1: osci_pass_b<NVFP4, RNE, true><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NVFP4 * 2 + SR) * 2: osci_pass_b<NVFP4, SR, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NVFP4 * 2 + SR) * 2 + 1: osci_pass_b<NVFP4, SR, true><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (MXFP4 * 2 + RNE) * 2: osci_pass_b<MXFP4, RNE, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (MXFP4 * 2 + RNE) * 2 + 1: osci_pass_b<MXFP4, RNE, true><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (MXFP4 * 2 + SR) * 2: osci_pass_b<MXFP4, SR, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (MXFP4 * 2 + SR) * 2 + 1: osci_pass_b<MXFP4, SR, true><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NV2L * 2 + RNE) * 2: osci_pass_b<NV2L, RNE, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NV2L * 2 + RNE) * 2 + 1: osci_pass_b<NV2L, RNE, true><<<grid, kOsciThreads, 0, s>>>(a); break;
    case (NV2L * 2 + SR) * 2: osci_pass_b<NV2L, SR, false><<<grid, kOsciThreads, 0, s>>>(a); break;
    default: osci_pass_b<NV2L, SR, true><<<grid, kOsciThreads, 0, s>>>(a); break;
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
