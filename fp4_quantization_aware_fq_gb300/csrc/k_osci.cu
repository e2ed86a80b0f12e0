// k_osci.cu -- OsciReset statistics and reset ("Resumo Técnico: TetraJet-v2"
// §2B): the oscillation risk of a weight is the distance its quantized value
// travelled (dist_Q) over the distance its master value travelled (dist_M);
// weights whose risk exceeds a threshold are moved to the quantized value of
// their current bin.
//
// An NVFP4 optimizer step is two passes over a group of tensors (e.g. all
// expert matrices of an MoE layer), each a persistent grid walking 16-byte
// chunks of FP32 master weights tile by tile across the whole group:
//   A: w += delta, dist_M += |w_t - w_{t-1}|, per-tensor amax of w_t (atomic);
//   B: fake-quantize w_t under the new tensor scale, decode w_{t-1}'s stored
//      codes, dist_Q += |xhat_t - xhat_{t-1}|, write codes/scales/xhat/mask
//      (one lane per 16-byte chunk; the lanes of a block share its scale).
// The tensor amax is the only dependency between the passes, hence the split.
// MXFP4 and the double block scale each block from its own values, so their
// step is pass B alone with pass A's update done in its registers (FUSED).
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kOsciThreads = 256;
constexpr int kOsciU = 4;   // chunks in flight per thread: the reset pass
// Pass A: eight chunks in flight per thread (128 registers: two CTAs per SM)
// measured 1% faster on the 32-expert step than four.
constexpr int kOsciAU = 8;
// Pass B, four CTAs per SM (at most 64 registers).  With the window-end reset
// (eleven streams per chunk) one chunk per thread at a time measured fastest
// on the 32-expert step: 7.10 ms, against 7.22 with two chunks and 7.84 with
// four.  The ordinary step's pass B (nine streams) holds two chunks per
// thread: 5.61 ms against 5.88 with one.
template <bool RESET, bool FUSED = false>
__host__ __device__ constexpr int osci_bu()
{
    return (RESET || FUSED) ? 1 : 2;
}
constexpr int kOsciBMinCtas = 4;

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
        for (int k0 = 0; k0 < kOsciTileChunks; k0 += kOsciThreads * kOsciAU) {
            float4 w[kOsciAU], d[kOsciAU], dm[kOsciAU];
#pragma unroll
            for (int k = 0; k < kOsciAU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch < nch) {
                    w[k] = ldf4_rw(T.master + ch * 4);
                    d[k] = ldf4(T.delta + ch * 4);
                    dm[k] = ldf4_rw(T.dist_m + ch * 4);
                }
            }
#pragma unroll
            for (int k = 0; k < kOsciAU; ++k) {
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

// Four E2M1 nibbles of four values (16 bits; element 2j in the low nibble of
// byte j), nearest-even and saturating.
__device__ __forceinline__ uint32_t e2m1_rn_pack4(float y0, float y1, float y2, float y3)
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
        : "f"(y0), "f"(y1), "f"(y2), "f"(y3));
    return out;
}

// Grid values of four E2M1 nibbles (the low 16 bits of q).
__device__ __forceinline__ void e2m1_decode4(uint32_t q, float *out)
{
    uint32_t h[2];
    asm("{\n\t"
        ".reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
        "}"
        : "=r"(h[0]), "=r"(h[1])
        : "r"(q));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[i]));
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// Maximum, and OR, over aligned groups of L lanes.
template <int L>
__device__ __forceinline__ float lanes_max(float v)
{
#pragma unroll
    for (int o = 1; o < L; o <<= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
template <int L>
__device__ __forceinline__ uint32_t lanes_or(uint32_t v)
{
#pragma unroll
    for (int o = 1; o < L; o <<= 1)
        v |= __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Pass B: one thread per 16-byte chunk of 4 master weights (osci_bu chunks
// per thread at a time), so every load and store of the per-weight arrays is
// a coalesced 16-byte vector per lane, as in pass A.  The B/4 lanes of a block
// (4; 8 for MXFP4) share its amax, scale and mask bits through shuffles; for
// the double block the 32 lanes of a warp hold one 128-element outer block.
// With RESET, this step also ends the OsciReset window: where the new
// dist_Q exceeds threshold * dist_M, the master weight becomes xhat_t, and
// both accumulators are written back as zero (the same bits as the separate
// reset pass after this update).
// FUSED (block-local scales: MXFP4 and the double block, which need no tensor
// amax): pass A's update is done here too, in the same registers -- w_t =
// w_{t-1} + delta and dist_M += |w_t - w_{t-1}| with the same FP32 operations
// -- so the step is one pass that reads the master weights once.
template <int FMT, int RND, bool RESET, bool FUSED>
__global__ void __launch_bounds__(kOsciThreads, kOsciBMinCtas)
    osci_pass_b(const __grid_constant__ OsciArgs a)
{
    constexpr int B = FmtInfo<FMT>::B;
    constexpr int L = B / 4;  // lanes per block
    __shared__ NvTables tab, tabp;  // NVFP4: this step's and the previous step's tensor scale
    const int64_t ntiles = a.tile_start[a.ntensors];
    const PhiloxKey &key = a.key;
    int t = 0, t_tab = -1;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (L - 1);  // this lane's chunk within its block
    unsigned long long cnt = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        while (a.tile_start[t + 1] <= tile)
            ++t;
        const OsciTensor &T = a.t[t];
        const int64_t nch = T.n / 4;
        const int64_t cbeg = (tile - a.tile_start[t]) * kOsciTileChunks;
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
            if (cbeg == 0 && threadIdx.x == 0)
                T.ntscale[0] = s_g;
        }
        constexpr int BU = osci_bu<RESET, FUSED>();
        for (int k0 = 0; k0 < kOsciTileChunks; k0 += kOsciThreads * BU) {
            float4 w[BU], dq[BU], dm[BU], dl[BU];
            uint32_t qp[BU], scp[BU];
            float so_p[BU];
#pragma unroll
            for (int k = 0; k < BU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                if (ch < nch) {
                    w[k] = ldf4_rw(T.master + ch * 4);
                    if (FUSED)
                        dl[k] = ldf4(T.delta + ch * 4);
                    dq[k] = ldf4_rw(T.dist_q + ch * 4);
                    dm[k] = (RESET || FUSED) ? ldf4_rw(T.dist_m + ch * 4)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    qp[k] = __ldg(reinterpret_cast<const uint16_t *>(T.pcodes) + ch);
                    scp[k] = __ldg(T.pscales + ch / L);
                    so_p[k] = (FMT == NV2L) ? __ldg(T.ptscale + ch / 32) : 0.0f;
                } else {
                    w[k] = dq[k] = dm[k] = dl[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    qp[k] = scp[k] = 0;
                    so_p[k] = 0.0f;
                }
            }
#pragma unroll
            for (int k = 0; k < BU; ++k) {
                const int64_t ch = cbeg + k0 + k * kOsciThreads + threadIdx.x;
                const bool valid = ch < nch;  // uniform over a block's lanes (nch % L == 0)
                const int64_t blk = ch / L;
                float v[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
                float m4[4] = {dm[k].x, dm[k].y, dm[k].z, dm[k].w};
                if (FUSED) {
                    // pass A in registers: the same operations as osci_pass_a
                    const float d4[4] = {dl[k].x, dl[k].y, dl[k].z, dl[k].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float wn = __fadd_rn(v[i], d4[i]);
                        m4[i] = __fadd_rn(m4[i], fabsf(__fsub_rn(wn, v[i])));
                        v[i] = wn;
                    }
                }
                float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
                am = lanes_max<L>(am);
                float s_o = s_g, inv6b = inv6;
                if (FMT == NV2L) {
                    s_o = outer_scale(lanes_max<32>(am));
                    inv6b = nv_inv6(s_o);
                }
                const Scale sc = block_scale<FMT>(am, s_o, inv6b, &tab);
                float y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    y[i] = __fmul_rn(v[i], sc.r);
                if (RND == SR) {
                    // elements 4ch .. 4ch+3: half ch % 2 of Philox group ch / 2
                    const uint4 rb = sr_bits8(key, (uint64_t)ch >> 1, 0u, a.offset);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        y[i] = e2m1_sr_value(y[i], sr_operand(rb, 4 * (int)(ch & 1) + i));
                }
                const uint32_t q = e2m1_rn_pack4(y[0], y[1], y[2], y[3]);
                uint32_t clip = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    clip |= (__float_as_uint(__fsub_rn(sc.lim, fabsf(v[i]))) >> 31) << i;
                const uint32_t mask = lanes_or<L>((~clip & 15u) << (4 * sub));
                if (!valid)
                    continue;
                const float seff_p = (FMT == NVFP4) ? tabp.e[scp[k] & 127u].x
                                                    : stored_s_eff<FMT>(scp[k], so_p[k]);
                float xh[4], xp[4];
                e2m1_decode4(q, xh);
                e2m1_decode4(qp[k], xp);
                const float q4[4] = {dq[k].x, dq[k].y, dq[k].z, dq[k].w};
                float dn[4];
                uint32_t hit = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xh[i] = __fmul_rn(xh[i], sc.s_eff);
                    xp[i] = __fmul_rn(xp[i], seff_p);
                    dn[i] = __fadd_rn(q4[i], fabsf(__fsub_rn(xh[i], xp[i])));
                    if (RESET && dn[i] > __fmul_rn(a.threshold, m4[i])) {
                        if (!FUSED)
                            T.master[ch * 4 + i] = xh[i];
                        hit |= 1u << i;
                    }
                }
                if (FUSED)  // w_t, or xhat_t where the window-end reset moves it
                    stf4(T.master + ch * 4,
                         make_float4((hit & 1u) ? xh[0] : v[0], (hit & 2u) ? xh[1] : v[1],
                                     (hit & 4u) ? xh[2] : v[2], (hit & 8u) ? xh[3] : v[3]));
                if (T.xhat) {
                    if (a.xhat_bf16)
                        *reinterpret_cast<uint2 *>((char *)T.xhat + ch * 8) =
                            make_uint2(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]));
                    else
                        stf4(reinterpret_cast<float *>(T.xhat) + ch * 4,
                             make_float4(xh[0], xh[1], xh[2], xh[3]));
                }
                if (RESET) {
                    stf4(T.dist_q + ch * 4, make_float4(0.f, 0.f, 0.f, 0.f));
                    stf4(T.dist_m + ch * 4, make_float4(0.f, 0.f, 0.f, 0.f));
                    cnt += __popc(hit);
                } else {
                    stf4(T.dist_q + ch * 4, make_float4(dn[0], dn[1], dn[2], dn[3]));
                    if (FUSED)
                        stf4(T.dist_m + ch * 4, make_float4(m4[0], m4[1], m4[2], m4[3]));
                }
                reinterpret_cast<uint16_t *>(T.ncodes)[ch] = (uint16_t)q;
                if (sub == 0) {
                    T.nscales[blk] = (uint8_t)sc.code;
                    if (T.mask) {
                        if (B == 16)
                            reinterpret_cast<uint16_t *>(T.mask)[blk] = (uint16_t)mask;
                        else
                            reinterpret_cast<uint32_t *>(T.mask)[blk] = mask;
                    }
                }
                if (FMT == NV2L && lane == 0)
                    T.ntscale[ch / 32] = s_o;
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

template <int FMT, int RND, bool RESET, bool FUSED>
static void pass_b(const OsciArgs &a, int grid, cudaStream_t s)
{
    osci_pass_b<FMT, RND, RESET, FUSED><<<grid, kOsciThreads, 0, s>>>(a);
}

template <int FMT, bool FUSED>
static void pass_b_fmt(const OsciArgs &a, int rnd, int grid, cudaStream_t s)
{
    if (rnd == RNE)
        a.reset ? pass_b<FMT, RNE, true, FUSED>(a, grid, s) : pass_b<FMT, RNE, false, FUSED>(a, grid, s);
    else
        a.reset ? pass_b<FMT, SR, true, FUSED>(a, grid, s) : pass_b<FMT, SR, false, FUSED>(a, grid, s);
}

cudaError_t launch_osci_update(const OsciArgs &a, int fmt, int rnd, cudaStream_t s)
{
    const int64_t ntiles = a.tile_start[a.ntensors];
    if (ntiles == 0)
        return cudaSuccess;
    const int grid = osci_grid(ntiles);
    if (fmt == NVFP4) {
        // the tensor scale of w_t needs all of w_t first: two passes
        cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(float) * (size_t)a.ntensors, s);
        if (e != cudaSuccess)
            return e;
        osci_pass_a<<<grid, kOsciThreads, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        pass_b_fmt<NVFP4, false>(a, rnd, grid, s);
    } else if (fmt == MXFP4) {
        pass_b_fmt<MXFP4, true>(a, rnd, grid, s);  // block-local scales: one pass
    } else {
        pass_b_fmt<NV2L, true>(a, rnd, grid, s);
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
