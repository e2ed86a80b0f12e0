// k_qad.cu -- the QAD distillation loss ("Quantization-Aware Distillation for
// NVFP4 Inference Accuracy Recovery", §2 Metodologia): per row of teacher and
// student logits, KL(softmax(zt / T) || softmax(zs / T)) and its gradient with
// respect to the student logits, g (q - p) / T, in one read of both tensors.
//
// A row (a vocabulary of up to a few hundred thousand logits) is spread over
// a thread-block cluster of C CTAs; each CTA pulls its chunk of both rows
// into shared memory with two bulk copies and keeps it there for the three
// sweeps the row needs (maxima, sums of exponentials, then p, q, the KL terms
// and the gradient).  The per-CTA maxima and sums are combined through
// distributed shared memory, so HBM sees each logit once and each gradient
// once.  Clusters are persistent over rows; the next row's copies are issued
// as soon as the current chunk has been read for the last time.
//
// Arithmetic is FP32 in base 2: a = zt log2(e) / T and b = zs log2(e) / T,
// each row's maximum G and S = sum 2^(a - G); then log2 p = (a - G_t) -
// log2 S_t, log2 q = (b - G_s) - log2 S_s, and KL = ln 2 * sum p (log2 p -
// log2 q).  Both logarithms stay small for every token with weight, so the
// result does not lose accuracy when the two rows' logits sit far apart.
#include <math.h>

#include "fq_async.cuh"
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kKlThreads = 512;
constexpr int kKlWarps = kKlThreads / 32;
constexpr int kKlMaxCluster = 8;
constexpr size_t kKlSmemTwoPerSm = 110 * 1024;  // two CTAs per SM
constexpr size_t kKlSmemOnePerSm = 220 * 1024;  // one CTA per SM

bool qad_plan(int64_t vocab, int esz, int *csize, int64_t *chunk, size_t *smem)
{
    for (size_t cap : {kKlSmemTwoPerSm, kKlSmemOnePerSm}) {
        for (int c = 1; c <= kKlMaxCluster; c *= 2) {
            const int64_t L = ((vocab + c - 1) / c + 7) / 8 * 8;
            const size_t b = 2 * (size_t)L * (size_t)esz;
            if (b <= cap) {
                *csize = c;
                *chunk = L;
                *smem = b;
                return true;
            }
        }
    }
    return false;
}

// Eight consecutive logits of a chunk in shared memory, as FP32.
template <typename T>
__device__ __forceinline__ void lds8(const T *base, int g, float *v)
{
    constexpr int E = VecInfo<T>::E;
    const uint4 *p = reinterpret_cast<const uint4 *>(base) + (size_t)g * (8 / E);
#pragma unroll
    for (int k = 0; k < 8 / E; ++k)
        unpack16<T>(p[k], v + k * E);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// CTA-wide reductions of two values; every thread gets the results.  The
// order of the additions is fixed (a butterfly in each warp, then the warps
// in index order), so the sums are reproducible.
__device__ __forceinline__ float2 cta_max2(float x, float y, float2 *red)
{
    x = warp_max(x);
    y = warp_max(y);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = make_float2(x, y);
    __syncthreads();
    float2 r = red[0];
#pragma unroll
    for (int w = 1; w < kKlWarps; ++w)
        r = make_float2(fmaxf(r.x, red[w].x), fmaxf(r.y, red[w].y));
    __syncthreads();
    return r;
}

__device__ __forceinline__ float2 cta_sum2(float x, float y, float2 *red)
{
    x = warp_sum(x);
    y = warp_sum(y);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = make_float2(x, y);
    __syncthreads();
    float2 r = red[0];
#pragma unroll
    for (int w = 1; w < kKlWarps; ++w)
        r = make_float2(r.x + red[w].x, r.y + red[w].y);
    __syncthreads();
    return r;
}

template <typename T>
__global__ void __launch_bounds__(kKlThreads) qad_kl_kernel(const KlArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    T *bt = reinterpret_cast<T *>(smem);
    T *bs = bt + a.chunk;
    __shared__ uint64_t bar;
    __shared__ float4 slot1;   // this CTA's (M_t, S_t, M_s, S_s), base 2
    __shared__ float4 slot2;   // this CTA's KL partial (x)
    __shared__ float4 comb;    // the row's maxima and log2 sums (G_t, G_s, log2 S_t, log2 S_s)
    __shared__ float2 red[kKlWarps];

    const uint32_t rank = cluster_rank();
    const int C = a.csize;
    const int64_t c0 = (int64_t)rank * a.chunk;
    int64_t len = a.vocab - c0;
    len = len < 0 ? 0 : (len > a.chunk ? a.chunk : len);
    const int ng = (int)(len / 8);
    const uint32_t bytes = (uint32_t)(len * (int64_t)sizeof(T));
    const int64_t row0 = cluster_id_x(), rstep = num_clusters_x();
    const float k2 = a.k2, gk = a.gk;

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    auto issue = [&](int64_t row) {
        mbar_arrive_expect_tx(&bar, 2 * bytes);
        if (bytes) {
            const int64_t off = (row * a.vocab + c0) * (int64_t)sizeof(T);
            bulk_g2s(bt, (const char *)a.zt + off, bytes, &bar);
            bulk_g2s(bs, (const char *)a.zs + off, bytes, &bar);
        }
    };
    if (threadIdx.x == 0 && row0 < a.rows)
        issue(row0);

    bool dead = false;  // a copy did not arrive in time: stop loading, keep the barriers
    uint32_t parity = 0;
    for (int64_t row = row0; row < a.rows; row += rstep) {
        if (!dead) {
            const bool late = !mbar_wait(&bar, parity);
            parity ^= 1u;
            if (__syncthreads_or(late)) {
                dead = true;
                if (threadIdx.x == 0 && a.err)
                    atomicOr(a.err, (int)kDevErrWaitTimeout);
            }
        }
        // sweep 1: maxima of the raw logits (scaling by k2 > 0 keeps the order)
        float mt = -INFINITY, ms = -INFINITY;
        for (int g = threadIdx.x; g < ng; g += kKlThreads) {
            float v[8], w[8];
            lds8<T>(bt, g, v);
            lds8<T>(bs, g, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mt = fmaxf(mt, v[i]);
                ms = fmaxf(ms, w[i]);
            }
        }
        const float2 m = cta_max2(mt, ms, red);
        const float m2t = m.x * k2, m2s = m.y * k2;
        // sweep 2: sums of 2^(a - M) under this CTA's maxima
        float st = 0.0f, ss = 0.0f;
        for (int g = threadIdx.x; g < ng; g += kKlThreads) {
            float v[8], w[8];
            lds8<T>(bt, g, v);
            lds8<T>(bs, g, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                st += exp2f(fmaf(v[i], k2, -m2t));
                ss += exp2f(fmaf(w[i], k2, -m2s));
            }
        }
        const float2 s = cta_sum2(st, ss, red);
        if (threadIdx.x == 0)
            slot1 = make_float4(m2t, s.x, m2s, s.y);
        cluster_sync();
        if (threadIdx.x == 0) {
            // combine the cluster's partials in rank order (identical in every CTA)
            float4 part[kKlMaxCluster];
            float gt = -INFINITY, gs = -INFINITY;
            for (int r = 0; r < C; ++r) {
                part[r] = dsmem_ld_f4(&slot1, (uint32_t)r);
                gt = fmaxf(gt, part[r].x);
                gs = fmaxf(gs, part[r].z);
            }
            float sum_t = 0.0f, sum_s = 0.0f;
            for (int r = 0; r < C; ++r) {
                sum_t += part[r].y * exp2f(part[r].x - gt);
                sum_s += part[r].w * exp2f(part[r].z - gs);
            }
            comb = make_float4(gt, gs, log2f(sum_t), log2f(sum_s));
        }
        __syncthreads();
        const float gt = comb.x, gs = comb.y, l2t = comb.z, l2s = comb.w;
        // sweep 3: p, q, the KL terms and the gradient
        float kl = 0.0f;
        char *dzrow = a.dz ? (char *)a.dz + (row * a.vocab + c0) * (a.dz_bf16 ? 2 : 4) : nullptr;
        for (int g = threadIdx.x; g < ng; g += kKlThreads) {
            float v[8], w[8], o[8];
            lds8<T>(bt, g, v);
            lds8<T>(bs, g, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // log2 p and log2 q relative to each row's own maximum: small
                // for every token that matters, whatever the logits' offset
                const float lp = fmaf(v[i], k2, -gt) - l2t;
                const float lq = fmaf(w[i], k2, -gs) - l2s;
                const float p = exp2f(lp);
                kl = fmaf(p, lp - lq, kl);
                if (dzrow)
                    o[i] = gk * (exp2f(lq) - p);
            }
            if (dzrow) {
                if (a.dz_bf16) {
                    *reinterpret_cast<uint4 *>(dzrow + (size_t)g * 16) =
                        make_uint4(bf16x2_rn(o[0], o[1]), bf16x2_rn(o[2], o[3]),
                                   bf16x2_rn(o[4], o[5]), bf16x2_rn(o[6], o[7]));
                } else {
                    float4 *d = reinterpret_cast<float4 *>(dzrow + (size_t)g * 32);
                    d[0] = make_float4(o[0], o[1], o[2], o[3]);
                    d[1] = make_float4(o[4], o[5], o[6], o[7]);
                }
            }
        }
        const float2 k = cta_sum2(kl, 0.0f, red);  // also: every thread is done with the chunk
        if (threadIdx.x == 0) {
            slot2 = make_float4(k.x, 0.0f, 0.0f, 0.0f);
            const int64_t next = row + rstep;
            if (!dead && next < a.rows) {
                fence_proxy_async_smem();
                issue(next);
            }
        }
        cluster_sync();
        if (rank == 0 && threadIdx.x == 0) {
            float tot = 0.0f;
            for (int r = 0; r < C; ++r)
                tot += dsmem_ld_f4(&slot2, (uint32_t)r).x;
            a.loss_rows[row] = tot * 0.693147180559945309f;
        }
    }
    cluster_sync();  // keep this CTA's slots alive until rank 0 has read them
}

// Mean of the per-row losses in double precision, in a fixed order.
constexpr int kMeanThreads = 1024;

__global__ void __launch_bounds__(kMeanThreads) qad_mean_kernel(const float *__restrict__ loss,
                                                                int64_t rows,
                                                                float *__restrict__ out)
{
    __shared__ double part[kMeanThreads / 32];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < rows; i += kMeanThreads)
        s += (double)loss[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kMeanThreads / 32; ++w)
            t += part[w];
        out[0] = rows ? (float)(t / (double)rows) : 0.0f;
    }
}

template <typename T>
static cudaError_t qad_go(KlArgs a, size_t smem, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(qad_kl_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kKlThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as fit on the GPU at once (persistent over rows)
    cfg.gridDim = dim3((unsigned)(a.csize * 1024));
    int fit = 0;
    if (cudaOccupancyMaxActiveClusters(&fit, qad_kl_kernel<T>, &cfg) != cudaSuccess || fit < 1)
        fit = sm_count() / a.csize > 0 ? sm_count() / a.csize : 1;
    (void)cudaGetLastError();
    const int64_t ncl = a.rows < fit ? a.rows : fit;
    cfg.gridDim = dim3((unsigned)(a.csize * ncl));
    return cudaLaunchKernelEx(&cfg, qad_kl_kernel<T>, a);
}

cudaError_t launch_qad_kl(const KlArgs &a, int bf16, size_t smem, float *loss_mean,
                          cudaStream_t s)
{
    if (a.rows > 0) {
        cudaError_t e = bf16 ? qad_go<__nv_bfloat16>(a, smem, s) : qad_go<float>(a, smem, s);
        if (e != cudaSuccess)
            return e;
    }
    if (loss_mean) {
        qad_mean_kernel<<<1, kMeanThreads, 0, s>>>(a.loss_rows, a.rows, loss_mean);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace fqk
