// k_qad.cu -- the QAD distillation loss ("Quantization-Aware Distillation for
// NVFP4 Inference Accuracy Recovery", §2 Metodologia): per row of teacher and
// student logits, KL(softmax(zt / T) || softmax(zs / T)) and its gradient with
// respect to the student logits, g (q - p) / T, in one read of both tensors.
//
// A row (a vocabulary of up to a few hundred thousand logits) is spread over
// a thread-block cluster of C CTAs; each CTA pulls its chunk of both rows
// into shared memory with two bulk copies and keeps it there for the two
// sweeps the row needs (maxima with the sums of exponentials under running
// maxima, then p, q, the KL terms and the gradient).  The per-CTA maxima and sums are combined through
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

constexpr int kKlMaxCluster = 8;
constexpr size_t kKlSmemTwoPerSm = 110 * 1024;  // two CTAs per SM
constexpr size_t kKlSmemOnePerSm = 220 * 1024;  // one CTA per SM

// Preference: two 512-thread CTAs per SM (one CTA's sweeps overlap the
// other's copies), else one 1024-thread CTA per SM; within each, the smallest
// cluster whose chunks fit.
bool qad_plan(int64_t vocab, int esz, QadPlan *p)
{
    struct Opt {
        int threads;
        size_t cap;
    };
    const Opt opts[2] = {{512, kKlSmemTwoPerSm}, {1024, kKlSmemOnePerSm}};
    for (const Opt &o : opts) {
        for (int c = 1; c <= kKlMaxCluster; c *= 2) {
            const int64_t L = ((vocab + c - 1) / c + 7) / 8 * 8;
            const size_t b = 2 * (size_t)L * (size_t)esz;
            if (b <= o.cap) {
                p->csize = c;
                p->chunk = L;
                p->smem = b;
                p->threads = o.threads;
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

// 2^x on the special-function unit (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 ex2x2(float2 x) { return make_float2(ex2(x.x), ex2(x.y)); }

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

// CTA-wide sum of two values; every thread gets the results.  The order of
// the additions is fixed (a butterfly in each warp, then the warps in index
// order), so the sums are reproducible.  One barrier: the caller alternates
// between two `red` buffers, so a buffer is written again only after further
// barriers that every reader of it has passed.
template <int NW>
__device__ __forceinline__ float2 cta_sum2(float x, float y, float2 *red)
{
    x = warp_sum(x);
    y = warp_sum(y);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = make_float2(x, y);
    __syncthreads();
    float2 r = red[0];
#pragma unroll
    for (int w = 1; w < NW; ++w)
        r = make_float2(r.x + red[w].x, r.y + red[w].y);
    return r;
}

// Combines each thread's (running maximum m, sum s of 2^(x k2 - m k2)) pairs
// of two tensors into the CTA's: the maximum M and the sum under it,
// sum s 2^(m k2 - M k2) (a thread or warp with no logits has m = -inf and
// s = 0 and adds nothing).  Returns (M_t, S_t, M_s, S_s) to every thread; the
// order of the additions is fixed, so the sums are reproducible.  Two
// barriers; as for cta_sum2, the caller alternates between two `red` buffers.
template <int NW>
__device__ __forceinline__ float4 cta_max_sum2(float mt, float st, float ms, float ss, float k2,
                                               float4 *red)
{
    static_assert(NW <= 32, "one warp combines the warps' pairs");
    const float wmt = warp_max(mt), wms = warp_max(ms);
    float ct = (wmt == -INFINITY) ? 0.0f : st * ex2(mt * k2 - wmt * k2);
    float cs = (wms == -INFINITY) ? 0.0f : ss * ex2(ms * k2 - wms * k2);
    ct = warp_sum(ct);
    cs = warp_sum(cs);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = make_float4(wmt, ct, wms, cs);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const float4 r = lane < NW ? red[lane] : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
        const float Mt = warp_max(r.x), Ms = warp_max(r.z);
        const float St = warp_sum(r.x == -INFINITY ? 0.0f : r.y * ex2(r.x * k2 - Mt * k2));
        const float Ss = warp_sum(r.z == -INFINITY ? 0.0f : r.w * ex2(r.z * k2 - Ms * k2));
        __syncwarp();
        if (lane == 0)
            red[NW] = make_float4(Mt, St, Ms, Ss);
    }
    __syncthreads();
    return red[NW];
}

// Cluster barrier after this CTA's threads 0..C-1 pushed their payload into
// other CTAs' shared memory: those threads fence (release); every thread
// arrives relaxed and waits with acquire semantics.
__device__ __forceinline__ void cluster_sync_pushed()
{
    if (threadIdx.x < kKlMaxCluster)
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The chunk arrives in kKlParts parts, each with its own mbarrier: the first
// sweep starts on part 0 while the later parts are still in flight, and the
// next row's part p is requested as soon as the last sweep has finished with
// it, while that sweep works on the later parts.
constexpr int kKlParts = 2;
template <typename T, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) qad_kl_kernel(const KlArgs a)
{
    constexpr int NW = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bar[kKlParts];  // one per part of the chunk
    // per row parity, filled by every CTA of the cluster (remote stores before
    // the row's cluster barrier): each rank's (M_t, S_t, M_s, S_s) in base 2,
    // and (rank 0 only) each rank's KL partial
    __shared__ float4 part1[2][kKlMaxCluster];
    __shared__ float part2[2][kKlMaxCluster];
    __shared__ float4 comb;    // the row's maxima and log2 sums (G_t, G_s, log2 S_t, log2 S_s)
    __shared__ float2 red[2][NW];      // by row parity
    __shared__ float4 red4[2][NW + 1];

    const uint32_t rank = cluster_rank();
    const int C = a.csize;
    const int64_t c0 = (int64_t)rank * a.chunk;
    int64_t len = a.vocab - c0;
    len = len < 0 ? 0 : (len > a.chunk ? a.chunk : len);
    const int ng = (int)(len / 8);    // groups of 8 logits in this CTA's chunk
    // part p covers groups gpart(p) .. gpart(p + 1) - 1
    auto gpart = [&](int p) { return (int)(((int64_t)ng * p) / kKlParts); };
    const int64_t row0 = cluster_id_x(), rstep = num_clusters_x();
    const float k2 = a.k2, gk = a.gk;
    T *bt = reinterpret_cast<T *>(smem);
    T *bs = bt + a.chunk;

    if (threadIdx.x == 0) {
        for (int p = 0; p < kKlParts; ++p)
            mbar_init(&bar[p], 1);
        mbar_init_fence();
    }
    __syncthreads();
    auto issue_part = [&](int64_t row, int p) {
        const int g0 = gpart(p), g1 = gpart(p + 1);
        const uint32_t bytes = (uint32_t)((g1 - g0) * 8 * (int)sizeof(T));
        mbar_arrive_expect_tx(&bar[p], 2 * bytes);
        if (bytes) {
            const int64_t off = (row * a.vocab + c0 + 8 * (int64_t)g0) * (int64_t)sizeof(T);
            bulk_g2s(bt + 8 * g0, (const char *)a.zt + off, bytes, &bar[p]);
            bulk_g2s(bs + 8 * g0, (const char *)a.zs + off, bytes, &bar[p]);
        }
    };
    if (threadIdx.x == 0 && row0 < a.rows)
        for (int p = 0; p < kKlParts; ++p)
            issue_part(row0, p);

    // A copy that did not arrive in time: this thread stops waiting (thread 0
    // also stops loading), records the error and keeps joining the barriers.
    // Every thread waits on the part's barrier itself, so no CTA barrier is
    // spent on the wait; after a timeout each thread gives up on its own, once.
    bool dead = false;
    auto wait_part = [&](int p, int it) {
        if (dead)
            return;
        if (!mbar_wait(&bar[p], (uint32_t)it & 1u)) {
            dead = true;
            if (a.err)
                atomicOr(a.err, (int)kDevErrWaitTimeout);
        }
    };
    int it = 0;
    for (int64_t row = row0; row < a.rows; row += rstep, ++it) {
        const int64_t next = row + rstep;
        // sweep 1: maxima and sums of exponentials in one pass.  Each thread
        // keeps a running maximum of the raw logits (scaling by k2 > 0 keeps
        // the order) and the sum of 2^(a - M) under it, rescaling the sum when
        // a group of 8 raises the maximum; the CTA then combines the threads'
        // (maximum, sum) pairs under the CTA's maximum.
        const float2 vk2 = make_float2(k2, k2);
        float mt = -INFINITY, ms = -INFINITY, st = 0.0f, ss = 0.0f;
        for (int p = 0; p < kKlParts; ++p) {
            wait_part(p, it);
            const int g1 = gpart(p + 1);
            for (int g = gpart(p) + threadIdx.x; g < g1; g += NT) {
                float v[8], w[8];
                lds8<T>(bt, g, v);
                lds8<T>(bs, g, w);
                float gmt = v[0], gms = w[0];
#pragma unroll
                for (int i = 1; i < 8; ++i) {
                    gmt = fmaxf(gmt, v[i]);
                    gms = fmaxf(gms, w[i]);
                }
                if (gmt > mt) {
                    st *= ex2(mt * k2 - gmt * k2);
                    mt = gmt;
                }
                if (gms > ms) {
                    ss *= ex2(ms * k2 - gms * k2);
                    ms = gms;
                }
                const float2 nmt = make_float2(-mt * k2, -mt * k2);
                const float2 nms = make_float2(-ms * k2, -ms * k2);
                float2 st2 = make_float2(0.0f, 0.0f), ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    st2 = add2(st2, ex2x2(fma2(make_float2(v[i], v[i + 1]), vk2, nmt)));
                    ss2 = add2(ss2, ex2x2(fma2(make_float2(w[i], w[i + 1]), vk2, nms)));
                }
                st += st2.x + st2.y;
                ss += ss2.x + ss2.y;
            }
        }
        const float4 ms4 = cta_max_sum2<NW>(mt, st, ms, ss, k2, red4[it & 1]);
        const float m2t = ms4.x * k2, m2s = ms4.z * k2;
        const float2 s = make_float2(ms4.y, ms4.w);
        // push this CTA's partials into every CTA of the cluster (lane r -> rank r)
        if (threadIdx.x < C)
            dsmem_st_f4(&part1[it & 1][rank], (uint32_t)threadIdx.x,
                        make_float4(m2t, s.x, m2s, s.y));
        // one cluster barrier per row: it publishes this row's partials and
        // the previous row's KL partials (stored at the end of that row)
        cluster_sync_pushed();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            if (rank == 0 && it > 0) {
                const float tot = warp_sum(lane < C ? part2[(it - 1) & 1][lane] : 0.0f);
                if (lane == 0)
                    a.loss_rows[row - rstep] = tot * 0.693147180559945309f;
            }
            // combine the cluster's partials (the same butterfly in every CTA)
            float4 pr = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
            if (lane < C)
                pr = part1[it & 1][lane];
            const float gt = warp_max(pr.x), gs = warp_max(pr.z);
            const float sum_t = warp_sum(lane < C ? pr.y * ex2(pr.x - gt) : 0.0f);
            const float sum_s = warp_sum(lane < C ? pr.w * ex2(pr.z - gs) : 0.0f);
            if (lane == 0)
                comb = make_float4(gt, gs, log2f(sum_t), log2f(sum_s));
        }
        __syncthreads();
        const float gt = comb.x, gs = comb.y, l2t = comb.z, l2s = comb.w;
        // sweep 3: p, q, the KL terms and the gradient, part by part
        const float2 ngt = make_float2(-gt, -gt), ngs = make_float2(-gs, -gs);
        const float2 vl2t = make_float2(l2t, l2t), vl2s = make_float2(l2s, l2s);
        const float2 vgk = make_float2(gk, gk);
        float2 kl2 = make_float2(0.0f, 0.0f);
        char *dzrow = a.dz ? (char *)a.dz + (row * a.vocab + c0) * (a.dz_bf16 ? 2 : 4) : nullptr;
        for (int part = 0; part < kKlParts; ++part) {
            const int g1 = gpart(part + 1);
            for (int g = gpart(part) + threadIdx.x; g < g1; g += NT) {
                float v[8], w[8], o[8];
                lds8<T>(bt, g, v);
                lds8<T>(bs, g, w);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    // log2 p and log2 q relative to each row's own maximum: small
                    // for every token that matters, whatever the logits' offset
                    const float2 lp = sub2(fma2(make_float2(v[i], v[i + 1]), vk2, ngt), vl2t);
                    const float2 lq = sub2(fma2(make_float2(w[i], w[i + 1]), vk2, ngs), vl2s);
                    const float2 p = ex2x2(lp);
                    kl2 = fma2(p, sub2(lp, lq), kl2);
                    if (dzrow) {
                        const float2 d = mul2(vgk, sub2(ex2x2(lq), p));
                        o[i] = d.x;
                        o[i + 1] = d.y;
                    }
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
            if (part + 1 < kKlParts) {
                // every thread is done with this part: request the next row's
                __syncthreads();
                if (threadIdx.x == 0 && !dead && next < a.rows) {
                    fence_proxy_async_smem();
                    issue_part(next, part);
                }
            }
        }
        const float2 k = cta_sum2<NW>(kl2.x + kl2.y, 0.0f, red[it & 1]);  // also: every thread is done with the last part
        if (threadIdx.x == 0) {
            dsmem_st_f32(&part2[it & 1][rank], 0u, k.x);  // to rank 0
            if (!dead && next < a.rows) {
                fence_proxy_async_smem();
                issue_part(next, kKlParts - 1);
            }
        }
    }
    // the last row's KL partials
    cluster_sync_pushed();
    if (rank == 0 && it > 0 && threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const float tot = warp_sum(lane < C ? part2[(it - 1) & 1][lane] : 0.0f);
        if (lane == 0)
            a.loss_rows[row0 + (int64_t)(it - 1) * rstep] = tot * 0.693147180559945309f;
    }
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

template <typename T, int NT>
static cudaError_t qad_go(const KlArgs &a, size_t smem, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(qad_kl_kernel<T, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(qad_kl_kernel<T, NT>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as fit on the GPU at once (persistent over rows)
    cfg.gridDim = dim3((unsigned)(a.csize * 1024));
    int fit = 0;
    if (cudaOccupancyMaxActiveClusters(&fit, qad_kl_kernel<T, NT>, &cfg) != cudaSuccess || fit < 1)
        fit = sm_count() / a.csize > 0 ? sm_count() / a.csize : 1;
    (void)cudaGetLastError();
    const int64_t ncl = a.rows < fit ? a.rows : fit;
    cfg.gridDim = dim3((unsigned)(a.csize * ncl));
    return cudaLaunchKernelEx(&cfg, qad_kl_kernel<T, NT>, a);
}

cudaError_t launch_qad_kl(const KlArgs &a0, int bf16, const QadPlan &p, float *loss_mean,
                          cudaStream_t s)
{
    KlArgs a = a0;
    a.csize = p.csize;
    a.chunk = p.chunk;
    if (a.rows > 0) {
        cudaError_t e;
        if (p.threads == 1024)
            e = bf16 ? qad_go<__nv_bfloat16, 1024>(a, p.smem, s) : qad_go<float, 1024>(a, p.smem, s);
        else
            e = bf16 ? qad_go<__nv_bfloat16, 512>(a, p.smem, s) : qad_go<float, 512>(a, p.smem, s);
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
