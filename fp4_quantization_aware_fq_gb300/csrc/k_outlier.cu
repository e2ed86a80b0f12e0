// k_outlier.cu -- static outlier retention ("Resumo Técnico: TetraJet-v2",
// §2C, OutControl): the channels with the largest norm over a short
// calibration window stay in FP8 (E4M3, static per-channel scale) while the
// rest of the activation is quantized to FP4 with those channels removed, so
// that they no longer inflate the block scales of their rows.
//
// channel_amax_kernel  running per-channel max |x| (the calibration norm)
// select_kernel        top-k channels (ties: lower index), bitmap, FP8 scales
// masked_amax_kernel   tensor amax without the retained channels (NVFP4)
// outlier_row_kernel   one thread per row block: FP4 of the block with the
//                      retained elements zeroed; FP8 codes of those elements
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kOutThreads = 256;

// Exclusive prefix sums of the popcounts of nwords bitmap words (shared or
// global) into pre[] (shared), by all NT threads of the CTA: each thread sums
// a contiguous run of words, the runs are scanned across the CTA, and the
// run is rewritten with its prefixes.  Ends with a __syncthreads.
template <int NT>
__device__ __forceinline__ void popc_prefix(const uint32_t *words, int nwords, int *pre)
{
    __shared__ int wsum[NT / 32];
    const int per = (nwords + NT - 1) / NT;
    const int w0 = threadIdx.x * per;
    const int w1 = w0 + per < nwords ? w0 + per : nwords;
    int run = 0;
    for (int w = w0; w < w1; ++w)
        run += __popc(words[w]);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o)
            inc += t;
    }
    if (lane == 31)
        wsum[warp] = inc;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < warp; ++i)
        base += wsum[i];
    int acc = base + inc - run;
    for (int w = w0; w < w1; ++w) {
        const int p = __popc(words[w]);
        pre[w] = acc;
        acc += p;
    }
    __syncthreads();
}

// ------------------------------------------------------------------ calibration
// A CTA covers 256 column vectors (16 bytes each) of a stripe of rows_per
// rows; four rows are loaded per iteration.
template <typename T>
__global__ void __launch_bounds__(kOutThreads) channel_amax_kernel(const void *__restrict__ x,
                                                                   int64_t rows, int64_t cols,
                                                                   int64_t rows_per,
                                                                   unsigned *__restrict__ amax)
{
    constexpr int E = VecInfo<T>::E;
    const int64_t cv = (int64_t)blockIdx.x * kOutThreads + threadIdx.x;  // column vector
    if (cv * E >= cols)
        return;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per;
    const int64_t r1 = r0 + rows_per < rows ? r0 + rows_per : rows;
    const char *p = (const char *)x + (r0 * cols + cv * E) * (int64_t)sizeof(T);
    const int64_t pitch = cols * (int64_t)sizeof(T);
    float m[E];
#pragma unroll
    for (int i = 0; i < E; ++i)
        m[i] = 0.0f;
    int64_t r = r0;
    for (; r + 4 <= r1; r += 4, p += 4 * pitch) {
        uint4 u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            u[k] = ld16(p + k * pitch);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v[E];
            unpack16<T>(u[k], v);
#pragma unroll
            for (int i = 0; i < E; ++i)
                m[i] = fmaxf(m[i], fabsf(v[i]));
        }
    }
    for (; r < r1; ++r, p += pitch) {
        float v[E];
        unpack16<T>(ld16(p), v);
#pragma unroll
        for (int i = 0; i < E; ++i)
            m[i] = fmaxf(m[i], fabsf(v[i]));
    }
#pragma unroll
    for (int i = 0; i < E; ++i)
        atomicMax(amax + cv * E + i, __float_as_uint(m[i]));
}

// ------------------------------------------------------------------ selection
// One CTA.  Channel c gets the unique 64-bit key (|amax_c| bits << 32) | ~c:
// a larger amax gives a larger key, and among equal amax the lower index.
// A most-significant-byte-first radix select (eight histogram passes over the
// keys) finds the k-th largest key K; the selected channels are exactly those
// with key >= K.  A popcount scan of the resulting bitmap then writes their
// indices in ascending order.
constexpr int kSelThreads = 1024;
constexpr int kMaxOutWords = 4096;  // channels up to 131072
constexpr int64_t kFastKept = 8192;  // retained channels listed in shared memory (12 B each)
constexpr int64_t kKeepImageCols = 16384;  // BF16 keep-mask image: 2 B per column (32 KB)

__host__ __device__ constexpr size_t align16(size_t n) { return (n + 15) & ~(size_t)15; }

// Dynamic shared memory of outlier_row_kernel: the prefix, the sorted list
// (fast), the keep-mask image (fast == 2).
static size_t outlier_smem(int64_t cols, int64_t k, int fast)
{
    const int64_t nwords = (cols + 31) / 32;
    size_t n = align16((size_t)nwords * 4);
    if (fast)
        n += align16((size_t)k * 12);
    if (fast == 2)
        n += (size_t)nwords * 64;
    return n;
}

__device__ __forceinline__ uint64_t channel_key(const float *amax, int c)
{
    return ((uint64_t)(__float_as_uint(__ldg(amax + c)) & 0x7FFFFFFFu) << 32) |
           (uint32_t)~(uint32_t)c;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float *__restrict__ amax,
                                                             int cols, int k,
                                                             int32_t *__restrict__ idx,
                                                             uint32_t *__restrict__ bitmap,
                                                             float *__restrict__ fp8_scale)
{
    __shared__ unsigned hist[256];
    __shared__ uint64_t s_prefix;
    __shared__ unsigned s_remaining;
    __shared__ uint32_t bm[kMaxOutWords];
    __shared__ int pre[kMaxOutWords];
    const int nwords = (cols + 31) / 32;
    uint64_t prefix = 0, pmask = 0;
    unsigned remaining = (unsigned)k;  // rank of K among the keys still matching
    for (int byte = 7; byte >= 0 && k > 0; --byte) {
        for (int i = threadIdx.x; i < 256; i += kSelThreads)
            hist[i] = 0u;
        __syncthreads();
        const int sh = 8 * byte;
        for (int c = threadIdx.x; c < cols; c += kSelThreads) {
            const uint64_t key = channel_key(amax, c);
            if ((key & pmask) == prefix)
                atomicAdd(&hist[(key >> sh) & 0xFFu], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned above = 0;
            int d = 255;
            for (; d > 0; --d) {
                if (above + hist[d] >= remaining)
                    break;
                above += hist[d];
            }
            s_prefix = prefix | ((uint64_t)d << sh);
            s_remaining = remaining - above;
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        pmask |= (uint64_t)0xFF << sh;
        __syncthreads();
    }
    for (int w = threadIdx.x; w < nwords; w += kSelThreads) {
        uint32_t bits = 0u;
        if (k > 0) {
            const int c1 = (w + 1) * 32 < cols ? (w + 1) * 32 : cols;
            for (int c = w * 32; c < c1; ++c)
                bits |= (uint32_t)(channel_key(amax, c) >= prefix) << (c & 31);
        }
        bm[w] = bits;
    }
    __syncthreads();
    popc_prefix<kSelThreads>(bm, nwords, pre);
    for (int w = threadIdx.x; w < nwords; w += kSelThreads) {
        uint32_t bits = bm[w];
        int j = pre[w];
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1;
            const int c = w * 32 + b;
            idx[j] = c;
            fp8_scale[j] = __fdiv_rn(__ldg(amax + c), 448.0f);
            ++j;
        }
        bitmap[w] = bm[w];
    }
}

// ------------------------------------------------------------------ masked amax
// A CTA covers 256 column vectors (16 bytes each) of a stripe of rows_per
// rows, as channel_amax_kernel: each thread's retained-channel bits are read
// once, and four rows' loads are in flight.
template <typename T>
__global__ void __launch_bounds__(kOutThreads) masked_amax_kernel(const void *__restrict__ x,
                                                                  int64_t rows, int64_t cols,
                                                                  int64_t rows_per,
                                                                  const uint32_t *__restrict__ bm,
                                                                  unsigned *__restrict__ out)
{
    constexpr int E = VecInfo<T>::E;
    constexpr int U = 4;
    const int64_t vpr = cols / E;
    const int64_t cv = (int64_t)blockIdx.x * kOutThreads + threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per;
    const int64_t r1 = r0 + rows_per < rows ? r0 + rows_per : rows;
    float m = 0.0f;
    if (cv < vpr) {
        const int64_t c0 = cv * E;
        const uint32_t bits = __ldg(bm + (c0 >> 5)) >> (c0 & 31);
        const char *col = (const char *)x + cv * 16;
        for (int64_t r = r0; r < r1; r += U) {
            uint4 raw[U];
#pragma unroll
            for (int k = 0; k < U; ++k)
                raw[k] = r + k < r1 ? ld16(col + (r + k) * vpr * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < U; ++k) {
                float v[E];
                unpack16<T>(raw[k], v);
#pragma unroll
                for (int i = 0; i < E; ++i)
                    if (!((bits >> i) & 1u))
                        m = fmaxf(m, fabsf(v[i]));
            }
        }
    }
    allow_dependent_launch();  // the split quantizer waits for this grid's atomics itself
    m = group_max<32>(m);
    __shared__ float wm[kOutThreads / 32];
    if ((threadIdx.x & 31) == 0)
        wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = wm[0];
        for (int w = 1; w < kOutThreads / 32; ++w)
            b = fmaxf(b, wm[w]);
        atomicMax(out, __float_as_uint(b));
    }
}

// ------------------------------------------------------------------ split quantization

// One scalar of x as FP32.
template <typename T>
__device__ __forceinline__ float ld_scalar(const void *x, int64_t e);
template <>
__device__ __forceinline__ float ld_scalar<float>(const void *x, int64_t e)
{
    return __ldg(reinterpret_cast<const float *>(x) + e);
}
template <>
__device__ __forceinline__ float ld_scalar<__nv_bfloat16>(const void *x, int64_t e)
{
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short *>(x) + e);
    return __uint_as_float((uint32_t)u << 16);
}

// Each thread quantizes one row block to FP4 with its kept elements zeroed
// (the kept columns are the same in every row, so 10% of the channels touch
// most blocks).  The kept elements themselves are then encoded by the warp
// together: the warp's kept elements are numbered by a scan of the per-thread
// counts and dealt out one per lane, so the FP8 work runs without divergence
// however the kept columns fall across the warp's blocks.  A lane finds the
// owner of its element by a binary search over the scan, re-reads the value
// (an L1 hit: the owner has just loaded it), writes the FP8 code and the
// kept value of xhat, and patches the owner's mask bits in shared memory.
template <typename T, int FMT, int RND>
__global__ void __launch_bounds__(kOutThreads) outlier_row_kernel(const __grid_constant__ OutlierArgs a, int fast)
{
    constexpr int B = FmtInfo<FMT>::B;
    __shared__ NvTables tab;
    __shared__ uint32_t mstage[kOutThreads];
    __shared__ float e4m3v[128];  // E4M3 magnitudes by code (0x7F unused)
    const int64_t cols = a.cols, rows = a.rows;
    const int nwords = (int)((cols + 31) / 32);
    const int kk = (int)a.k;
    // Dynamic shared memory (sizes from outlier_smem): the bitmap's popcount
    // prefix (one int per word); with fast, the retained columns in ascending
    // order, then 1 / s_j and s_j for each; with fast == 2 (BF16), a keep-mask
    // image of one row, one 16-bit half per column (0 for a retained column,
    // 0xFFFF otherwise), with which a block's retained elements are zeroed by
    // ANDing its raw words.  Each part starts on a 16-byte boundary.
    extern __shared__ __align__(16) unsigned char osm[];
    int *pre = reinterpret_cast<int *>(osm);
    int *kcols = reinterpret_cast<int *>(osm + align16((size_t)nwords * 4));
    float *krcp = reinterpret_cast<float *>(kcols + kk);
    float *ksj = krcp + kk;
    uint32_t *keep = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(kcols) +
                                                  align16((size_t)kk * 12));
    wait_prior_grid();
    popc_prefix<kOutThreads>(a.bitmap, nwords, pre);
    if (fast) {
        for (int w = threadIdx.x; w < nwords; w += kOutThreads) {
            uint32_t wd = __ldg(a.bitmap + w);
            for (int idx = pre[w]; wd; wd &= wd - 1u, ++idx)
                if (idx < kk)
                    kcols[idx] = 32 * w + __ffs(wd) - 1;
        }
        for (int t = threadIdx.x; t < kk; t += kOutThreads) {
            const float sj = __ldg(a.fp8_scale + t);
            krcp[t] = (sj == 0.0f) ? 0.0f : __frcp_rn(sj);
            ksj[t] = sj;
        }
        for (int c = threadIdx.x; c < 128; c += kOutThreads)
            e4m3v[c] = c < 0x7F ? e4m3_value((uint32_t)c) : 0.0f;
        if (fast == 2) {
            // one bitmap word (32 columns) per thread: 16 image words
            for (int w = threadIdx.x; w < nwords; w += kOutThreads) {
                const uint32_t wd = __ldg(a.bitmap + w);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    keep[16 * w + j] = (((wd >> (2 * j)) & 1u) ? 0u : 0x0000FFFFu) |
                                       (((wd >> (2 * j + 1)) & 1u) ? 0u : 0xFFFF0000u);
            }
        }
        __syncthreads();
    }
    float s_g = 0.0f, inv6 = 0.0f;
    if (FMT == NVFP4) {
        s_g = outer_scale(*a.amax);
        inv6 = nv_inv6(s_g);
        nv_tables_fill(tab, s_g);
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.codes)
            a.tscale[0] = s_g;
    }
    __syncthreads();
    const PhiloxKey &key = a.key;
    const bool xhat32 = (reinterpret_cast<uintptr_t>(a.xhat) & 31u) == 0;
    const int64_t bpr = cols / B;
    const int64_t nblk = rows * bpr;
    const int lane = threadIdx.x & 31;
    const int wbase = threadIdx.x & ~31;
    // (row, block column) of this thread's block: one division for the first,
    // then each grid step advances them with a carry
    const int64_t gstep = (int64_t)gridDim.x * kOutThreads;
    const int64_t dr = gstep / bpr, dcb = gstep - dr * bpr;
    int64_t rn = ((int64_t)blockIdx.x * kOutThreads + threadIdx.x) / bpr;
    int64_t cbn = (int64_t)blockIdx.x * kOutThreads + threadIdx.x - rn * bpr;
    for (int64_t base = (int64_t)blockIdx.x * kOutThreads; base < nblk; base += gstep) {
        const int64_t blk = base + threadIdx.x;
        const bool valid = blk < nblk;
        const int64_t r = rn, c0 = cbn * B;
        cbn += dcb;
        rn += dr;
        if (cbn >= bpr) {
            cbn -= bpr;
            ++rn;
        }
        float v[B];
        uint32_t ret = 0u;
        float am = 0.0f;
        if (sizeof(T) == 2 && fast == 2) {
            // BF16 with the keep-mask image: retained elements zeroed in the
            // raw words, the amax from a tree over the packed pairs
            constexpr int NV = B / 8;
            uint4 raw[NV];
            const char *src = (const char *)a.x + blk * B * (int64_t)sizeof(T);
            const uint4 *km = reinterpret_cast<const uint4 *>(keep + c0 / 2);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                raw[k] = valid ? ld16(src + 16 * k) : make_uint4(0, 0, 0, 0);
                const uint4 m = km[k];
                raw[k].x &= m.x;
                raw[k].y &= m.y;
                raw[k].z &= m.z;
                raw[k].w &= m.w;
            }
            am = block_amax<T, B>(raw);
#pragma unroll
            for (int k = 0; k < NV; ++k)
                unpack16<T>(raw[k], v + 8 * k);
        } else {
            float x[B];
            if (valid)
                load_block<T, B>((const char *)a.x + blk * B * (int64_t)sizeof(T), x);
            else
#pragma unroll
                for (int i = 0; i < B; ++i)
                    x[i] = 0.0f;
            const uint32_t word = valid ? __ldg(a.bitmap + (c0 >> 5)) : 0u;
            ret = (B == 32) ? word : ((word >> (c0 & 31)) & 0xFFFFu);
#pragma unroll
            for (int i = 0; i < B; ++i)
                v[i] = ((ret >> i) & 1u) ? 0.0f : x[i];
#pragma unroll
            for (int i = 0; i < B; ++i)
                am = fmaxf(am, fabsf(v[i]));
        }
        float s_o = s_g, inv6b = inv6;
        if (FMT == NV2L) {
            s_o = outer_scale(group_max<8>(am));
            inv6b = nv_inv6(s_o);
        }
        const Scale sc = block_scale<FMT>(am, s_o, inv6b, &tab);
        uint32_t q[B / 8];
        encode_block<B, RND>(v, sc, key, (uint64_t)blk * B, 0u, a.offset, q);
        uint32_t mask = block_mask<B>(v, sc.lim);
        if (valid) {
            if (a.codes) {
                if (B == 16)
                    *reinterpret_cast<uint2 *>(a.codes + blk * 8) = make_uint2(q[0], q[1]);
                else
                    *reinterpret_cast<uint4 *>(a.codes + blk * 16) =
                        make_uint4(q[0], q[1], q[2], q[3]);
                a.scales[blk] = (uint8_t)sc.code;
                if (FMT == NV2L && (lane & 7) == 0)
                    a.tscale[blk >> 3] = s_o;
            }
            if (a.xhat && a.xhat_bf16 && xhat32) {
                // whole 32-byte sectors: one store per 16 values
#pragma unroll
                for (int w = 0; w < B / 8; w += 2)
                    st32((char *)a.xhat + (blk * B + w * 8) * 2, xhat8_bf16(q[w], sc.s_eff),
                         xhat8_bf16(q[w + 1], sc.s_eff));
            } else if (a.xhat) {
#pragma unroll
                for (int w = 0; w < B / 8; ++w) {
                    float h[8];
                    e2m1_decode8(q[w], h);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const float2 p = mul2(make_float2(h[i], h[i + 1]),
                                              make_float2(sc.s_eff, sc.s_eff));
                        h[i] = p.x;
                        h[i + 1] = p.y;
                    }
                    if (a.xhat_bf16)
                        *reinterpret_cast<uint4 *>((char *)a.xhat + (blk * B + w * 8) * 2) =
                            make_uint4(bf16x2_rn(h[0], h[1]), bf16x2_rn(h[2], h[3]),
                                       bf16x2_rn(h[4], h[5]), bf16x2_rn(h[6], h[7]));
                    else if (xhat32) {
                        st32((char *)a.xhat + (blk * B + w * 8) * 4,
                             make_uint4(__float_as_uint(h[0]), __float_as_uint(h[1]),
                                        __float_as_uint(h[2]), __float_as_uint(h[3])),
                             make_uint4(__float_as_uint(h[4]), __float_as_uint(h[5]),
                                        __float_as_uint(h[6]), __float_as_uint(h[7])));
                    } else {
                        float4 *dst =
                            reinterpret_cast<float4 *>((char *)a.xhat + (blk * B + w * 8) * 4);
                        dst[0] = make_float4(h[0], h[1], h[2], h[3]);
                        dst[1] = make_float4(h[4], h[5], h[6], h[7]);
                    }
                }
            }
        }
        // ---- the warp's kept elements, one per lane
        if (fast) {
            // The warp's 32 blocks are one span of 32 B columns of one row (a row
            // holds a whole number of spans): its retained elements are the
            // slice [s0, s1) of the sorted column list, their ranks s0 .. s1 - 1.
            mstage[threadIdx.x] = mask;
            __syncwarp();  // also orders the owners' xhat stores before the patches
            const int64_t blk0 = base + wbase;
            if (blk0 < nblk) {  // warp-uniform: the span is all in or all out
                // the span lies in this thread's row, and lane 0's block starts it
                const int64_t r_w = r;
                const int64_t cspan = c0 - (int64_t)lane * B;
                const int64_t cend = cspan + 32 * B;
                const int s0 = pre[cspan >> 5];
                int s1 = cend >= cols ? kk : pre[cend >> 5];
                s1 = s1 < kk ? s1 : kk;
                // the span's row, with 32-bit offsets inside it
                const T *xrow = reinterpret_cast<const T *>(a.x) + r_w * cols + cspan;
                uint8_t *fp8row = a.fp8 ? a.fp8 + r_w * a.k : nullptr;
                char *xhrow = a.xhat ? (char *)a.xhat + (r_w * cols + cspan) * (a.xhat_bf16 ? 2 : 4)
                                     : nullptr;
                const int c0s = (int)cspan;
                for (int t = s0 + lane; t < s1; t += 32) {
                    const int off = kcols[t] - c0s;  // column inside the span
                    const int owner = off / B, i = off % B;
                    const float xv = ld_scalar<T>(xrow, off);
                    const float y = __fmul_rn(xv, krcp[t]);
                    const uint32_t code =
                        e4m3_rn_sat(fabsf(y)) | ((__float_as_uint(y) >> 24) & 0x80u);
                    const float sj = ksj[t];
                    if (fp8row)
                        fp8row[t] = (uint8_t)code;
                    if (xhrow) {
                        const float m = __fmul_rn(e4m3v[code & 0x7Fu], sj);
                        const float h = (code & 0x80u) ? -m : m;
                        if (a.xhat_bf16)
                            reinterpret_cast<unsigned short *>(xhrow)[off] =
                                (unsigned short)(bf16x2_rn(h, 0.0f) & 0xFFFFu);
                        else
                            reinterpret_cast<float *>(xhrow)[off] = h;
                    }
                    // the owner's FP4 pass set this bit (a zeroed element is never
                    // clipped); clear it where the FP8 value clips
                    if (!(fabsf(xv) <= __fmul_rn(448.0f, sj)))
                        atomicAnd(&mstage[wbase + owner], ~(1u << i));
                }
            }
            __syncwarp();
            mask = mstage[threadIdx.x];
            if (valid && a.mask) {
                if (B == 16)
                    reinterpret_cast<uint16_t *>(a.mask)[blk] = (uint16_t)mask;
                else
                    reinterpret_cast<uint32_t *>(a.mask)[blk] = mask;
            }
            continue;
        }
        const uint32_t cnt = valid ? (uint32_t)__popc(ret) : 0u;
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += t;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        if (total) {  // warp-uniform
            mstage[threadIdx.x] = mask;
            __syncwarp();  // also orders the owners' xhat stores before the patches
            for (uint32_t t0 = 0; t0 < total; t0 += 32) {
                const uint32_t t = t0 + (uint32_t)lane;
                int pos = 0;  // the first lane whose inclusive count exceeds t
#pragma unroll
                for (int step = 16; step >= 1; step >>= 1) {
                    const uint32_t cv = __shfl_sync(0xFFFFFFFFu, incl, pos + step - 1);
                    if (cv <= t)
                        pos += step;
                }
                const uint32_t ret_o = __shfl_sync(0xFFFFFFFFu, ret, pos);
                const uint32_t ex_o = __shfl_sync(0xFFFFFFFFu, incl - cnt, pos);
                const int64_t r_o = __shfl_sync(0xFFFFFFFFu, r, pos);
                const int64_t c0_o = __shfl_sync(0xFFFFFFFFu, c0, pos);
                if (t >= total)
                    continue;
                uint32_t rest = ret_o;  // drop the owner's first t - ex_o kept positions
                for (uint32_t n = t - ex_o; n > 0; --n)
                    rest &= rest - 1u;
                const int i = __ffs(rest) - 1;
                const int64_t c = c0_o + i;
                const uint32_t wd = __ldg(a.bitmap + (c >> 5));
                const int j = pre[c >> 5] + __popc(wd & ((1u << (c & 31)) - 1u));
                if (j >= a.k)  // more bits set than k: outside the contract, stay in bounds
                    continue;
                const int64_t e = r_o * cols + c;
                const float xv = ld_scalar<T>(a.x, e);
                const float sj = __ldg(a.fp8_scale + j);
                const float rcp = (sj == 0.0f) ? 0.0f : __frcp_rn(sj);
                const float y = __fmul_rn(xv, rcp);
                const uint32_t code = e4m3_rn_sat(fabsf(y)) | ((__float_as_uint(y) >> 24) & 0x80u);
                if (a.fp8)
                    a.fp8[r_o * a.k + j] = (uint8_t)code;
                if (a.xhat) {
                    const float m = __fmul_rn(e4m3_value(code & 0x7Fu), sj);
                    const float h = (code & 0x80u) ? -m : m;
                    if (a.xhat_bf16)
                        reinterpret_cast<unsigned short *>(a.xhat)[e] =
                            (unsigned short)(bf16x2_rn(h, 0.0f) & 0xFFFFu);
                    else
                        reinterpret_cast<float *>(a.xhat)[e] = h;
                }
                const uint32_t bit = 1u << i;
                if (fabsf(xv) <= __fmul_rn(448.0f, sj))
                    atomicOr(&mstage[wbase + (int)pos], bit);
                else
                    atomicAnd(&mstage[wbase + (int)pos], ~bit);
            }
            __syncwarp();
            mask = mstage[threadIdx.x];
        }
        if (valid && a.mask) {
            if (B == 16)
                reinterpret_cast<uint16_t *>(a.mask)[blk] = (uint16_t)mask;
            else
                reinterpret_cast<uint32_t *>(a.mask)[blk] = mask;
        }
    }
}

// ------------------------------------------------------------------ launchers
static int grid_cap(int64_t need, int per_sm)
{
    const int64_t cap = (int64_t)sm_count() * per_sm;
    return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

cudaError_t launch_channel_amax(const void *x, int bf16, int64_t rows, int64_t cols,
                                float *amax, cudaStream_t s)
{
    if (rows == 0 || cols == 0)
        return cudaSuccess;
    const int E = bf16 ? 8 : 4;
    const int64_t gx = (cols / E + kOutThreads - 1) / kOutThreads;
    // enough row stripes for about eight CTAs per SM, at least 16 rows each
    int64_t gy = ((int64_t)sm_count() * 8 + gx - 1) / gx;
    const int64_t max_gy = (rows + 15) / 16;
    gy = gy < max_gy ? gy : max_gy;
    gy = gy < 65535 ? gy : 65535;
    const int64_t rows_per = (rows + gy - 1) / gy;
    gy = (rows + rows_per - 1) / rows_per;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (bf16)
        channel_amax_kernel<__nv_bfloat16><<<grid, kOutThreads, 0, s>>>(x, rows, cols, rows_per,
                                                                        (unsigned *)amax);
    else
        channel_amax_kernel<float><<<grid, kOutThreads, 0, s>>>(x, rows, cols, rows_per,
                                                                (unsigned *)amax);
    return cudaGetLastError();
}

cudaError_t launch_select(const float *amax, int cols, int k, int32_t *idx, uint32_t *bitmap,
                          float *fp8_scale, cudaStream_t s)
{
    select_kernel<<<1, kSelThreads, 0, s>>>(amax, cols, k, idx, bitmap, fp8_scale);
    return cudaGetLastError();
}

cudaError_t launch_masked_amax(const void *x, int bf16, int64_t rows, int64_t cols,
                               const uint32_t *bitmap, float *out, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), s);
    if (e != cudaSuccess || rows == 0 || cols == 0)
        return e;
    const int E = bf16 ? 8 : 4;
    const int64_t gx = (cols / E + kOutThreads - 1) / kOutThreads;
    // enough row stripes for about eight CTAs per SM, at least 16 rows each
    int64_t gy = ((int64_t)sm_count() * 8 + gx - 1) / gx;
    const int64_t max_gy = (rows + 15) / 16;
    gy = gy < max_gy ? gy : max_gy;
    gy = gy < 65535 ? gy : 65535;
    const int64_t rows_per = (rows + gy - 1) / gy;
    gy = (rows + rows_per - 1) / rows_per;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (bf16)
        masked_amax_kernel<__nv_bfloat16><<<grid, kOutThreads, 0, s>>>(x, rows, cols, rows_per,
                                                                       bitmap, (unsigned *)out);
    else
        masked_amax_kernel<float><<<grid, kOutThreads, 0, s>>>(x, rows, cols, rows_per, bitmap,
                                                               (unsigned *)out);
    return cudaGetLastError();
}

template <typename T, int FMT, int RND>
static cudaError_t outlier_go(const OutlierArgs &a, cudaStream_t s)
{
    constexpr int B = FmtInfo<FMT>::B;
    const int64_t nblk = a.rows * (a.cols / B);
    if (nblk == 0)
        return cudaSuccess;
    // the sorted-list path: the list fits in shared memory and every row is a
    // whole number of 32-block warp spans
    int fast = a.k > 0 && a.k <= kFastKept && (a.cols / B) % 32 == 0;
    // BF16 rows of up to 16384 columns also get the keep-mask image: 16 words
    // per bitmap word (cols is a multiple of 512 on this path, so the bitmap
    // words are whole)
    if (fast && sizeof(T) == 2 && a.cols <= kKeepImageCols)
        fast = 2;
    const size_t smem = outlier_smem(a.cols, a.k, fast);
    // the kernel's static shared memory counts against the default 48 KB too,
    // so the dynamic size is declared for every launch
    {
        const cudaError_t e = cudaFuncSetAttribute(outlier_row_kernel<T, FMT, RND>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    return launch_dependent(outlier_row_kernel<T, FMT, RND>,
                            dim3(grid_cap((nblk + kOutThreads - 1) / kOutThreads, 8)),
                            dim3(kOutThreads), smem, s, a, fast);
}

template <typename T>
static cudaError_t outlier_fmt(const OutlierArgs &a, int fmt, int rnd, cudaStream_t s)
{
    switch (fmt * 2 + rnd) {
    case NVFP4 * 2 + RNE: return outlier_go<T, NVFP4, RNE>(a, s);
    case NVFP4 * 2 + SR: return outlier_go<T, NVFP4, SR>(a, s);
    case MXFP4 * 2 + RNE: return outlier_go<T, MXFP4, RNE>(a, s);
    case MXFP4 * 2 + SR: return outlier_go<T, MXFP4, SR>(a, s);
    case NV2L * 2 + RNE: return outlier_go<T, NV2L, RNE>(a, s);
    default: return outlier_go<T, NV2L, SR>(a, s);
    }
}

cudaError_t launch_outlier_quant(const OutlierArgs &a, int bf16, int fmt, int rnd, cudaStream_t s)
{
    return bf16 ? outlier_fmt<__nv_bfloat16>(a, fmt, rnd, s) : outlier_fmt<float>(a, fmt, rnd, s);
}

}  // namespace fqk
