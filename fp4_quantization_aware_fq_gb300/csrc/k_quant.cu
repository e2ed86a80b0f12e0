// k_quant.cu -- tensor amax, row-wise quantization and the tiled row +
// column-wise quantization kernels.
//
// Row-wise ("Resumo Técnico: TetraJet-v2" §2A, 1x16 groups; MXFP4 1x32 as
// named on "Aprimorando gpt-oss ...", "O que há de novo"): each thread owns
// one 16-byte vector of the input (8 BF16 or 4 FP32 values); the lanes that
// share a block combine their partial amax with warp shuffles, derive the
// scale in registers, and write packed codes, scales, the fake-quantized
// values and the STE mask with coalesced stores.
//
// Column-wise (§2A, the transposed 1x16 groups of the backward pass): a CTA
// stages a tile of x in shared memory while doing the row-wise pass on it,
// then quantizes 16x1 column blocks out of shared memory and writes the
// transposed codes through a shared-memory staging buffer.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kThreads = 256;
// CTAs per SM the register allocation must allow, measured: row kernels 4
// (at most 64 registers; the double-block SR call 3-4% faster despite a few
// spills), BF16 tile kernels 3 (80 registers; the Hadamard-transformed SR call
// 2% faster, the NVFP4 row + column call 1.5%).  The FP32 tile kernels, whose
// tiles need far more registers, are left free.
constexpr int kRowMinCtas = 4;
template <typename T, int FMT>
constexpr int tile_min_ctas()
{
    return sizeof(T) == 2 ? 3 : 1;
}

// ------------------------------------------------------------------ amax
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_kernel(const void *__restrict__ x, int64_t nch,
                                                        unsigned *__restrict__ out)
{
    constexpr int E = VecInfo<T>::E;
    constexpr int U = 4;
    float m = 0.0f;
    const int64_t stride = (int64_t)gridDim.x * kThreads * U;
    for (int64_t base = (int64_t)blockIdx.x * kThreads * U; base < nch; base += stride) {
        uint4 raw[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t ch = base + k * kThreads + threadIdx.x;
            raw[k] = ch < nch ? ld16((const char *)x + ch * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float v[E];
            unpack16<T>(raw[k], v);
#pragma unroll
            for (int i = 0; i < E; ++i)
                m = fmaxf(m, fabsf(v[i]));
        }
    }
    m = group_max<32>(m);
    __shared__ float wm[kThreads / 32];
    if ((threadIdx.x & 31) == 0)
        wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = wm[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w)
            b = fmaxf(b, wm[w]);
        atomicMax(out, __float_as_uint(b));  // non-negative floats order like their bits
    }
}

// ------------------------------------------------------------------ row-wise core
// Outputs of the row-wise pass (any pointer may be NULL: not written).
struct RowOut {
    uint8_t *codes;
    uint8_t *scales;
    float *tscale;
    void *xhat;
    int xhat_bf16;
    uint8_t *mask;
};

// Quantize one row-wise block of B values held by this thread.  `blk` is the
// flat block index in the tensor (flat element index blk * B).  For the double
// block, the 8 inner blocks of an outer block sit on 8 consecutive lanes, and
// all 32 lanes of the warp must call this together.
template <int FMT, int RND>
__device__ __forceinline__ void row_block(float *v, int64_t blk, bool valid, float s_g,
                                          float inv6, const NvTables *tab, const RowOut &o,
                                          const PhiloxKey &key, uint32_t offset,
                                          uint32_t stream_id, bool rht, uint32_t signs)
{
    constexpr int B = FmtInfo<FMT>::B;
    if (FMT != NVFP4 && rht) {
#pragma unroll
        for (int j = 0; j < B / 16; ++j)
            rht16(v + 16 * j, signs);
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < B; ++i)
        am = fmaxf(am, fabsf(v[i]));
    float s_o = s_g;
    if (FMT == NV2L) {
        s_o = outer_scale(group_max<8>(am));
        inv6 = nv_inv6(s_o);
    }
    const Scale sc = block_scale<FMT>(am, s_o, inv6, tab);
    uint32_t q[B / 8];
    encode_block<B, RND>(v, sc, key, (uint64_t)blk * B, stream_id, offset, q);
    if (!valid)
        return;
    const int lane = threadIdx.x & 31;
    if (o.codes) {
        if (B == 16)
            *reinterpret_cast<uint2 *>(o.codes + blk * 8) = make_uint2(q[0], q[1]);
        else
            *reinterpret_cast<uint4 *>(o.codes + blk * 16) = make_uint4(q[0], q[1], q[2], q[3]);
        o.scales[blk] = (uint8_t)sc.code;
        if (FMT == NV2L && (lane & 7) == 0)
            o.tscale[blk >> 3] = s_o;
    }
    if (o.xhat) {
#pragma unroll
        for (int w = 0; w < B / 8; ++w) {
            float xh[8];
            e2m1_decode8(q[w], xh);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                xh[i] = __fmul_rn(xh[i], sc.s_eff);
            if (o.xhat_bf16) {
                *reinterpret_cast<uint4 *>((char *)o.xhat + (blk * B + w * 8) * 2) =
                    make_uint4(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]),
                               bf16x2_rn(xh[4], xh[5]), bf16x2_rn(xh[6], xh[7]));
            } else {
                float4 *dst = reinterpret_cast<float4 *>((char *)o.xhat + (blk * B + w * 8) * 4);
                dst[0] = make_float4(xh[0], xh[1], xh[2], xh[3]);
                dst[1] = make_float4(xh[4], xh[5], xh[6], xh[7]);
            }
        }
    }
    if (o.mask) {
        const uint32_t mask = block_mask<B>(v, sc.lim);
        if (B == 16)
            reinterpret_cast<uint16_t *>(o.mask)[blk] = (uint16_t)mask;
        else
            reinterpret_cast<uint32_t *>(o.mask)[blk] = mask;
    }
}

// One thread per block; each iteration a thread holds BPT blocks' loads in
// flight (about 64 bytes).
template <typename T, int FMT, int RND>
__global__ void __launch_bounds__(kThreads, kRowMinCtas) row_kernel(RowArgs a)
{
    constexpr int B = FmtInfo<FMT>::B;
    constexpr int BPT = (B * sizeof(T) >= 64) ? 1 : 2;
    const int64_t nblk = a.n / B;
    __shared__ NvTables tab;
    float s_g = 0.0f, inv6 = 0.0f;
    if (FMT == NVFP4) {
        s_g = outer_scale(*a.amax);
        inv6 = nv_inv6(s_g);
        nv_tables_fill(tab, s_g);
        __syncthreads();
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.tscale)
            a.tscale[0] = s_g;
    }
    const RowOut o{a.codes, a.scales, a.tscale, a.xhat, a.xhat_bf16, a.mask};
    const PhiloxKey key = philox_key(a.seed);
    const bool rht = a.rht_seed != 0;
    const uint32_t signs = rht ? rht_signs(a.rht_seed, a.offset) : 0u;
    const int64_t stride = (int64_t)gridDim.x * kThreads * BPT;
    for (int64_t base = (int64_t)blockIdx.x * kThreads * BPT; base < nblk; base += stride) {
        float v[BPT][B];
#pragma unroll
        for (int k = 0; k < BPT; ++k) {
            const int64_t blk = base + k * kThreads + threadIdx.x;
            if (blk < nblk)
                load_block<T, B>((const char *)a.x + blk * B * (int64_t)sizeof(T), v[k]);
            else
#pragma unroll
                for (int i = 0; i < B; ++i)
                    v[k][i] = 0.0f;
        }
#pragma unroll
        for (int k = 0; k < BPT; ++k) {
            const int64_t blk = base + k * kThreads + threadIdx.x;
            row_block<FMT, RND>(v[k], blk, blk < nblk, s_g, inv6, &tab, o, key, a.offset,
                                a.stream_id, rht, signs);
        }
    }
}

// ------------------------------------------------------------------ tiled row + column
template <int FMT>
struct TileShape {
    static constexpr int TR = 128;                       // tile rows
    static constexpr int TC = (FMT == NV2L) ? 128 : 64;  // tile cols
    static constexpr int BC = FmtInfo<FMT>::B;           // column block (rows)
    static constexpr int CP = TR / 2 + 8;                // staged code bytes per column (padded)
};

template <typename T, int FMT>
constexpr size_t tile_smem_bytes()
{
    using S = TileShape<FMT>;
    return (size_t)S::TR * S::TC * sizeof(T)          // x tile
           + (size_t)S::TC * S::CP                    // staged column codes
           + (size_t)S::TC * (S::TR / S::BC)          // staged column scales
           + (FMT == NV2L ? (size_t)S::TC * (S::TR / S::BC) * 4 : 0);  // inner amax
}

template <typename T, int FMT, int RND>
__global__ void __launch_bounds__(kThreads, tile_min_ctas<T, FMT>()) tile_kernel(TileArgs a)
{
    using S = TileShape<FMT>;
    constexpr int E = VecInfo<T>::E;
    constexpr int TR = S::TR, TC = S::TC, BC = S::BC, CP = S::CP;
    constexpr int BR = FmtInfo<FMT>::B;  // row block
    constexpr int RBPR = TC / BR;         // row blocks per tile row
    constexpr int NRB = TR / BC;          // column blocks per tile column
    extern __shared__ __align__(16) unsigned char smem[];
    T *tile = reinterpret_cast<T *>(smem);
    uint8_t *ccs = smem + (size_t)TR * TC * sizeof(T);   // [TC][CP]
    uint8_t *css = ccs + (size_t)TC * CP;                // [TC][NRB]
    float *am16 = reinterpret_cast<float *>(css + (size_t)TC * NRB);  // [NRB][TC]

    const int64_t rows = a.rows, cols = a.cols;
    __shared__ NvTables tab;
    float s_g = 0.0f, inv6 = 0.0f;
    if (FMT == NVFP4) {
        s_g = outer_scale(*a.amax);
        inv6 = nv_inv6(s_g);
        nv_tables_fill(tab, s_g);
        __syncthreads();
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            if (a.ctscale)
                a.ctscale[0] = s_g;
            if (a.do_row && a.rtscale)
                a.rtscale[0] = s_g;
        }
    }
    const RowOut o{a.rcodes, a.rscales, a.rtscale, a.xhat, a.xhat_bf16, a.mask};
    const PhiloxKey key = philox_key(a.seed);
    const bool rht = a.rht_seed != 0;
    const uint32_t signs = rht ? rht_signs(a.rht_seed, a.offset) : 0u;
    const int64_t ntc = (cols + TC - 1) / TC;
    const int64_t ntiles = ntc * ((rows + TR - 1) / TR);

    // Each thread owns RPT row blocks of a tile.  The loads of the next tile
    // are issued before the current tile is processed, so they overlap its
    // column pass and write-out.
    constexpr int RPT = (TR * RBPR + kThreads - 1) / kThreads;
    uint4 nxt[RPT][BR / E];
    auto load_tile = [&](int64_t id) {
        const int64_t lr0 = (id / ntc) * TR, lc0 = (id % ntc) * TC;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int t = threadIdx.x + j * kThreads;
            const int tr = t / RBPR, tb = t % RBPR;
            const int64_t gr = lr0 + tr, gc = lc0 + (int64_t)tb * BR;
            const bool valid = t < TR * RBPR && gr < rows && gc < cols;
#pragma unroll
            for (int k = 0; k < BR / E; ++k)
                nxt[j][k] = valid ? ld16((const char *)a.x +
                                         ((gr * cols + gc) + k * E) * (int64_t)sizeof(T))
                                  : make_uint4(0, 0, 0, 0);
        }
    };
    if ((int64_t)blockIdx.x < ntiles)
        load_tile(blockIdx.x);

    // Persistent CTAs walk the tiles in row-major order.
    for (int64_t tile_id = blockIdx.x; tile_id < ntiles; tile_id += gridDim.x) {
    const int64_t r0 = (tile_id / ntc) * TR;
    const int64_t c0 = (tile_id % ntc) * TC;
    uint4 cur[RPT][BR / E];
#pragma unroll
    for (int j = 0; j < RPT; ++j)
#pragma unroll
        for (int k = 0; k < BR / E; ++k)
            cur[j][k] = nxt[j][k];
    if (tile_id + gridDim.x < ntiles)
        load_tile(tile_id + gridDim.x);

    // Phase 1: stage the tile's row blocks in shared memory and, when asked,
    // run the row-wise pass on them.
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int t = threadIdx.x + j * kThreads;
        if (RPT * kThreads > TR * RBPR && t >= TR * RBPR)
            break;
        const int tr = t / RBPR, tb = t % RBPR;
        const int64_t gr = r0 + tr, gc = c0 + (int64_t)tb * BR;
        const bool valid = gr < rows && gc < cols;
        float v[BR];
#pragma unroll
        for (int k = 0; k < BR / E; ++k) {
            *reinterpret_cast<uint4 *>(tile + tr * TC + tb * BR + k * E) = cur[j][k];
            unpack16<T>(cur[j][k], v + k * E);
        }
        if (a.do_row)
            row_block<FMT, RND>(v, (gr * cols + gc) / BR, valid, s_g, inv6, &tab, o, key,
                                a.offset, 0u, rht, signs);
    }
    __syncthreads();

    // Phase 2: column blocks (BC rows x 1 column) out of shared memory.  BF16
    // NVFP4 tiles are read two columns at a time (one 32-bit word per row).
    const uint32_t *tile32 = reinterpret_cast<const uint32_t *>(tile);
    auto col_amax = [&](float *w) {  // double block: inner amax for the outer scale
        if (rht) {
#pragma unroll
            for (int j = 0; j < BC / 16; ++j)
                rht16(w + 16 * j, signs);
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < BC; ++i)
            m = fmaxf(m, fabsf(w[i]));
        return m;
    };
    if (FMT == NV2L) {
        for (int task = threadIdx.x; task < TC * NRB; task += kThreads) {
            const int c = task % TC, rb = task / TC;
            float w[BC];
#pragma unroll
            for (int i = 0; i < BC; ++i)
                w[i] = static_cast<float>(tile[(rb * BC + i) * TC + c]);
            am16[rb * TC + c] = col_amax(w);
        }
        __syncthreads();
    }
    // quantize column block (c, rb) of the tile, held in v, into the staging buffers
    auto col_quant = [&](int c, int rb, float *v) {
        const int64_t gc = c0 + c, gr0 = r0 + (int64_t)rb * BC;
        if (FMT != NVFP4 && rht) {
#pragma unroll
            for (int j = 0; j < BC / 16; ++j)
                rht16(v + 16 * j, signs);
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < BC; ++i)
            m = fmaxf(m, fabsf(v[i]));
        float s_o = s_g, inv6c = inv6;
        if (FMT == NV2L) {
            float mo = 0.0f;
#pragma unroll
            for (int j = 0; j < NRB; ++j)
                mo = fmaxf(mo, am16[j * TC + c]);
            s_o = outer_scale(mo);
            inv6c = nv_inv6(s_o);
            if (rb == 0)
                a.ctscale[gc * (rows / 128) + r0 / 128] = s_o;
        }
        const Scale sc = block_scale<FMT>(m, s_o, inv6c, &tab);
        uint32_t q[BC / 8];
        // flat index in X^T of the block's first element
        encode_block<BC, RND>(v, sc, key, (uint64_t)gc * (uint64_t)rows + (uint64_t)gr0, 1u,
                              a.offset, q);
        uint32_t *dst = reinterpret_cast<uint32_t *>(ccs + c * CP + rb * (BC / 2));
#pragma unroll
        for (int w = 0; w < BC / 8; ++w)
            dst[w] = q[w];
        css[c * NRB + rb] = (uint8_t)sc.code;
    };
    if constexpr (sizeof(T) == 2 && FMT == NVFP4) {
        // cols is a multiple of the row block, hence even: a pair is all in or out
        for (int task = threadIdx.x; task < (TC / 2) * NRB; task += kThreads) {
            const int c = 2 * (task % (TC / 2)), rb = task / (TC / 2);
            if (c0 + c >= cols || r0 + (int64_t)rb * BC >= rows)
                continue;
            uint32_t wd[BC];
            float v[BC];
#pragma unroll
            for (int i = 0; i < BC; ++i)
                wd[i] = tile32[((rb * BC + i) * TC + c) / 2];
#pragma unroll
            for (int i = 0; i < BC; ++i)
                v[i] = __uint_as_float(wd[i] << 16);
            col_quant(c, rb, v);
#pragma unroll
            for (int i = 0; i < BC; ++i)
                v[i] = __uint_as_float(wd[i] & 0xFFFF0000u);
            col_quant(c + 1, rb, v);
        }
    } else {
        for (int task = threadIdx.x; task < TC * NRB; task += kThreads) {
            const int c = task % TC, rb = task / TC;
            if (c0 + c >= cols || r0 + (int64_t)rb * BC >= rows)
                continue;
            float v[BC];
#pragma unroll
            for (int i = 0; i < BC; ++i)
                v[i] = static_cast<float>(tile[(rb * BC + i) * TC + c]);
            col_quant(c, rb, v);
        }
    }
    __syncthreads();

    // Phase 3: write the staged column outputs (rows of X^T).
    constexpr int U8 = TR / 16;  // 8-byte units of codes per tile column
    for (int u = threadIdx.x; u < TC * U8; u += kThreads) {
        const int c = u / U8, j = u % U8;
        const int64_t gc = c0 + c, gr = r0 + (int64_t)j * 16;
        if (gc < cols && gr < rows)
            *reinterpret_cast<uint2 *>(a.ccodes + gc * (rows / 2) + gr / 2) =
                *reinterpret_cast<const uint2 *>(ccs + c * CP + j * 8);
    }
    for (int u = threadIdx.x; u < TC * NRB; u += kThreads) {
        const int c = u / NRB, j = u % NRB;
        const int64_t gc = c0 + c, gr = r0 + (int64_t)j * BC;
        if (gc < cols && gr < rows)
            a.cscales[gc * (rows / BC) + gr / BC] = css[c * NRB + j];
    }
    __syncthreads();  // the next tile overwrites the tile and staging buffers
    }
}

// ------------------------------------------------------------------ launchers
int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 132;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 132;
    return n;
}

static int persistent_grid(int64_t work_items, int per_cta, int ctas_per_sm)
{
    const int64_t need = (work_items + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)sm_count() * ctas_per_sm;
    return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

cudaError_t launch_amax(const void *x, int bf16, int64_t n, float *out, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), s);
    if (e != cudaSuccess)
        return e;
    if (n == 0)
        return cudaSuccess;
    const int E = bf16 ? 8 : 4;
    const int64_t nch = n / E;
    const int grid = persistent_grid(nch, kThreads * 4, 4);
    if (bf16)
        amax_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(x, nch, (unsigned *)out);
    else
        amax_kernel<float><<<grid, kThreads, 0, s>>>(x, nch, (unsigned *)out);
    return cudaGetLastError();
}

template <typename T, int FMT, int RND>
static cudaError_t row_go(const RowArgs &a, cudaStream_t s)
{
    constexpr int B = FmtInfo<FMT>::B;
    constexpr int BPT = (B * sizeof(T) >= 64) ? 1 : 2;
    const int64_t nblk = a.n / B;
    if (nblk == 0)
        return cudaSuccess;
    const int grid = persistent_grid(nblk, kThreads * BPT, 8);
    row_kernel<T, FMT, RND><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t row_fmt(const RowArgs &a, int fmt, int rnd, cudaStream_t s)
{
    switch (fmt * 2 + rnd) {
    case NVFP4 * 2 + RNE: return row_go<T, NVFP4, RNE>(a, s);
    case NVFP4 * 2 + SR: return row_go<T, NVFP4, SR>(a, s);
    case MXFP4 * 2 + RNE: return row_go<T, MXFP4, RNE>(a, s);
    case MXFP4 * 2 + SR: return row_go<T, MXFP4, SR>(a, s);
    case NV2L * 2 + RNE: return row_go<T, NV2L, RNE>(a, s);
    default: return row_go<T, NV2L, SR>(a, s);
    }
}

cudaError_t launch_row(const RowArgs &a, int bf16, int fmt, int rnd, cudaStream_t s)
{
    return bf16 ? row_fmt<__nv_bfloat16>(a, fmt, rnd, s) : row_fmt<float>(a, fmt, rnd, s);
}

template <typename T, int FMT, int RND>
static cudaError_t tile_go(const TileArgs &a, cudaStream_t s)
{
    using S = TileShape<FMT>;
    if (a.rows == 0 || a.cols == 0)
        return cudaSuccess;
    constexpr size_t smem = tile_smem_bytes<T, FMT>();
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(tile_kernel<T, FMT, RND>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int64_t ntiles = ((a.cols + S::TC - 1) / S::TC) * ((a.rows + S::TR - 1) / S::TR);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tile_kernel<T, FMT, RND>, kThreads,
                                                      smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const unsigned grid = (unsigned)(ntiles < cap ? ntiles : cap);
    tile_kernel<T, FMT, RND><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t tile_fmt(const TileArgs &a, int fmt, int rnd, cudaStream_t s)
{
    switch (fmt * 2 + rnd) {
    case NVFP4 * 2 + RNE: return tile_go<T, NVFP4, RNE>(a, s);
    case NVFP4 * 2 + SR: return tile_go<T, NVFP4, SR>(a, s);
    case MXFP4 * 2 + RNE: return tile_go<T, MXFP4, RNE>(a, s);
    case MXFP4 * 2 + SR: return tile_go<T, MXFP4, SR>(a, s);
    case NV2L * 2 + RNE: return tile_go<T, NV2L, RNE>(a, s);
    default: return tile_go<T, NV2L, SR>(a, s);
    }
}

cudaError_t launch_tile(const TileArgs &a, int bf16, int fmt, int rnd, cudaStream_t s)
{
    return bf16 ? tile_fmt<__nv_bfloat16>(a, fmt, rnd, s) : tile_fmt<float>(a, fmt, rnd, s);
}

}  // namespace fqk
