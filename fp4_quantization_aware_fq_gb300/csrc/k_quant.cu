// k_quant.cu -- tensor amax, row-wise quantization and the tiled row +
// column-wise quantization kernels.
//
// Row-wise ("Resumo Técnico: TetraJet-v2" §2A, 1x16 groups; MXFP4 1x32 as
// named on "Aprimorando gpt-oss ...", "O que há de novo"): one thread per
// block.  The thread loads the block's 16-byte vectors, takes its amax (for
// BF16 1x16 blocks from a max tree over the packed pairs), derives the scale
// once and writes the packed codes, the scale, the fake-quantized values and
// the STE mask bits of its block.  The double block's 8 inner blocks of a
// 1x128 outer block sit on 8 consecutive lanes, which share the outer amax
// by shuffles.
//
// Column-wise (§2A, the transposed 1x16 groups of the backward pass): a CTA
// stages a tile of x in shared memory while doing the row-wise pass on it,
// then quantizes column blocks (16x1; 32x1 for MXFP4) out of shared memory
// and writes the transposed codes through a shared-memory staging buffer.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kThreads = 256;
// CTAs per SM the register allocation must allow, measured: row kernels 4
// (at most 64 registers; the double-block SR call 3-4% faster despite a few
// spills), BF16 tile kernels 3 (80 registers; the Hadamard-transformed SR call
// 2% faster, the NVFP4 row + column call 1.5%; the NVFP4 tile kernel fits 60
// registers without spills, but four CTAs per SM ran 2.5% slower than three).
// The FP32 tile kernels, whose tiles need far more registers, are left free.
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

// The same over the rows of a tensor whose rows lie ld elements apart: the
// CTAs take whole rows, each thread one 16-byte vector of the row at a time.
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_rows_kernel(const void *__restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ld,
                                                             unsigned *__restrict__ out)
{
    constexpr int E = VecInfo<T>::E;
    const int64_t vpr = cols / E;
    float m = 0.0f;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const char *row = (const char *)x + r * ld * (int64_t)sizeof(T);
        for (int64_t c = threadIdx.x; c < vpr; c += kThreads) {
            float v[E];
            unpack16<T>(ld16(row + c * 16), v);
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
        atomicMax(out, __float_as_uint(b));
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
    bool xhat32;  // xhat is 32-byte aligned (whole-sector stores)
};

// Quantize one row-wise block of B values held by this thread (v) whose
// amax is am (recomputed here after the Hadamard transform, when there is
// one).  `blk` is the flat block index in the tensor (flat element index
// blk * B).  For the double block, the 8 inner blocks of an outer block sit on
// 8 consecutive lanes, and all 32 lanes of the warp must call this together.
template <int FMT, int RND>
__device__ __forceinline__ void row_block(float *v, float am, int64_t blk, bool valid, float s_g,
                                          float inv6, const NvTables *tab, const RowOut &o,
                                          const PhiloxKey &key, uint32_t offset,
                                          uint32_t stream_id, bool rht, uint32_t signs)
{
    constexpr int B = FmtInfo<FMT>::B;
    if (FMT != NVFP4 && rht) {
#pragma unroll
        for (int j = 0; j < B / 16; ++j)
            rht16(v + 16 * j, signs);
        am = 0.0f;
#pragma unroll
        for (int i = 0; i < B; ++i)
            am = fmaxf(am, fabsf(v[i]));
    }
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
    // the mask first: after it the block's values are no longer needed
    const uint32_t mbits = o.mask ? block_mask<B>(v, sc.lim) : 0u;
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
    if (o.xhat && o.xhat_bf16 && o.xhat32) {
        // whole 32-byte sectors: one store per 16 values
#pragma unroll
        for (int w = 0; w < B / 8; w += 2)
            st32((char *)o.xhat + (blk * B + w * 8) * 2, xhat8_bf16(q[w], sc.s_eff),
                 xhat8_bf16(q[w + 1], sc.s_eff));
    } else if (o.xhat) {
#pragma unroll
        for (int w = 0; w < B / 8; ++w) {
            float xh[8];
            e2m1_decode8(q[w], xh);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 p = mul2(make_float2(xh[i], xh[i + 1]), make_float2(sc.s_eff, sc.s_eff));
                xh[i] = p.x;
                xh[i + 1] = p.y;
            }
            if (o.xhat_bf16) {
                *reinterpret_cast<uint4 *>((char *)o.xhat + (blk * B + w * 8) * 2) =
                    make_uint4(bf16x2_rn(xh[0], xh[1]), bf16x2_rn(xh[2], xh[3]),
                               bf16x2_rn(xh[4], xh[5]), bf16x2_rn(xh[6], xh[7]));
            } else if (o.xhat32) {
                st32((char *)o.xhat + (blk * B + w * 8) * 4,
                     make_uint4(__float_as_uint(xh[0]), __float_as_uint(xh[1]),
                                __float_as_uint(xh[2]), __float_as_uint(xh[3])),
                     make_uint4(__float_as_uint(xh[4]), __float_as_uint(xh[5]),
                                __float_as_uint(xh[6]), __float_as_uint(xh[7])));
            } else {
                float4 *dst = reinterpret_cast<float4 *>((char *)o.xhat + (blk * B + w * 8) * 4);
                dst[0] = make_float4(xh[0], xh[1], xh[2], xh[3]);
                dst[1] = make_float4(xh[4], xh[5], xh[6], xh[7]);
            }
        }
    }
    if (o.mask) {
        if (B == 16)
            reinterpret_cast<uint16_t *>(o.mask)[blk] = (uint16_t)mbits;
        else
            reinterpret_cast<uint32_t *>(o.mask)[blk] = mbits;
    }
}

// One thread per block; each iteration a thread holds BPT blocks' loads in
// flight (about 64 bytes).
// STRIDED: the rows of x lie a.ld elements apart; block b (in row-major
// order) starts at element (b / (cols / B)) * ld + (b % (cols / B)) * B.
template <typename T, int FMT, int RND, bool STRIDED>
__global__ void __launch_bounds__(kThreads, kRowMinCtas) row_kernel(const __grid_constant__ RowArgs a)
{
    constexpr int B = FmtInfo<FMT>::B;
    constexpr int BPT = (B * sizeof(T) >= 64) ? 1 : 2;
    const int64_t nblk = a.n / B;
    auto src_of = [&](int64_t b) {
        int64_t e = b * B;
        if constexpr (STRIDED) {
            const int64_t bpr = a.cols / B;
            const int64_t r = b / bpr;
            e = r * a.ld + (b - r * bpr) * B;
        }
        return (const char *)a.x + e * (int64_t)sizeof(T);
    };
    __shared__ NvTables tab;
    wait_prior_grid();
    float s_g = 0.0f, inv6 = 0.0f;
    if (FMT == NVFP4) {
        s_g = outer_scale(*a.amax);
        inv6 = nv_inv6(s_g);
        nv_tables_fill(tab, s_g);
        __syncthreads();
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.tscale)
            a.tscale[0] = s_g;
    }
    const RowOut o{a.codes, a.scales, a.tscale, a.xhat, a.xhat_bf16, a.mask,
                   (reinterpret_cast<uintptr_t>(a.xhat) & 31u) == 0};
    const PhiloxKey &key = a.key;
    const bool rht = a.rht_seed != 0;
    const uint32_t signs = rht ? rht_signs(a.rht_seed, a.offset) : 0u;
    const int64_t stride = (int64_t)gridDim.x * kThreads * BPT;
    constexpr int NV = B / VecInfo<T>::E;  // 16-byte vectors per block
    // NVFP4 follows a full read of x (the tensor amax) and walks the blocks
    // from the end of x back to the start, so that it first meets the part of
    // x that the amax pass left in L2.
    auto block_at = [&](int64_t b) { return FMT == NVFP4 ? nblk - 1 - b : b; };
    for (int64_t base = (int64_t)blockIdx.x * kThreads * BPT; base < nblk; base += stride) {
        if constexpr (B == 16) {
            // 1x16 blocks: the amax comes from the raw vectors (packed pairs
            // for BF16), then the values are widened.
            uint4 raw[BPT][NV];
#pragma unroll
            for (int k = 0; k < BPT; ++k) {
                const int64_t b = base + k * kThreads + threadIdx.x;
                const char *src = src_of(block_at(b));
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    raw[k][i] = (b < nblk) ? ld16(src + 16 * i) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < BPT; ++k) {
                const int64_t b = base + k * kThreads + threadIdx.x;
                const float am = block_amax<T, B>(raw[k]);
                float v[B];
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    unpack16<T>(raw[k][i], v + i * VecInfo<T>::E);
                row_block<FMT, RND>(v, am, block_at(b), b < nblk, s_g, inv6, &tab, o, key,
                                    a.offset, a.stream_id, rht, signs);
            }
        } else {
            // 1x32 blocks (one per thread): widened as they load, which keeps
            // the raw vectors out of the register budget.
            static_assert(BPT == 1, "one 1x32 block per thread and iteration");
            const int64_t b = base + threadIdx.x;
            float v[B];
            if (b < nblk)
                load_block<T, B>(src_of(block_at(b)), v);
            else
#pragma unroll
                for (int i = 0; i < B; ++i)
                    v[i] = 0.0f;
            float am = 0.0f;
#pragma unroll
            for (int i = 0; i < B; ++i)
                am = fmaxf(am, fabsf(v[i]));
            row_block<FMT, RND>(v, am, block_at(b), b < nblk, s_g, inv6, &tab, o, key, a.offset,
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
// Row stride of the staged x tile in elements: one 16-byte vector of padding
// shifts each row by four banks, so the 8 threads of a quarter warp that stage
// two rows of BF16 1x16 blocks hit distinct banks.
template <typename T, int FMT>
__host__ __device__ constexpr int tile_pitch()
{
    return TileShape<FMT>::TC + 16 / (int)sizeof(T);
}

template <typename T, int FMT>
constexpr size_t tile_smem_bytes()
{
    using S = TileShape<FMT>;
    return (size_t)S::TR * tile_pitch<T, FMT>() * sizeof(T)  // x tile
           + (size_t)S::TC * S::CP                    // staged column codes
           + (size_t)S::TC * (S::TR / S::BC)          // staged column scales
           + (FMT == NV2L ? (size_t)S::TC * (S::TR / S::BC) * 4 : 0);  // inner amax
}

// STRIDED: the rows of x lie a.ld elements apart (else a.cols).
template <typename T, int FMT, int RND, bool STRIDED>
__global__ void __launch_bounds__(kThreads, tile_min_ctas<T, FMT>())
    tile_kernel(const __grid_constant__ TileArgs a)
{
    using S = TileShape<FMT>;
    constexpr int E = VecInfo<T>::E;
    constexpr int TR = S::TR, TC = S::TC, BC = S::BC, CP = S::CP;
    constexpr int BR = FmtInfo<FMT>::B;  // row block
    constexpr int RBPR = TC / BR;         // row blocks per tile row
    constexpr int NRB = TR / BC;          // column blocks per tile column
    extern __shared__ __align__(16) unsigned char smem[];
    T *tile = reinterpret_cast<T *>(smem);
    constexpr int TCP = tile_pitch<T, FMT>();
    uint8_t *ccs = smem + (size_t)TR * TCP * sizeof(T);  // [TC][CP]
    uint8_t *css = ccs + (size_t)TC * CP;                // [TC][NRB]
    float *am16 = reinterpret_cast<float *>(css + (size_t)TC * NRB);  // [NRB][TC]

    const int64_t rows = a.rows, cols = a.cols;
    __shared__ NvTables tab;
    wait_prior_grid();
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
    const RowOut o{a.rcodes, a.rscales, a.rtscale, a.xhat, a.xhat_bf16, a.mask,
                   (reinterpret_cast<uintptr_t>(a.xhat) & 31u) == 0};
    const PhiloxKey &key = a.key;
    const bool rht = a.rht_seed != 0;
    const uint32_t signs = rht ? rht_signs(a.rht_seed, a.offset) : 0u;

    // Each thread owns RPT row blocks of a tile.  The loads of the next tile
    // are issued once the current tile is staged in shared memory, so they
    // overlap its row pass, column pass and write-out.
    constexpr int RPT = (TR * RBPR + kThreads - 1) / kThreads;
    constexpr int NV = BR / E;  // 16-byte vectors per row block
    uint4 nxt[RPT][NV];
    // whole-sector loads: x and its row pitch on 32-byte boundaries (row blocks
    // start at multiples of 16 elements)
    const bool tal32 = ((reinterpret_cast<uintptr_t>(a.x) |
                         (uintptr_t)((STRIDED ? a.ld : cols) * (int64_t)sizeof(T))) & 31u) == 0;
    auto load_tile = [&](int ty, int tx) {
        const int64_t lr0 = (int64_t)ty * TR, lc0 = (int64_t)tx * TC;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int t = threadIdx.x + j * kThreads;
            const int tr = t / RBPR, tb = t % RBPR;
            const int64_t gr = lr0 + tr, gc = lc0 + (int64_t)tb * BR;
            const bool valid = t < TR * RBPR && gr < rows;
            const char *src =
                (const char *)a.x + (gr * (STRIDED ? a.ld : cols) + gc) * (int64_t)sizeof(T);
            // Each 16-byte vector is fetched only if it lies inside the row:
            // a column-only MXFP4 call admits cols % 32 == 16, where the last
            // 1x32 row block of a row holds only 16 elements (cols is a
            // multiple of 16, hence of E, so a vector is all in or all out).
            if (valid && tal32 && gc + (int64_t)NV * E <= cols) {
                load_vecs<NV>(src, nxt[j], true);
            } else {
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    nxt[j][k] = (valid && gc + (int64_t)k * E < cols) ? ld16(src + 16 * k)
                                                                      : make_uint4(0, 0, 0, 0);
            }
        }
    };

    // Persistent CTAs walk the tiles in row-major order, gridDim.x tiles per
    // step: (ty, tx) advances by (dy, dx) with a carry, without a division.
    // The launcher keeps both tile counts below 2^31.
    const int ntr = (int)((rows + TR - 1) / TR), ntc = (int)((cols + TC - 1) / TC);
    const int dy = (int)gridDim.x / ntc, dx = (int)gridDim.x % ntc;
    int ty = (int)blockIdx.x / ntc, tx = (int)blockIdx.x % ntc;
    // NVFP4 follows a full read of x (the tensor amax): its walk visits the
    // tiles in reverse order (tile (ty, tx) of the walk is tile (ntr - 1 - ty,
    // ntc - 1 - tx) of x), so that it starts on the part of x that the amax
    // pass left in L2.
    auto tr_of = [&](int y) { return FMT == NVFP4 ? ntr - 1 - y : y; };
    auto tc_of = [&](int x) { return FMT == NVFP4 ? ntc - 1 - x : x; };
    if (ty < ntr)
        load_tile(tr_of(ty), tc_of(tx));
    while (ty < ntr) {
    const int64_t r0 = (int64_t)tr_of(ty) * TR;
    const int64_t c0 = (int64_t)tc_of(tx) * TC;
    int ny = ty + dy, nx = tx + dx;
    if (nx >= ntc) {
        nx -= ntc;
        ++ny;
    }

    // Phase 1: stage the tile's row blocks in shared memory, start the next
    // tile's loads, then (when asked) run the row-wise pass on the staged
    // blocks, each thread reading back its own.
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int t = threadIdx.x + j * kThreads;
        if (RPT * kThreads > TR * RBPR && t >= TR * RBPR)
            break;
        const int tr = t / RBPR, tb = t % RBPR;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            *reinterpret_cast<uint4 *>(tile + tr * TCP + tb * BR + k * E) = nxt[j][k];
    }
    if (ny < ntr)
        load_tile(tr_of(ny), tc_of(nx));
    if (a.do_row) {
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int t = threadIdx.x + j * kThreads;
            if (RPT * kThreads > TR * RBPR && t >= TR * RBPR)
                break;
            const int tr = t / RBPR, tb = t % RBPR;
            const int64_t gr = r0 + tr, gc = c0 + (int64_t)tb * BR;
            const bool valid = gr < rows && gc < cols;
            uint4 raw[NV];
#pragma unroll
            for (int k = 0; k < NV; ++k)
                raw[k] = *reinterpret_cast<const uint4 *>(tile + tr * TCP + tb * BR + k * E);
            const float am = block_amax<T, BR>(raw);
            float v[BR];
#pragma unroll
            for (int k = 0; k < NV; ++k)
                unpack16<T>(raw[k], v + k * E);
            row_block<FMT, RND>(v, am, (gr * cols + gc) / BR, valid, s_g, inv6, &tab, o, key,
                                a.offset, 0u, rht, signs);
        }
    }
    __syncthreads();

    // Phase 2: column blocks (BC rows x 1 column) out of shared memory.  BF16
    // NVFP4 tiles are read two columns at a time (one 32-bit word per row).
    const uint32_t *tile32 = reinterpret_cast<const uint32_t *>(tile);
    auto abs_max = [&](const float *v) {
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < BC; ++i)
            m = fmaxf(m, fabsf(v[i]));
        return m;
    };
    // column c, rows rb * BC .. rb * BC + BC - 1 of the tile, widened to FP32
    // (and Hadamard-transformed, if asked: not for NVFP4)
    auto load_col = [&](int c, int rb, float *v) {
#pragma unroll
        for (int i = 0; i < BC; ++i)
            v[i] = static_cast<float>(tile[(rb * BC + i) * TCP + c]);
        if (FMT != NVFP4 && rht) {
#pragma unroll
            for (int j = 0; j < BC / 16; ++j)
                rht16(v + 16 * j, signs);
        }
    };
    // Double block: a first sweep stores the amax of every 16 x 1 block, for
    // the 128-row outer scales.  In both sweeps a thread's column is the same
    // for each of its tasks (TC divides the thread count), so the quantize
    // sweep derives its outer scale once per tile and takes each block's
    // amax from the first sweep.
    static_assert(FMT != NV2L || kThreads % TC == 0, "a thread's column must not change");
    if (FMT == NV2L) {
        for (int task = threadIdx.x; task < TC * NRB; task += kThreads) {
            const int c = task % TC, rb = task / TC;
            float v[BC];
            load_col(c, rb, v);
            am16[rb * TC + c] = abs_max(v);
        }
        __syncthreads();
    }
    // quantize column block (c, rb) of the tile into the staging buffers: v
    // holds the block (after the Hadamard transform, if any), m its amax
    auto col_quant = [&](int c, int rb, float *v, float m, float s_o, float inv6c) {
        const int64_t gc = c0 + c, gr0 = r0 + (int64_t)rb * BC;
        if (FMT == NV2L && rb == 0)
            a.ctscale[gc * (rows / 128) + r0 / 128] = s_o;
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
                wd[i] = tile32[((rb * BC + i) * TCP + c) / 2];
            // both columns' amax from one tree over the packed pairs
            const uint32_t mw = bf16x2_absmax_tree<BC>(wd);
#pragma unroll
            for (int i = 0; i < BC; ++i)
                v[i] = __uint_as_float(wd[i] << 16);
            col_quant(c, rb, v, bf16_lo_abs(mw), s_g, inv6);
#pragma unroll
            for (int i = 0; i < BC; ++i)
                v[i] = __uint_as_float(wd[i] & 0xFFFF0000u);
            col_quant(c + 1, rb, v, bf16_hi_abs(mw), s_g, inv6);
        }
    } else if constexpr (FMT == NV2L) {
        // the outer scale of this thread's column: the largest inner amax of
        // the column over the tile's 128 rows
        const int c = threadIdx.x % TC;
        float mo = 0.0f;
#pragma unroll
        for (int j = 0; j < NRB; ++j)
            mo = fmaxf(mo, am16[j * TC + c]);
        const float s_o = outer_scale(mo), inv6c = nv_inv6(s_o);
        for (int task = threadIdx.x; task < TC * NRB; task += kThreads) {
            const int rb = task / TC;
            if (c0 + c >= cols || r0 + (int64_t)rb * BC >= rows)
                continue;
            float v[BC];
            load_col(c, rb, v);  // the same values as in the amax sweep
            col_quant(c, rb, v, am16[rb * TC + c], s_o, inv6c);
        }
    } else {
        for (int task = threadIdx.x; task < TC * NRB; task += kThreads) {
            const int c = task % TC, rb = task / TC;
            if (c0 + c >= cols || r0 + (int64_t)rb * BC >= rows)
                continue;
            float v[BC];
            load_col(c, rb, v);
            col_quant(c, rb, v, abs_max(v), s_g, inv6);
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
    if constexpr (NRB == 8) {
        // a column's 8 scales are 8 consecutive bytes of its row of X^T; the
        // row offset gc * (rows / 16) + r0 / 16 is a multiple of 8 when rows is
        // a multiple of 128 (else the bytes go one at a time)
        for (int c = threadIdx.x; c < TC; c += kThreads) {
            const int64_t gc = c0 + c;
            if (gc >= cols)
                continue;
            uint8_t *dst = a.cscales + gc * (rows / BC) + r0 / BC;
            if ((rows % 128) == 0 && r0 + TR <= rows) {
                *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(css + c * NRB);
            } else {
#pragma unroll
                for (int j = 0; j < NRB; ++j)
                    if (r0 + (int64_t)j * BC < rows)
                        dst[j] = css[c * NRB + j];
            }
        }
    } else {
        for (int u = threadIdx.x; u < TC * NRB; u += kThreads) {
            const int c = u / NRB, j = u % NRB;
            const int64_t gc = c0 + c, gr = r0 + (int64_t)j * BC;
            if (gc < cols && gr < rows)
                a.cscales[gc * (rows / BC) + gr / BC] = css[c * NRB + j];
        }
    }
    // No barrier here: the next tile's phase 1 writes only the x tile, which
    // every thread finished reading before the barrier that ended phase 2;
    // the staging buffers read above are written again in the next tile's
    // phase 2, after the barrier that ends its phase 1, which every thread
    // reaches only once it is done here.
    ty = ny;
    tx = nx;
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
    // eight CTAs per SM keep 128 KB of loads in flight per SM (four: 1.3 us
    // slower on the NVFP4 activation's amax)
    const int grid = persistent_grid(nch, kThreads * 4, 8);
    if (bf16)
        amax_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(x, nch, (unsigned *)out);
    else
        amax_kernel<float><<<grid, kThreads, 0, s>>>(x, nch, (unsigned *)out);
    return cudaGetLastError();
}

cudaError_t launch_amax_rows(const void *x, int bf16, int64_t rows, int64_t cols, int64_t ld,
                             float *out, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), s);
    if (e != cudaSuccess)
        return e;
    if (rows == 0 || cols == 0)
        return cudaSuccess;
    const int grid = persistent_grid(rows, 1, 8);
    if (bf16)
        amax_rows_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(x, rows, cols, ld, (unsigned *)out);
    else
        amax_rows_kernel<float><<<grid, kThreads, 0, s>>>(x, rows, cols, ld, (unsigned *)out);
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
    // Stochastic rounding is bound by its arithmetic: a grid of sixteen CTAs
    // per SM walks the tensor, four of them resident at a time (68.4-68.5 us
    // for the double-block SR gradient with 12 to 32 per SM, 69.3 us with 8,
    // 72.7 us with 4, 71.7 us with one CTA per 256 x BPT blocks).  Nearest-even rounding is bound by
    // memory: one CTA per 256 x BPT blocks, handed out in address order, keeps
    // the reads sequential (MXFP4 weight [32768, 4096]: 98 us against 118 us
    // for the grid-stride walk).
    const int grid = persistent_grid(nblk, kThreads * BPT, RND == SR ? 16 : 1 << 20);
    if (a.ld != a.cols)
        return launch_dependent(row_kernel<T, FMT, RND, true>, dim3(grid), dim3(kThreads), 0, s, a);
    return launch_dependent(row_kernel<T, FMT, RND, false>, dim3(grid), dim3(kThreads), 0, s, a);
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
    const auto kern =
        a.ld != a.cols ? tile_kernel<T, FMT, RND, true> : tile_kernel<T, FMT, RND, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int64_t ntc = (a.cols + S::TC - 1) / S::TC, ntr = (a.rows + S::TR - 1) / S::TR;
    if (ntc >= INT32_MAX || ntr >= INT32_MAX)
        return cudaErrorInvalidValue;
    const int64_t ntiles = ntc * ntr;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads,
                                                      smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    // Nearest-even tiles are bound by memory: one wave of resident CTAs walks
    // them.  Stochastic rounding is bound by arithmetic: three CTAs for each
    // resident slot, the later ones starting as the first finish, even out
    // the walk's tail (Hadamard + SR both orientations on [16384, 4096]:
    // 181.5 us against 190.3 with one wave, 183.4 with two, 183.0 with four;
    // two waves took the NVFP4 row + column call from 98.9 to 100.5 us).
    const int64_t cap = (int64_t)sm_count() * per_sm * (RND == SR ? 3 : 1);
    const unsigned grid = (unsigned)(ntiles < cap ? ntiles : cap);
    return launch_dependent(kern, dim3(grid), dim3(kThreads), smem, s, a);
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
