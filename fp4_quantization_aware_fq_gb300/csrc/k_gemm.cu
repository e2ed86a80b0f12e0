// k_gemm.cu -- block-scaled FP4 GEMM on the 5th-generation tensor cores:
// C[M, N] = alpha * A[M, K] B[N, K]^T for NVFP4 or MXFP4 operands exactly as
// the quantizers store them (packed E2M1 codes; one E4M3 scale per 1x16 block
// along K and an FP32 tensor scale each for NVFP4, one E8M0 scale per 1x32
// block for MXFP4) -- the forward GEMM of a QAT linear layer
// ("Aprimorando gpt-oss para Precisão e Desempenho com Treinamento Consciente
// à Quantização", "O que há de novo": NVFP4 with FP8 E4M3 block scales;
// "Resumo Técnico: TetraJet-v2", §2A: 1x16 groups along the reduction).
//
// The tensor cores take the block scales from tensor memory in 4-column
// groups, one per 4 scales of every row: TMEM lane 32q + i, column c + q
// holds the four scales of row 32q + i.  That is what
// tcgen05.cp.32x128b.warpx4 produces from a 512-byte atom in which byte
// (m % 32) * 16 + (m / 32) * 4 + j is the scale of row m, block j, so
// sf_to_mma_kernel first rearranges each operand's row-major scales into such
// atoms ([row block][group of 4 blocks], 512 bytes each) in the caller's
// workspace.  An NVFP4 atom covers K = 64, one MMA (scale_vec::4X); an MXFP4
// atom covers K = 128, two MMAs of K = 64 that take two scales each
// (scale_vec::2X), the second selecting bytes 2-3 of each cell through the
// instruction's scale-factor ids.
//
// One CTA computes a 128 x 128 tile of C with warp-specialised roles:
//   warp 0   producer: per K-tile of 256 elements, the A and B code tiles by
//            TMA (128 rows x 128 bytes, 128-byte swizzle) and the A and B
//            scale atoms (4 x 512 bytes each, one bulk copy per operand) into
//            one of kGemmStages shared buffers;
//   warp 1   owns the tensor memory; one thread copies each MMA's scale atoms
//            into tensor memory (tcgen05.cp) and issues the four block-scaled
//            MMAs of the K-tile (tcgen05.mma kind::mxf4nvf4, scale_vec::4X,
//            K = 64 each), then commits them to the stage's "empty" barrier;
//   warps 2-5 epilogue: tcgen05.ld of the FP32 accumulator, times alpha =
//            s_A s_B, stored as FP32 or BF16.
// Every mbarrier wait is bounded (fq_async.cuh); on a timeout the CTA records
// it in the caller's error word, stops issuing work, waits (bounded) for what
// it already issued and frees its tensor memory before it exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "fq_async.cuh"
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fqk {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 128;
constexpr int kGemmBK = 256;                        // FP4 elements per K-tile
constexpr int kGemmStages = 3;
constexpr int kGemmThreads = 192;
constexpr uint32_t kTileBytesA = kGemmBM * kGemmBK / 2;   // 16 KB
constexpr uint32_t kTileBytesB = kGemmBN * kGemmBK / 2;   // 16 KB
constexpr uint32_t kTmemCols = 256;  // accumulator (128) + per-stage scale columns (32 each)
constexpr uint32_t kSfColBase = 128;
constexpr uint32_t kSfAtomBytes = 512;  // the scales of 128 rows x one group of 4 blocks

// Per-format layout of one pipeline stage (codes, then the scale atoms).
template <int FMT>
struct GemmFmt {
    static constexpr int SB = (FMT == MXFP4) ? 32 : 16;         // elements per scale
    static constexpr uint32_t kSfBytesA = kGemmBM * (kGemmBK / SB);  // NVFP4 2 KB, MXFP4 1 KB
    static constexpr uint32_t kSfBytesB = kGemmBN * (kGemmBK / SB);
    static constexpr uint32_t kStageBytes = kTileBytesA + kTileBytesB + kSfBytesA + kSfBytesB;
    static constexpr int kAtoms = kGemmBK / (4 * SB);              // scale atoms per K-tile
};
size_t gemm_smem_bytes()
{
    // the larger (NVFP4) stage, + alignment slack for the 1 KB swizzle atoms
    return (size_t)kGemmStages * GemmFmt<NVFP4>::kStageBytes + 1024;
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all in 16-byte units), descriptor version 1, swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// Instruction descriptor of the block-scaled FP4 kinds: A and B E2M1, both
// K-major, N >> 3 at bit 17, scale type at bit 23 (0 UE4M3, 1 UE8M0), M >> 4
// at bit 24, the B and A scale-factor ids (byte offsets inside each 32-bit
// scale cell) at bits 4 and 29.
__host__ __device__ constexpr uint32_t gemm_idesc(uint32_t ue8m0, uint32_t sf_id)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(kGemmBN >> 3) << 17) | (ue8m0 << 23) |
           ((uint32_t)(kGemmBM >> 4) << 24) | (sf_id << 4) | (sf_id << 29);
}

// ---------------------------------------------------------------- tcgen05 / TMA wrappers
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 rows x 16 bytes of shared memory into TMEM columns taddr .. taddr + 3 of
// each of the four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

template <int FMT>
__device__ __forceinline__ void tc_mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                           uint32_t accumulate)
{
    if (FMT == MXFP4)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive FP32 columns of this warp's 32 accumulator lanes.
__device__ __forceinline__ void tc_ld_32cols(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32"
                 " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
                 " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
                 " [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- kernel
template <int FMT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b, const GemmArgs g)
{
    using F = GemmFmt<FMT>;
    constexpr uint32_t kStageBytes = F::kStageBytes, kSfBytesA = F::kSfBytesA,
                       kSfBytesB = F::kSfBytesB;
    extern __shared__ __align__(1024) unsigned char gsm_raw[];
    // 1 KB alignment for the 128-byte-swizzle atoms
    unsigned char *gsm = gsm_raw + ((1024u - (smem_u32(gsm_raw) & 1023u)) & 1023u);
    __shared__ uint64_t full[kGemmStages], empty[kGemmStages], done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kGemmBM, n0 = blockIdx.x * kGemmBN;
    const int kt_n = (int)((g.k + kGemmBK - 1) / kGemmBK);  // the last K-tile zero-filled past k

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init_fence();
        abort_flag = 0;
    }
    if (warp == 1)
        tc_alloc(&tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    auto stage_ptr = [&](int s) { return gsm + (size_t)s * kStageBytes; };

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        for (int kt = 0; kt < kt_n; ++kt) {
            const int s = kt % kGemmStages;
            if (kt >= kGemmStages && !mbar_wait(&empty[s], ((kt / kGemmStages) - 1) & 1)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*(volatile int *)&abort_flag)
                break;
            unsigned char *st = stage_ptr(s);
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(st, &map_a, kt * (kGemmBK / 2), m0, &full[s]);
            tma_load_2d(st + kTileBytesA, &map_b, kt * (kGemmBK / 2), n0, &full[s]);
            // the K-tile's scale atoms of each operand are contiguous
            const int64_t kgroups = (int64_t)kt_n * F::kAtoms;  // padded to whole K-tiles
            const uint8_t *sfa =
                g.sfa_mma + ((int64_t)blockIdx.y * kgroups + F::kAtoms * kt) * kSfAtomBytes;
            const uint8_t *sfb =
                g.sfb_mma + ((int64_t)blockIdx.x * kgroups + F::kAtoms * kt) * kSfAtomBytes;
            bulk_g2s(st + kTileBytesA + kTileBytesB, sfa, kSfBytesA, &full[s]);
            bulk_g2s(st + kTileBytesA + kTileBytesB + kSfBytesA, sfb, kSfBytesB, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t ue8m0 = FMT == MXFP4 ? 1u : 0u;
        for (int kt = 0; kt < kt_n; ++kt) {
            const int s = kt % kGemmStages;
            if (!mbar_wait(&full[s], (kt / kGemmStages) & 1)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*(volatile int *)&abort_flag)
                break;
            tc_fence_after();
            unsigned char *st = stage_ptr(s);
            const uint32_t a_addr = smem_u32(st), b_addr = smem_u32(st + kTileBytesA);
            const uint32_t sfa_addr = smem_u32(st + kTileBytesA + kTileBytesB);
            const uint32_t sfb_addr = sfa_addr + kSfBytesA;
            // per stage 16 TMEM columns of A scales then 16 of B scales (4 per atom)
            const uint32_t sfa_t = tmem + kSfColBase + (uint32_t)s * 32;
            const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
            for (int at = 0; at < F::kAtoms; ++at) {
                // a scale atom: 32 rows of 16 bytes, 8-row core matrices 128 B apart
                tc_cp_32x128b_x4(sfa_t + 4u * at,
                                 smem_desc(sfa_addr + kSfAtomBytes * at, 16, 128, kSwizzleNone));
                tc_cp_32x128b_x4(sfb_t + 4u * at,
                                 smem_desc(sfb_addr + kSfAtomBytes * at, 16, 128, kSwizzleNone));
            }
#pragma unroll
            for (int kk = 0; kk < kGemmBK / 64; ++kk) {
                // each MMA takes K = 64 FP4 elements = 32 bytes of every row; an
                // NVFP4 MMA reads a whole atom, an MXFP4 MMA half of one
                const int at = (FMT == MXFP4) ? kk / 2 : kk;
                const uint32_t idesc = gemm_idesc(ue8m0, (FMT == MXFP4) ? 2u * (kk & 1) : 0u);
                const uint64_t ad = smem_desc(a_addr + 32u * kk, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(b_addr + 32u * kk, 16, 1024, kSwizzle128B);
                tc_mma_fp4<FMT>(tmem, ad, bd, idesc, sfa_t + 4u * at, sfb_t + 4u * at,
                                (kt | kk) ? 1u : 0u);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(&done);  // every MMA issued above (none if the loop ended early)
    }

    // ---- epilogue (warps 2..5 hold TMEM lane quarters warp % 4)
    if (warp >= 2) {
        const bool ok = mbar_wait(&done, 0);
        if (!ok)
            atomicExch(&abort_flag, 1);
        tc_fence_after();
        // warp-uniform decision: tcgen05.ld is a warp-wide (.sync.aligned) operation
        if (__all_sync(0xFFFFFFFFu, ok && !*(volatile int *)&abort_flag)) {
            const int q = warp & 3;
            const int row = m0 + 32 * q + lane;
            const bool row_ok = row < g.m;  // rows past m hold the tile's zero padding
            const bool c32 = (reinterpret_cast<uintptr_t>(g.c) & 31u) == 0;
            float alpha = 1.0f;
            if (g.tscale_a && g.tscale_b)
                alpha = __fmul_rn(__ldg(g.tscale_a), __ldg(g.tscale_b));
#pragma unroll 1
            for (int c = 0; c < kGemmBN / 32; ++c) {
                float v[32];
                tc_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * c), v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = __fmul_rn(v[i], alpha);
                const int64_t off = (int64_t)row * g.n + n0 + 32 * c;
                if (!row_ok || n0 + 32 * c >= g.n)  // n % 32 == 0: a 32-column chunk is all in or out
                    continue;
                if (g.c_bf16 && c32) {
                    // whole 32-byte sectors, one store per 16 values
                    char *dst = (char *)g.c + off * 2;
#pragma unroll
                    for (int i = 0; i < 4; i += 2)
                        st32(dst + 16 * i,
                             make_uint4(bf16x2_rn(v[8 * i], v[8 * i + 1]),
                                        bf16x2_rn(v[8 * i + 2], v[8 * i + 3]),
                                        bf16x2_rn(v[8 * i + 4], v[8 * i + 5]),
                                        bf16x2_rn(v[8 * i + 6], v[8 * i + 7])),
                             make_uint4(bf16x2_rn(v[8 * i + 8], v[8 * i + 9]),
                                        bf16x2_rn(v[8 * i + 10], v[8 * i + 11]),
                                        bf16x2_rn(v[8 * i + 12], v[8 * i + 13]),
                                        bf16x2_rn(v[8 * i + 14], v[8 * i + 15])));
                } else if (g.c_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>((char *)g.c + off * 2);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(bf16x2_rn(v[8 * i], v[8 * i + 1]),
                                            bf16x2_rn(v[8 * i + 2], v[8 * i + 3]),
                                            bf16x2_rn(v[8 * i + 4], v[8 * i + 5]),
                                            bf16x2_rn(v[8 * i + 6], v[8 * i + 7]));
                } else if (c32) {
                    char *dst = (char *)g.c + off * 4;
#pragma unroll
                    for (int i = 0; i < 8; i += 2)
                        st32(dst + 16 * i,
                             make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                        __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])),
                             make_uint4(__float_as_uint(v[4 * i + 4]), __float_as_uint(v[4 * i + 5]),
                                        __float_as_uint(v[4 * i + 6]), __float_as_uint(v[4 * i + 7])));
                } else {
                    float4 *dst = reinterpret_cast<float4 *>((char *)g.c + off * 4);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *(volatile int *)&abort_flag && g.err)
        atomicOr(g.err, (int)kDevErrWaitTimeout);
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D byte tensor [rows, row_bytes] with a box of box_rows x box_bytes.
static bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t row_bytes,
                     uint32_t box_bytes, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major scales [rows, kb] (kb = k / B) -> MMA atoms [ceil(rows / 128)]
// [kgroups][512 B], kgroups = 4-scale groups padded to whole K-tiles: one
// thread per 4-byte word of the output (the four scales of one row and one
// group).  Rows past `rows` and scales past kb are written as 0 (a finite
// scale: the codes the tensor map reads there are zero-filled).
__global__ void __launch_bounds__(256) sf_to_mma_kernel(const uint8_t *__restrict__ scales,
                                                        int64_t rows, int64_t kb,
                                                        int64_t kgroups,
                                                        uint32_t *__restrict__ out)
{
    const int64_t words = (rows + 127) / 128 * kgroups * 128;
    for (int64_t w = (int64_t)blockIdx.x * 256 + threadIdx.x; w < words;
         w += (int64_t)gridDim.x * 256) {
        const int pos = (int)(w & 127);
        const int64_t atom = w >> 7;
        const int64_t kg = atom % kgroups, rb = atom / kgroups;
        const int64_t m = rb * 128 + 32 * (pos & 3) + (pos >> 2);
        uint32_t word = 0;
        if (m < rows) {
            const uint8_t *src = scales + m * kb + 4 * kg;
            if ((kb & 3) == 0 && 4 * kg + 3 < kb) {
                word = __ldg(reinterpret_cast<const uint32_t *>(src));  // aligned, in range
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (4 * kg + j < kb)
                        word |= (uint32_t)__ldg(src + j) << (8 * j);
            }
        }
        out[w] = word;
    }
}

// Both operands' scale atoms, rows padded to 128 and k to whole K-tiles
// (NVFP4's size; MXFP4 needs half).
static int64_t pad_to(int64_t v, int64_t q) { return (v + q - 1) / q * q; }

size_t gemm_workspace_bytes(int64_t m, int64_t n, int64_t k)
{
    return (size_t)(pad_to(m, 128) + pad_to(n, 128)) * (size_t)(pad_to(k, kGemmBK) / 16);
}

template <int FMT>
static cudaError_t gemm_go(const GemmArgs &g0, void *ws, cudaStream_t s)
{
    using F = GemmFmt<FMT>;
    GemmArgs g = g0;
    const int64_t kgroups = pad_to(g.k, kGemmBK) / (4 * F::SB);
    uint8_t *sfa = static_cast<uint8_t *>(ws);
    uint8_t *sfb = sfa + (size_t)pad_to(g.m, 128) * (size_t)kgroups * 4;
    g.sfa_mma = sfa;
    g.sfb_mma = sfb;
    CUtensorMap ma, mb;
    if (!make_map(&ma, g.a_codes, (uint64_t)g.m, (uint64_t)g.k / 2, kGemmBK / 2, kGemmBM,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mb, g.b_codes, (uint64_t)g.n, (uint64_t)g.k / 2, kGemmBK / 2, kGemmBN,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int cap = sm_count() * 8;
    for (int op = 0; op < 2; ++op) {
        const int64_t rows = op ? g.n : g.m;
        const int64_t words = pad_to(rows, 128) * kgroups;
        const int64_t need = (words + 255) / 256;
        sf_to_mma_kernel<<<(unsigned)(need < cap ? need : cap), 256, 0, s>>>(
            op ? g.b_scales : g.a_scales, rows, g.k / F::SB, kgroups,
            reinterpret_cast<uint32_t *>(op ? sfb : sfa));
    }
    const size_t smem = gemm_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(gemm_fp4_kernel<FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((g.n + kGemmBN - 1) / kGemmBN), (unsigned)((g.m + kGemmBM - 1) / kGemmBM));
    gemm_fp4_kernel<FMT><<<grid, kGemmThreads, smem, s>>>(ma, mb, g);
    return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs &g, int fmt, void *ws, cudaStream_t s)
{
    return fmt == MXFP4 ? gemm_go<MXFP4>(g, ws, s) : gemm_go<NVFP4>(g, ws, s);
}

}  // namespace fqk
