// fq_internal.h -- argument blocks and launchers shared between the C ABI
// (fq_api.cu) and the kernel translation units.  Host-side only types.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define FQK_HD __host__ __device__
#else
#define FQK_HD
#endif

namespace fqk {

// Round keys of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): the key (seed low, seed high) plus r
// times the two Weyl constants for rounds r = 0..9.  The host computes them
// once per call and passes them in the kernel arguments, where the kernels
// read them as constants.
struct PhiloxKey {
    uint32_t k0[10], k1[10];
};

FQK_HD inline PhiloxKey philox_key(uint64_t seed)
{
    PhiloxKey k;
    for (int r = 0; r < 10; ++r) {
        k.k0[r] = (uint32_t)seed + 0x9E3779B9u * (uint32_t)r;
        k.k1[r] = (uint32_t)(seed >> 32) + 0xBB67AE85u * (uint32_t)r;
    }
    return k;
}

// Row-wise quantization of a dense tensor seen as a flat array of n elements
// (n a multiple of the block length).
struct RowArgs {
    const void *x;
    int64_t n;
    int64_t cols, ld;   // row length and row pitch of x in elements (ld == cols: dense)
    const float *amax;  // NVFP4: device pointer to the tensor amax
    uint8_t *codes;
    uint8_t *scales;
    float *tscale;      // NVFP4: s_g (1 float); double block: one per 128 elements
    void *xhat;         // optional fake-quantized output
    int xhat_bf16;
    uint8_t *mask;      // optional STE mask (1 bit per element)
    uint64_t seed;
    uint32_t offset;
    uint32_t stream_id;
    uint32_t rht_seed;  // 0: no Hadamard transform
    PhiloxKey key;      // round keys of seed
};

// Tiled quantization producing the column-wise (transposed) output and,
// optionally, the row-wise outputs from the same read of x.
struct TileArgs {
    const void *x;
    int64_t rows, cols;
    const float *amax;
    int do_row;
    uint8_t *rcodes;
    uint8_t *rscales;
    float *rtscale;
    void *xhat;
    int xhat_bf16;
    uint8_t *mask;
    uint8_t *ccodes;
    uint8_t *cscales;
    float *ctscale;
    uint64_t seed;
    uint32_t offset;
    uint32_t rht_seed;  // 0: no Hadamard transform
    PhiloxKey key;      // round keys of seed
    int64_t ld;         // row pitch of x in elements (>= cols)
};

struct DequantArgs {
    const uint8_t *codes;
    const uint8_t *scales;
    const float *tscale;
    int64_t n;
    int64_t cols, ldy;  // row length and row pitch of y in elements (ldy == cols: dense)
    void *y;
    int y_bf16;
};

// Grouped OsciReset passes: up to kOsciMaxTensors tensors per launch.  Tiles
// of kOsciTileChunks 16-byte chunks are numbered across the group; tile_start
// holds the prefix sums (tile_start[i] = first tile of tensor i).
constexpr int kOsciMaxTensors = 64;
constexpr int kOsciTileChunks = 2048;

struct OsciTensor {
    float *master;
    const float *delta;
    float *dist_q;
    float *dist_m;
    const uint8_t *pcodes;
    const uint8_t *pscales;
    const float *ptscale;
    uint8_t *ncodes;
    uint8_t *nscales;
    float *ntscale;
    void *xhat;
    uint8_t *mask;
    int64_t n;
};

struct OsciArgs {
    int ntensors;
    int xhat_bf16;
    int reset;                         // update: also end the OsciReset window
    uint64_t seed;
    uint32_t offset;
    PhiloxKey key;                     // round keys of seed
    float threshold;
    float *amax;                       // one float per tensor (workspace)
    unsigned long long *n_reset;
    int64_t tile_start[kOsciMaxTensors + 1];
    OsciTensor t[kOsciMaxTensors];
};

// Split FP4 / FP8 quantization of an activation with retained channels.
struct OutlierArgs {
    const void *x;
    int64_t rows, cols;
    const uint32_t *bitmap;   // retained channels, bit c % 32 of word c / 32
    int64_t k;                // number of retained channels
    const float *fp8_scale;   // [k] static scale of the j-th retained channel
    const float *amax;        // NVFP4: amax of x without the retained channels
    uint8_t *codes;
    uint8_t *scales;
    float *tscale;
    uint8_t *fp8;             // [rows, k] E4M3 codes of the retained elements
    void *xhat;
    int xhat_bf16;
    uint8_t *mask;
    uint64_t seed;
    uint32_t offset;
    PhiloxKey key;            // round keys of seed
};

// QAD distillation loss over [rows, vocab] teacher / student logits; each row
// is split over a cluster of csize CTAs holding `chunk` logits of each.
struct KlArgs {
    const void *zt;
    const void *zs;
    int64_t rows, vocab;
    int64_t chunk;
    int csize;
    float k2;          // log2(e) / T
    float gk;          // grad_scale / T
    float *loss_rows;
    void *dz;          // optional gradient with respect to zs
    int dz_bf16;
    int *err;          // optional device error word
};

// Block-scaled FP4 GEMM C[m, n] = alpha A[m, k] B[n, k]^T (NVFP4 or MXFP4
// operands; alpha = the two NVFP4 tensor scales, 1 for MXFP4).
struct GemmArgs {
    const uint8_t *a_codes, *a_scales;
    const uint8_t *b_codes, *b_scales;
    const float *tscale_a, *tscale_b;
    int64_t m, n, k;
    const uint8_t *sfa_mma, *sfb_mma;  // scales rearranged for the tensor cores (workspace)
    void *c;
    int c_bf16;
    int *err;
};

int sm_count();

cudaError_t launch_amax(const void *x, int bf16, int64_t n, float *out, cudaStream_t s);
cudaError_t launch_amax_rows(const void *x, int bf16, int64_t rows, int64_t cols, int64_t ld,
                             float *out, cudaStream_t s);
cudaError_t launch_row(const RowArgs &a, int bf16, int fmt, int rnd, cudaStream_t s);
cudaError_t launch_tile(const TileArgs &a, int bf16, int fmt, int rnd, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs &a, int fmt, cudaStream_t s);
cudaError_t launch_ste(const void *dy, int bf16, const uint8_t *mask, int64_t n, void *dx,
                       cudaStream_t s);
cudaError_t launch_osci_update(const OsciArgs &a, int fmt, int rnd, cudaStream_t s);
cudaError_t launch_osci_reset(const OsciArgs &a, int fmt, cudaStream_t s);
cudaError_t launch_channel_amax(const void *x, int bf16, int64_t rows, int64_t cols, float *amax,
                                cudaStream_t s);
cudaError_t launch_select(const float *amax, int cols, int k, int32_t *idx, uint32_t *bitmap,
                          float *fp8_scale, cudaStream_t s);
cudaError_t launch_masked_amax(const void *x, int bf16, int64_t rows, int64_t cols,
                               const uint32_t *bitmap, float *out, cudaStream_t s);
cudaError_t launch_outlier_quant(const OutlierArgs &a, int bf16, int fmt, int rnd,
                                 cudaStream_t s);
size_t gemm_smem_bytes();
size_t gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);
cudaError_t launch_gemm(const GemmArgs &g, int fmt, void *ws, cudaStream_t s);
struct QadPlan {
    int csize;        // CTAs per cluster (one row per cluster)
    int64_t chunk;    // logits of each tensor per CTA
    size_t smem;      // dynamic shared memory per CTA
    int threads;      // threads per CTA
};
bool qad_plan(int64_t vocab, int esz, QadPlan *p);
cudaError_t launch_qad_kl(const KlArgs &a, int bf16, const QadPlan &p, float *loss_mean,
                          cudaStream_t s);

}  // namespace fqk
