// fq_api.cu -- the C ABI declared in include/fq.h: host-side argument
// checks, workspace handling, and launches on the caller's stream.
#include <cmath>
#include <cstring>

#include "fq.h"
#include "fq_device.cuh"
#include "fq_internal.h"

using namespace fqk;

namespace {

inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline bool valid_cfg(const fq_config *c)
{
    return c && (c->format == FQ_NVFP4 || c->format == FQ_MXFP4 || c->format == FQ_NVFP4_2LEVEL) &&
           (c->rounding == FQ_RNE || c->rounding == FQ_SR);
}

inline bool valid_dtype(int32_t d)
{
    return d == FQ_F32 || d == FQ_BF16;
}

inline int64_t block_len(int fmt)
{
    return fmt == FQ_MXFP4 ? 32 : 16;
}

// Row-pass block constraint on the last dimension.
inline int64_t row_multiple(int fmt)
{
    return fmt == FQ_NVFP4_2LEVEL ? 128 : block_len(fmt);
}

inline fq_status cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? FQ_OK : FQ_ERR_CUDA;
}

// Checks a quantized-tensor descriptor that will be written or read.
fq_status check_q(const fq_qtensor *q, int fmt)
{
    if (!q || !q->codes || !q->scales)
        return FQ_ERR_INVALID_ARG;
    if (fmt != FQ_MXFP4 && !q->tscale)
        return FQ_ERR_INVALID_ARG;
    if (!aligned16(q->codes) || !aligned16(q->scales) || (q->tscale && !aligned16(q->tscale)))
        return FQ_ERR_ALIGN;
    return FQ_OK;
}

constexpr size_t kWsAmaxBytes = 256;

// Shared body of fq_quantize and fq_fakequant_ste.
// A row pitch: at least the row length, rows 16-byte aligned, and the
// strided extent addressable.
fq_status check_pitch(int64_t rows, int64_t cols, int64_t ld, int esize)
{
    if (ld < cols)
        return FQ_ERR_SHAPE;
    if ((ld * esize) % 16 != 0)
        return FQ_ERR_ALIGN;
    if (rows > 0 && ld > INT64_MAX / 4 / rows)
        return FQ_ERR_SHAPE;
    return FQ_OK;
}

fq_status quantize_common(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                          int64_t cols, int64_t ld, bool want_row_q, const fq_qtensor *row_out,
                          const fq_qtensor *col_out, void *xhat, int32_t xhat_dtype,
                          uint8_t *mask, const float *amax_in, void *ws, size_t ws_bytes,
                          void *stream)
{
    if (!valid_cfg(cfg) || !valid_dtype(x_dtype) || !x)
        return FQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0)
        return FQ_ERR_SHAPE;
    const int fmt = cfg->format;
    if (cfg->rht_seed && fmt == FQ_NVFP4)
        return FQ_ERR_UNSUPPORTED;
    const bool do_row = want_row_q || xhat || mask;
    const bool do_col = col_out != nullptr;
    if (do_row && cols % row_multiple(fmt) != 0)
        return FQ_ERR_SHAPE;
    if (do_col) {
        const int64_t rm = fmt == FQ_NVFP4_2LEVEL ? 128 : block_len(fmt);
        if (rows % rm != 0 || cols % 16 != 0)
            return FQ_ERR_SHAPE;

    }
    fq_status st = check_pitch(rows, cols, ld, x_dtype == FQ_BF16 ? 2 : 4);
    if (st != FQ_OK)
        return st;
    if (!aligned16(x) || (xhat && !aligned16(xhat)) || (mask && !aligned16(mask)) ||
        (amax_in && (reinterpret_cast<uintptr_t>(amax_in) & 3u)))
        return FQ_ERR_ALIGN;
    if (want_row_q && (st = check_q(row_out, fmt)) != FQ_OK)
        return st;
    if (do_col && (st = check_q(col_out, fmt)) != FQ_OK)
        return st;
    if (xhat && !valid_dtype(xhat_dtype))
        return FQ_ERR_INVALID_ARG;
    const float *amax = amax_in;
    if (fmt == FQ_NVFP4 && !amax_in) {
        if (!ws || ws_bytes < sizeof(float))
            return FQ_ERR_WORKSPACE;
        if (!aligned16(ws))
            return FQ_ERR_ALIGN;
    }
    const int64_t n = rows * cols;
    if (n == 0)
        return FQ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int bf16 = x_dtype == FQ_BF16;
    if (fmt == FQ_NVFP4 && !amax_in) {
        cudaError_t e = ld == cols ? launch_amax(x, bf16, n, static_cast<float *>(ws), s)
                                   : launch_amax_rows(x, bf16, rows, cols, ld,
                                                      static_cast<float *>(ws), s);
        if (e != cudaSuccess)
            return FQ_ERR_CUDA;
        amax = static_cast<const float *>(ws);
    }
    if (!do_col) {
        RowArgs a{};
        a.x = x;
        a.n = n;
        a.cols = cols;
        a.ld = ld;
        a.amax = amax;
        if (want_row_q) {
            a.codes = row_out->codes;
            a.scales = row_out->scales;
            a.tscale = row_out->tscale;
        }
        a.xhat = xhat;
        a.xhat_bf16 = xhat_dtype == FQ_BF16;
        a.mask = mask;
        a.seed = cfg->seed;
        a.offset = cfg->offset;
        a.stream_id = 0;
        a.rht_seed = cfg->rht_seed;
        a.key = philox_key(cfg->seed);
        return cuda_status(launch_row(a, bf16, fmt, cfg->rounding, s));
    }
    TileArgs t{};
    t.x = x;
    t.rows = rows;
    t.cols = cols;
    t.ld = ld;
    t.amax = amax;
    t.do_row = do_row ? 1 : 0;
    if (want_row_q) {
        t.rcodes = row_out->codes;
        t.rscales = row_out->scales;
        t.rtscale = row_out->tscale;
    }
    t.xhat = xhat;
    t.xhat_bf16 = xhat_dtype == FQ_BF16;
    t.mask = mask;
    t.ccodes = col_out->codes;
    t.cscales = col_out->scales;
    t.ctscale = col_out->tscale;
    t.seed = cfg->seed;
    t.offset = cfg->offset;
    t.rht_seed = cfg->rht_seed;
    t.key = philox_key(cfg->seed);
    return cuda_status(launch_tile(t, bf16, fmt, cfg->rounding, s));
}

fq_status check_group(int32_t ntensors, const int64_t *rows, const int64_t *cols, int fmt)
{
    if (ntensors < 0 || (ntensors > 0 && (!rows || !cols)))
        return FQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < ntensors; ++i) {
        if (rows[i] < 0 || cols[i] < 0)
            return FQ_ERR_SHAPE;
        if (cols[i] % row_multiple(fmt) != 0)
            return FQ_ERR_SHAPE;
    }
    return FQ_OK;
}

// Fills the tile prefix table of one group [i0, i0 + cnt).
void fill_tiles(OsciArgs &a, const int64_t *rows, const int64_t *cols, int32_t i0, int32_t cnt)
{
    a.ntensors = cnt;
    a.tile_start[0] = 0;
    for (int32_t j = 0; j < cnt; ++j) {
        const int64_t n = rows[i0 + j] * cols[i0 + j];
        a.t[j].n = n;
        const int64_t nch = n / 4;
        a.tile_start[j + 1] = a.tile_start[j] + (nch + kOsciTileChunks - 1) / kOsciTileChunks;
    }
}

}  // namespace

static fq_status osci_update_impl(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                         const int64_t *cols, float *const *master, const float *const *delta,
                         float *const *dist_q, float *const *dist_m, const fq_qtensor *prev,
                         const fq_qtensor *next, void *const *xhat, int32_t xhat_dtype,
                         uint8_t *const *mask, void *workspace, size_t workspace_bytes,
                         void *stream, int reset, float threshold, unsigned long long *n_reset)
{
    if (!valid_cfg(cfg))
        return FQ_ERR_INVALID_ARG;
    if (cfg->rht_seed)
        return FQ_ERR_UNSUPPORTED;
    const int fmt = cfg->format;
    fq_status st = check_group(ntensors, rows, cols, fmt);
    if (st != FQ_OK)
        return st;
    if (ntensors == 0)
        return FQ_OK;
    if (!master || !delta || !dist_q || !dist_m || !prev || !next)
        return FQ_ERR_INVALID_ARG;
    if (xhat && !valid_dtype(xhat_dtype))
        return FQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < ntensors; ++i) {
        if (!master[i] || !delta[i] || !dist_q[i] || !dist_m[i])
            return FQ_ERR_INVALID_ARG;
        if (!aligned16(master[i]) || !aligned16(delta[i]) || !aligned16(dist_q[i]) ||
            !aligned16(dist_m[i]) || (xhat && xhat[i] && !aligned16(xhat[i])) ||
            (mask && mask[i] && !aligned16(mask[i])))
            return FQ_ERR_ALIGN;
        if ((st = check_q(&prev[i], fmt)) != FQ_OK || (st = check_q(&next[i], fmt)) != FQ_OK)
            return st;
    }
    if (!workspace || workspace_bytes < fq_osci_workspace_size(ntensors))
        return FQ_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return FQ_ERR_ALIGN;
    if (n_reset && (reinterpret_cast<uintptr_t>(n_reset) & 7u))
        return FQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (reset && n_reset && cudaMemsetAsync(n_reset, 0, sizeof(unsigned long long), s) != cudaSuccess)
        return FQ_ERR_CUDA;
    static thread_local OsciArgs a;
    for (int32_t i0 = 0; i0 < ntensors; i0 += kOsciMaxTensors) {
        const int32_t cnt = ntensors - i0 < kOsciMaxTensors ? ntensors - i0 : kOsciMaxTensors;
        std::memset(&a, 0, sizeof(a));
        fill_tiles(a, rows, cols, i0, cnt);
        a.xhat_bf16 = xhat_dtype == FQ_BF16;
        a.reset = reset;
        a.threshold = threshold;
        a.n_reset = reset ? n_reset : nullptr;
        a.seed = cfg->seed;
        a.offset = cfg->offset;
        a.key = philox_key(cfg->seed);
        a.amax = static_cast<float *>(workspace);
        for (int32_t j = 0; j < cnt; ++j) {
            const int32_t i = i0 + j;
            OsciTensor &t = a.t[j];
            t.master = master[i];
            t.delta = delta[i];
            t.dist_q = dist_q[i];
            t.dist_m = dist_m[i];
            t.pcodes = prev[i].codes;
            t.pscales = prev[i].scales;
            t.ptscale = prev[i].tscale;
            t.ncodes = next[i].codes;
            t.nscales = next[i].scales;
            t.ntscale = next[i].tscale;
            t.xhat = xhat ? xhat[i] : nullptr;
            t.mask = mask ? mask[i] : nullptr;
        }
        cudaError_t e = launch_osci_update(a, fmt, cfg->rounding, s);
        if (e != cudaSuccess)
            return FQ_ERR_CUDA;
    }
    return FQ_OK;
}


extern "C" {

size_t fq_workspace_size(const fq_config *cfg, int64_t rows, int64_t cols)
{
    (void)rows;
    (void)cols;
    if (!valid_cfg(cfg))
        return 0;
    return cfg->format == FQ_NVFP4 ? kWsAmaxBytes : 0;
}

size_t fq_osci_workspace_size(int32_t ntensors)
{
    if (ntensors <= 0)
        return 0;
    const int32_t g = ntensors < kOsciMaxTensors ? ntensors : kOsciMaxTensors;
    return ((size_t)g * sizeof(float) + 255) / 256 * 256;
}

fq_status fq_amax(const void *x, int32_t x_dtype, int64_t n, float *amax_out, void *stream)
{
    if (!x || !amax_out || !valid_dtype(x_dtype))
        return FQ_ERR_INVALID_ARG;
    if (n < 0 || n % 8 != 0)
        return FQ_ERR_SHAPE;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax_out) & 3u))
        return FQ_ERR_ALIGN;
    return cuda_status(launch_amax(x, x_dtype == FQ_BF16, n, amax_out,
                                   static_cast<cudaStream_t>(stream)));
}

fq_status fq_quantize(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                      int64_t cols, int64_t ld, int32_t orient, const fq_qtensor *row_out,
                      const fq_qtensor *col_out, const float *amax_in, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    if (orient != FQ_ROW && orient != FQ_COL && orient != FQ_ROWCOL)
        return FQ_ERR_INVALID_ARG;
    const bool want_row = (orient & FQ_ROW) != 0;
    const bool want_col = (orient & FQ_COL) != 0;
    if ((want_row && !row_out) || (want_col && !col_out))
        return FQ_ERR_INVALID_ARG;
    return quantize_common(cfg, x, x_dtype, rows, cols, ld, want_row, row_out,
                           want_col ? col_out : nullptr, nullptr, FQ_F32, nullptr, amax_in,
                           workspace, workspace_bytes, stream);
}

fq_status fq_fakequant_ste(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                           int64_t cols, int64_t ld, void *xhat, int32_t xhat_dtype, uint8_t *mask,
                           const fq_qtensor *row_out, const fq_qtensor *col_out,
                           const float *amax_in, void *workspace, size_t workspace_bytes,
                           void *stream)
{
    if (!xhat)
        return FQ_ERR_INVALID_ARG;
    return quantize_common(cfg, x, x_dtype, rows, cols, ld, row_out != nullptr, row_out, col_out,
                           xhat, xhat_dtype, mask, amax_in, workspace, workspace_bytes, stream);
}

fq_status fq_dequantize(const fq_config *cfg, const fq_qtensor *q, int64_t rows, int64_t cols,
                        void *y, int32_t y_dtype, int64_t ldy, void *stream)
{
    if (!valid_cfg(cfg) || !y || !valid_dtype(y_dtype))
        return FQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % row_multiple(cfg->format) != 0)
        return FQ_ERR_SHAPE;
    fq_status st = check_pitch(rows, cols, ldy, y_dtype == FQ_BF16 ? 2 : 4);
    if (st != FQ_OK)
        return st;
    st = check_q(q, cfg->format);
    if (st != FQ_OK)
        return st;
    if (!aligned16(y))
        return FQ_ERR_ALIGN;
    DequantArgs a{};
    a.codes = q->codes;
    a.scales = q->scales;
    a.tscale = q->tscale;
    a.n = rows * cols;
    a.cols = cols;
    a.ldy = ldy;
    a.y = y;
    a.y_bf16 = y_dtype == FQ_BF16;
    return cuda_status(launch_dequant(a, cfg->format, static_cast<cudaStream_t>(stream)));
}

fq_status fq_ste_backward(const void *dy, int32_t dtype, const uint8_t *mask, int64_t n,
                          void *dx, void *stream)
{
    if (!dy || !mask || !dx || !valid_dtype(dtype))
        return FQ_ERR_INVALID_ARG;
    if (n < 0 || n % 8 != 0)
        return FQ_ERR_SHAPE;
    if (!aligned16(dy) || !aligned16(dx))
        return FQ_ERR_ALIGN;
    return cuda_status(
        launch_ste(dy, dtype == FQ_BF16, mask, n, dx, static_cast<cudaStream_t>(stream)));
}

fq_status fq_osci_update(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                         const int64_t *cols, float *const *master, const float *const *delta,
                         float *const *dist_q, float *const *dist_m, const fq_qtensor *prev,
                         const fq_qtensor *next, void *const *xhat, int32_t xhat_dtype,
                         uint8_t *const *mask, void *workspace, size_t workspace_bytes,
                         void *stream)
{
    return osci_update_impl(cfg, ntensors, rows, cols, master, delta, dist_q, dist_m, prev, next,
                            xhat, xhat_dtype, mask, workspace, workspace_bytes, stream, 0, 0.0f,
                            nullptr);
}

fq_status fq_osci_update_reset(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                               const int64_t *cols, float *const *master,
                               const float *const *delta, float *const *dist_q,
                               float *const *dist_m, const fq_qtensor *prev,
                               const fq_qtensor *next, void *const *xhat, int32_t xhat_dtype,
                               uint8_t *const *mask, float threshold,
                               unsigned long long *n_reset, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    return osci_update_impl(cfg, ntensors, rows, cols, master, delta, dist_q, dist_m, prev, next,
                            xhat, xhat_dtype, mask, workspace, workspace_bytes, stream, 1,
                            threshold, n_reset);
}

fq_status fq_osci_reset(const fq_config *cfg, int32_t ntensors, const int64_t *rows,
                        const int64_t *cols, float *const *master, float *const *dist_q,
                        float *const *dist_m, const fq_qtensor *cur, float threshold,
                        unsigned long long *n_reset, void *stream)
{
    if (!valid_cfg(cfg))
        return FQ_ERR_INVALID_ARG;
    const int fmt = cfg->format;
    fq_status st = check_group(ntensors, rows, cols, fmt);
    if (st != FQ_OK)
        return st;
    if (ntensors > 0 && (!master || !dist_q || !dist_m || !cur))
        return FQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < ntensors; ++i) {
        if (!master[i] || !dist_q[i] || !dist_m[i])
            return FQ_ERR_INVALID_ARG;
        if (!aligned16(master[i]) || !aligned16(dist_q[i]) || !aligned16(dist_m[i]))
            return FQ_ERR_ALIGN;
        if ((st = check_q(&cur[i], fmt)) != FQ_OK)
            return st;
    }
    if (n_reset && (reinterpret_cast<uintptr_t>(n_reset) & 7u))
        return FQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n_reset && cudaMemsetAsync(n_reset, 0, sizeof(unsigned long long), s) != cudaSuccess)
        return FQ_ERR_CUDA;
    static thread_local OsciArgs a;
    for (int32_t i0 = 0; i0 < ntensors; i0 += kOsciMaxTensors) {
        const int32_t cnt = ntensors - i0 < kOsciMaxTensors ? ntensors - i0 : kOsciMaxTensors;
        std::memset(&a, 0, sizeof(a));
        fill_tiles(a, rows, cols, i0, cnt);
        a.threshold = threshold;
        a.n_reset = n_reset;
        for (int32_t j = 0; j < cnt; ++j) {
            const int32_t i = i0 + j;
            OsciTensor &t = a.t[j];
            t.master = master[i];
            t.dist_q = dist_q[i];
            t.dist_m = dist_m[i];
            t.pcodes = cur[i].codes;
            t.pscales = cur[i].scales;
            t.ptscale = cur[i].tscale;
        }
        cudaError_t e = launch_osci_reset(a, fmt, s);
        if (e != cudaSuccess)
            return FQ_ERR_CUDA;
    }
    return FQ_OK;
}

fq_status fq_channel_amax(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                          float *amax_inout, void *stream)
{
    if (!valid_dtype(x_dtype) || !x || !amax_inout)
        return FQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 16 != 0)
        return FQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(amax_inout))
        return FQ_ERR_ALIGN;
    return cuda_status(launch_channel_amax(x, x_dtype == FQ_BF16, rows, cols, amax_inout,
                                           static_cast<cudaStream_t>(stream)));
}

fq_status fq_select_channels(const float *channel_amax, int64_t cols, int64_t k, int32_t *idx,
                             uint32_t *bitmap, float *fp8_scale, void *stream)
{
    if (!channel_amax || !bitmap || (k > 0 && (!idx || !fp8_scale)))
        return FQ_ERR_INVALID_ARG;
    if (cols < 0 || cols > FQ_MAX_CHANNELS)
        return FQ_ERR_SHAPE;
    if (k < 0 || k > cols)
        return FQ_ERR_INVALID_ARG;
    if (!aligned16(channel_amax) || !aligned16(bitmap) || (idx && !aligned16(idx)) ||
        (fp8_scale && !aligned16(fp8_scale)))
        return FQ_ERR_ALIGN;
    if (cols == 0)
        return FQ_OK;
    return cuda_status(launch_select(channel_amax, (int)cols, (int)k, idx, bitmap, fp8_scale,
                                     static_cast<cudaStream_t>(stream)));
}

fq_status fq_quantize_outliers(const fq_config *cfg, const void *x, int32_t x_dtype, int64_t rows,
                               int64_t cols, const uint32_t *bitmap, int64_t k,
                               const float *fp8_scale, const fq_qtensor *out, uint8_t *fp8,
                               void *xhat, int32_t xhat_dtype, uint8_t *mask, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    if (!valid_cfg(cfg) || !valid_dtype(x_dtype) || !x || !bitmap || (k > 0 && !fp8_scale))
        return FQ_ERR_INVALID_ARG;
    if (xhat && !valid_dtype(xhat_dtype))
        return FQ_ERR_INVALID_ARG;
    const int fmt = cfg->format;
    if (cfg->rht_seed)
        return FQ_ERR_UNSUPPORTED;
    if (rows < 0 || cols < 0 || cols % row_multiple(fmt) != 0 || cols > FQ_MAX_CHANNELS)
        return FQ_ERR_SHAPE;
    if (k < 0 || k > cols)
        return FQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(bitmap) || (fp8_scale && !aligned16(fp8_scale)) ||
        (fp8 && !aligned16(fp8)) || (xhat && !aligned16(xhat)) || (mask && !aligned16(mask)))
        return FQ_ERR_ALIGN;
    fq_status st;
    if (out && (st = check_q(out, fmt)) != FQ_OK)
        return st;
    if (fmt == FQ_NVFP4) {
        if (!workspace || workspace_bytes < sizeof(float))
            return FQ_ERR_WORKSPACE;
        if (!aligned16(workspace))
            return FQ_ERR_ALIGN;
    }
    if (rows * cols == 0)
        return FQ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int bf16 = x_dtype == FQ_BF16;
    OutlierArgs a{};
    if (fmt == FQ_NVFP4) {
        float *am = static_cast<float *>(workspace);
        cudaError_t e = launch_masked_amax(x, bf16, rows, cols, bitmap, am, s);
        if (e != cudaSuccess)
            return FQ_ERR_CUDA;
        a.amax = am;
    }
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.bitmap = bitmap;
    a.k = k;
    a.fp8_scale = fp8_scale;
    if (out) {
        a.codes = out->codes;
        a.scales = out->scales;
        a.tscale = out->tscale;
    }
    a.fp8 = fp8;
    a.xhat = xhat;
    a.xhat_bf16 = xhat_dtype == FQ_BF16;
    a.mask = mask;
    a.seed = cfg->seed;
    a.offset = cfg->offset;
    a.key = philox_key(cfg->seed);
    return cuda_status(launch_outlier_quant(a, bf16, fmt, cfg->rounding, s));
}

fq_status fq_qad_kl(const void *teacher, const void *student, int32_t dtype, int64_t rows,
                    int64_t vocab, float temperature, float grad_scale, float *loss_rows,
                    float *loss_mean, void *dstudent, int32_t dstudent_dtype, int32_t *err,
                    void *stream)
{
    if (!valid_dtype(dtype) || (rows > 0 && (!teacher || !student || !loss_rows)))
        return FQ_ERR_INVALID_ARG;
    if (dstudent && !valid_dtype(dstudent_dtype))
        return FQ_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !(temperature < INFINITY) || !(fabsf(grad_scale) < INFINITY))
        return FQ_ERR_INVALID_ARG;
    if (rows < 0 || vocab <= 0 || vocab % 8 != 0)
        return FQ_ERR_SHAPE;
    if (!aligned16(teacher) || !aligned16(student) || !aligned16(loss_rows) ||
        (loss_mean && (reinterpret_cast<uintptr_t>(loss_mean) & 3u)) ||
        (dstudent && !aligned16(dstudent)) || (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return FQ_ERR_ALIGN;
    KlArgs a{};
    QadPlan plan{};
    if (!qad_plan(vocab, dtype == FQ_BF16 ? 2 : 4, &plan))
        return FQ_ERR_UNSUPPORTED;
    a.zt = teacher;
    a.zs = student;
    a.rows = rows;
    a.vocab = vocab;
    a.k2 = (float)(1.4426950408889634 / (double)temperature);
    a.gk = (float)((double)grad_scale / (double)temperature);
    a.loss_rows = loss_rows;
    a.dz = dstudent;
    a.dz_bf16 = dstudent_dtype == FQ_BF16;
    a.err = err;
    return cuda_status(launch_qad_kl(a, dtype == FQ_BF16, plan, loss_mean,
                                     static_cast<cudaStream_t>(stream)));
}

size_t fq_gemm_workspace_size(int64_t m, int64_t n, int64_t k)
{
    if (m < 0 || n < 0 || k < 0)
        return 0;
    return gemm_workspace_bytes(m, n, k);
}

fq_status fq_gemm(const fq_config *cfg, const fq_qtensor *a, const fq_qtensor *b, int64_t m,
                  int64_t n, int64_t k, void *c, int32_t c_dtype, void *workspace,
                  size_t workspace_bytes, int32_t *err, void *stream)
{
    if (!valid_cfg(cfg) || !c || !valid_dtype(c_dtype))
        return FQ_ERR_INVALID_ARG;
    if ((cfg->format != FQ_NVFP4 && cfg->format != FQ_MXFP4) || cfg->rht_seed)
        return FQ_ERR_UNSUPPORTED;
    fq_status st;
    if ((st = check_q(a, cfg->format)) != FQ_OK || (st = check_q(b, cfg->format)) != FQ_OK)
        return st;
    // k: the codes' row pitch (k / 2 bytes) must be a multiple of 16 for the tensor maps;
    // n: the epilogue stores 32-column chunks
    if (m < 0 || n < 0 || k < 0 || n % 32 || k % 32 || (m + 127) / 128 > 65535)
        return FQ_ERR_SHAPE;
    if (!aligned16(c) || (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return FQ_ERR_ALIGN;
    if (m == 0 || n == 0)
        return FQ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (k == 0)
        return cuda_status(cudaMemsetAsync(c, 0, (size_t)(m * n) * (c_dtype == FQ_BF16 ? 2 : 4), s));
    if (!workspace || workspace_bytes < gemm_workspace_bytes(m, n, k))
        return FQ_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return FQ_ERR_ALIGN;
    GemmArgs g{};
    g.a_codes = a->codes;
    g.a_scales = a->scales;
    g.b_codes = b->codes;
    g.b_scales = b->scales;
    g.tscale_a = cfg->format == FQ_NVFP4 ? a->tscale : nullptr;
    g.tscale_b = cfg->format == FQ_NVFP4 ? b->tscale : nullptr;
    g.m = m;
    g.n = n;
    g.k = k;
    g.c = c;
    g.c_bf16 = c_dtype == FQ_BF16;
    g.err = err;
    return cuda_status(launch_gemm(g, cfg->format, workspace, s));
}

const char *fq_status_string(fq_status status)
{
    switch (status) {
    case FQ_OK: return "ok";
    case FQ_ERR_INVALID_ARG: return "invalid argument";
    case FQ_ERR_SHAPE: return "shape is not a multiple of the block length";
    case FQ_ERR_ALIGN: return "pointer is not 16-byte aligned";
    case FQ_ERR_WORKSPACE: return "workspace missing or too small";
    case FQ_ERR_UNSUPPORTED: return "unsupported combination";
    case FQ_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

}  // extern "C"
