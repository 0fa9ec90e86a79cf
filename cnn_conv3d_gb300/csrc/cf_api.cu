// cf_api.cu -- the C ABI of libcfconv3d.so (declared in include/cf_conv3d.h):
// argument validation, workspace layout, per-device context (SM count,
// device status word, tensor-map encoder) and the launch sequence of each
// operation.  No entry point allocates or frees device memory.
#include <algorithm>
#include <mutex>

#include "cf_internal.h"
#include "cf_ptx.cuh"

namespace cf {

__device__ int g_status;  // device status word (0 = OK)

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
int g_num_sms[kMaxDevices] = {0};
int* g_status_ptr[kMaxDevices] = {nullptr};
uint64_t g_wait_ns = 2000000000ull;

// Per-device set-up, once: SM count and the device address of the status word.
bool device_ctx(LaunchCtx* ctx, void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_num_sms[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return false;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return false;
        g_status_ptr[dev] = static_cast<int*>(p);
        g_num_sms[dev] = sms;
    }
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return false;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->num_sms = g_num_sms[dev];
    ctx->status = g_status_ptr[dev];
    ctx->wait_ns = g_wait_ns;
    return true;
}

}  // namespace

// The per-device launch context for the other translation units' entry points.
bool cf_device_ctx(LaunchCtx* ctx, void* stream) { return device_ctx(ctx, stream); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int desc_stride(const cf_conv_desc* d) { return d->stride == 2 ? 2 : 1; }

bool desc_ok(const cf_conv_desc* d) {
    if (d == nullptr) return false;
    if (d->n <= 0 || d->d <= 0 || d->h <= 0 || d->w <= 0 || d->c_in <= 0 || d->c_out <= 0) return false;
    if (d->stride < 0 || d->stride > 2) return false;
    // every index the kernels form stays below 2^31 per dimension and 2^62 in total
    if (d->d > (1 << 20) || d->h > (1 << 20) || d->w > (1 << 20) || d->n > (1 << 24)) return false;
    const double elems = (double)d->n * d->d * d->h * d->w * (double)(d->c_in > d->c_out ? d->c_in : d->c_out);
    return elems < 4.0e18;
}

int64_t dense_grad_elems(const cf_conv_desc* d) { return d->n * d->d * d->h * d->w * (int64_t)d->c_out; }

// Workspace bytes of the zero-inserted output gradient of a stride-2 conv
// (input sizes x c_out bf16), 0 for stride 1.
size_t upsample_bytes(const cf_conv_desc* d) {
    return desc_stride(d) == 2 ? round_up((size_t)dense_grad_elems(d) * 2, 256) : 0;
}

}  // namespace

bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz,
                 const uint32_t* elem_strides) {
    if (g_encode == nullptr) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = elem_strides ? elem_strides[i] : 1;
        if (i < rank - 1) gs[i] = strides_bytes[i];
    }
    CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace cf

using namespace cf;

extern "C" {

const char* cf_status_string(cf_status s) {
    switch (s) {
        case CF_OK: return "ok";
        case CF_ERR_INVALID_ARG: return "invalid argument";
        case CF_ERR_UNSUPPORTED: return "unsupported shape or layout";
        case CF_ERR_WORKSPACE: return "workspace too small";
        case CF_ERR_CUDA: return "CUDA error";
        case CF_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

cf_status cf_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return CF_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    g_wait_ns = ns;
    return CF_OK;
}

cf_status cf_last_device_status(void* stream) {
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    if (cudaStreamSynchronize(ctx.stream) != cudaSuccess) return CF_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ctx.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CF_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CF_ERR_CUDA;
        return CF_ERR_TIMEOUT;
    }
    return CF_OK;
}

cf_status cf_debug_wait_timeout_probe(void* stream) {
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_timeout_probe(ctx);
}

// Workspace of cf_conv3d_dgrad after the flipped filter: the channel-sum
// partials (whichever of the fused rows or the separate pass is larger).
static size_t dgrad_sum_bytes(int num_sms, int c_in) {
    return round_up(std::max((size_t)num_sms * c_in * sizeof(float), channel_sums_workspace_bytes(num_sms, c_in)),
                    256);
}

size_t cf_workspace_size(int op, const cf_conv_desc* desc) {
    if (!desc_ok(desc)) return 0;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, nullptr)) return 0;
    const size_t wt = round_up((size_t)desc->c_out * 27 * desc->c_in * 2, 256);
    const size_t dense = round_up((size_t)dense_grad_elems(desc) * 2, 256);
    const size_t part = round_up(
        wgrad_workspace_bytes(ctx.num_sms, desc->n, desc->d, desc->h, desc->w, desc->c_in, desc->c_out), 256);
    const size_t up = upsample_bytes(desc);
    switch (op) {
        case CF_OP_FWD: return 0;
        case CF_OP_DGRAD: return wt + dgrad_sum_bytes(ctx.num_sms, desc->c_in) + up;
        case CF_OP_DGRAD_ROUTED: return wt + dgrad_sum_bytes(ctx.num_sms, desc->c_in) + dense;
        case CF_OP_WGRAD: return part + up;
        case CF_OP_WGRAD_ROUTED: return part + (wgrad_routed_fused(desc->c_in) ? 0 : dense);
        case CF_OP_POOL_BWD: return round_up(pool_bwd_workspace_bytes(ctx.num_sms, desc->c_out), 256);
        case CF_OP_BN: return round_up(bn_workspace_bytes(ctx.num_sms, desc->c_out), 256);
    }
    return 0;
}

cf_status cf_conv3d_fwd(const cf_conv_desc* desc, const uint16_t* x, const uint16_t* w, const cf_pool_epi* epi,
                        uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
    (void)ws;
    (void)ws_bytes;
    if (!desc_ok(desc) || x == nullptr || w == nullptr || y == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return CF_ERR_INVALID_ARG;
    const int stride = desc_stride(desc);
    const int pool = epi ? epi->pool : CF_POOL_NONE;
    if (epi != nullptr) {
        if (pool < CF_POOL_MAX || pool > CF_POOL_NONE) return CF_ERR_INVALID_ARG;
        if ((epi->bias && !aligned16(epi->bias)) || (epi->argmax && !aligned16(epi->argmax)))
            return CF_ERR_INVALID_ARG;
        const int64_t od = (desc->d + stride - 1) / stride, oh = (desc->h + stride - 1) / stride,
                      ow = (desc->w + stride - 1) / stride;
        if (pool != CF_POOL_NONE && ((od | oh | ow) & 1)) return CF_ERR_UNSUPPORTED;
    }
    const int ci = desc->c_in, co = desc->c_out;
    const bool small = ci == 1 || ci == 4;
    if (!small && ci % 16 != 0) return CF_ERR_UNSUPPORTED;
    if (small && stride != 1) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    // epilogue: pooled (max / average), or plain with the optional activation
    const bool pooled = epi != nullptr && pool != CF_POOL_NONE;
    const int mode = pooled ? EPI_POOL : EPI_PLAIN;
    const int pool_kind = pool == CF_POOL_AVG ? 1 : 0;
    const int act = epi != nullptr && pool == CF_POOL_NONE ? 1 : 0;
    const float* bias = epi ? epi->bias : nullptr;
    uint8_t* idx = pooled ? epi->argmax : nullptr;
    const float slope = epi ? epi->slope : 0.f;
    if (small && mode == EPI_POOL && pool_kind == 0 && quad_path_supported(desc->d, desc->h, desc->w, ci, co))
        return launch_conv_quad(ctx, desc->n, desc->d, desc->h, desc->w, co, x, w, y, idx, bias, slope);
    if (small)
        return launch_conv_smallc(ctx, desc->n, desc->d, desc->h, desc->w, ci, co, x, w, mode, y, idx, bias, slope,
                                  pool_kind, act);
    if (stride == 1 && halo_path_supported(ci, co))
        return launch_conv_halo(ctx, desc->n, desc->d, desc->h, desc->w, ci, co, x, w, mode, y, idx, bias, nullptr,
                                slope, nullptr, pool_kind, act);
    return launch_conv_igemm(ctx, desc->n, desc->d, desc->h, desc->w, ci, co, x, w, mode, y, idx, bias, nullptr, slope,
                             pool_kind, act, stride);
}

// Backward data; prev_idx / prev_dz (both or neither): the previous block's
// max-pool backward fused into the epilogue (see cf_conv3d_dgrad_pool_bwd).
// w is the forward filter, or (flipped) already the backward-data filter.
static cf_status dgrad_impl(const cf_conv_desc* desc, const uint16_t* dz, const uint8_t* idx, const uint16_t* w,
                            const uint16_t* x_act, float slope, uint16_t* dx, float* dsum, const uint8_t* prev_idx,
                            uint16_t* prev_dz, void* ws, size_t ws_bytes, void* stream, bool flipped = false) {
    if (!desc_ok(desc) || dz == nullptr || w == nullptr || dx == nullptr) return CF_ERR_INVALID_ARG;
    if ((prev_idx == nullptr) != (prev_dz == nullptr)) return CF_ERR_INVALID_ARG;
    if ((prev_idx && !aligned16(prev_idx)) || (prev_dz && !aligned16(prev_dz))) return CF_ERR_INVALID_ARG;
    if (!aligned16(dz) || !aligned16(w) || !aligned16(dx) || (x_act && !aligned16(x_act)) ||
        (idx && !aligned16(idx)) || (ws && !aligned16(ws)) || (dsum && !aligned16(dsum)))
        return CF_ERR_INVALID_ARG;
    const int ci = desc->c_in, co = desc->c_out;
    if (co % 16 != 0 || ci % 16 != 0) return CF_ERR_UNSUPPORTED;
    if (idx && ((desc->d | desc->h | desc->w) & 1)) return CF_ERR_UNSUPPORTED;
    const int stride = desc_stride(desc);
    if (stride == 2 && idx) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    const size_t wt_bytes = round_up((size_t)co * 27 * ci * 2, 256);
    const size_t sum_bytes = dgrad_sum_bytes(ctx.num_sms, ci);
    const size_t need = wt_bytes + sum_bytes + (idx ? round_up((size_t)dense_grad_elems(desc) * 2, 256) : 0) +
                        upsample_bytes(desc);
    if (ws == nullptr || ws_bytes < need) return CF_ERR_WORKSPACE;
    const uint16_t* wt = w;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + wt_bytes);
    cf_status st = CF_OK;
    if (!flipped) {
        uint16_t* buf = static_cast<uint16_t*>(ws);
        st = launch_flip_transpose(ctx, co, ci, w, buf);
        if (st != CF_OK) return st;
        wt = buf;
    }
    const uint16_t* dz_dense = dz;
    if (stride == 2) {
        // zeros at the odd positions: the stride-2 backward as a stride-1 one
        uint16_t* buf = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + wt_bytes + sum_bytes);
        st = launch_upsample2(ctx, desc->n, desc->d, desc->h, desc->w, co, dz, buf);
        if (st != CF_OK) return st;
        dz_dense = buf;
    }
    if (idx) {
        uint16_t* buf = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + wt_bytes + sum_bytes);
        st = launch_pool_bwd(ctx, desc->n, desc->d, desc->h, desc->w, co, dz, nullptr, idx, 1.f, buf, nullptr,
                             nullptr, nullptr, 0);
        if (st != CF_OK) return st;
        dz_dense = buf;
    }
    // backward data = forward conv of dZ with the flipped, transposed filter:
    // GEMM input channels c_out, output channels c_in.  Channel sums of dx: in
    // the halo kernel's epilogue when c_in <= 32 (one row of partials per CTA,
    // rows of CTAs that get no tile stay zero), else a separate pass over dx.
    const int epi = x_act ? EPI_DGRAD : EPI_PLAIN;
    if (halo_path_supported(co, ci)) {
        const bool fused = dsum != nullptr && ci <= 32;
        if (fused && cudaMemsetAsync(part, 0, (size_t)ctx.num_sms * ci * sizeof(float), ctx.stream) != cudaSuccess)
            return CF_ERR_CUDA;
        st = launch_conv_halo(ctx, desc->n, desc->d, desc->h, desc->w, co, ci, dz_dense, wt, epi, dx, nullptr,
                              nullptr, x_act, slope, fused ? part : nullptr, 0, 0, prev_dz, prev_idx);
        if (st != CF_OK || dsum == nullptr) return st;
        if (fused) return launch_colsum(ctx, part, ctx.num_sms, ci, dsum);
    } else {
        st = launch_conv_igemm(ctx, desc->n, desc->d, desc->h, desc->w, co, ci, dz_dense, wt, epi, dx, nullptr,
                               nullptr, x_act, slope, 0, 0, 1, prev_dz, prev_idx);
        if (st != CF_OK || dsum == nullptr) return st;
    }
    return launch_channel_sums(ctx, dx, desc->n * desc->d * desc->h * desc->w, ci, part, dsum);
}

cf_status cf_conv3d_dgrad(const cf_conv_desc* desc, const uint16_t* dz, const uint8_t* idx, const uint16_t* w,
                          const uint16_t* x_act, float slope, uint16_t* dx, float* dsum, void* ws,
                          size_t ws_bytes, void* stream) {
    return dgrad_impl(desc, dz, idx, w, x_act, slope, dx, dsum, nullptr, nullptr, ws, ws_bytes, stream);
}

cf_status cf_conv3d_dgrad_flipped(const cf_conv_desc* desc, const uint16_t* dz, const uint8_t* idx,
                                  const uint16_t* wt, const uint16_t* x_act, float slope, uint16_t* dx, float* dsum,
                                  void* ws, size_t ws_bytes, void* stream) {
    return dgrad_impl(desc, dz, idx, wt, x_act, slope, dx, dsum, nullptr, nullptr, ws, ws_bytes, stream, true);
}

cf_status cf_filter_flip(int32_t c_out, int32_t c_in, const uint16_t* w, uint16_t* wt, void* stream) {
    if (w == nullptr || wt == nullptr || c_out <= 0 || c_in <= 0 || !aligned16(w) || !aligned16(wt))
        return CF_ERR_INVALID_ARG;
    if (c_out % 16 != 0 || c_in % 16 != 0) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_flip_transpose(ctx, c_out, c_in, w, wt);
}

cf_status cf_conv3d_dgrad_pool_bwd(const cf_conv_desc* desc, const uint16_t* dz, const uint16_t* w,
                                   const uint16_t* x_act, float slope, uint16_t* dx, float* dsum,
                                   const uint8_t* prev_idx, uint16_t* prev_dz, void* ws, size_t ws_bytes,
                                   void* stream) {
    if (prev_idx == nullptr || prev_dz == nullptr) return CF_ERR_INVALID_ARG;
    if (desc_stride(desc) != 1 || !desc_ok(desc)) return desc_ok(desc) ? CF_ERR_UNSUPPORTED : CF_ERR_INVALID_ARG;
    return dgrad_impl(desc, dz, nullptr, w, x_act, slope, dx, dsum, prev_idx, prev_dz, ws, ws_bytes, stream);
}

cf_status cf_conv3d_wgrad(const cf_conv_desc* desc, const uint16_t* x, const uint16_t* dz, const uint8_t* idx,
                          float* dw, int accumulate, void* ws, size_t ws_bytes, void* stream) {
    if (!desc_ok(desc) || x == nullptr || dz == nullptr || dw == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(dz) || !aligned16(dw) || (idx && !aligned16(idx)) || (ws && !aligned16(ws)))
        return CF_ERR_INVALID_ARG;
    if (idx && ((desc->d | desc->h | desc->w) & 1)) return CF_ERR_UNSUPPORTED;
    const int stride = desc_stride(desc);
    if (!wgrad_shape_supported(desc->c_in, desc->c_out)) return CF_ERR_UNSUPPORTED;
    if (stride == 2 && (idx || desc->c_in == 1 || desc->c_in == 4)) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    const size_t part = round_up(
        wgrad_workspace_bytes(ctx.num_sms, desc->n, desc->d, desc->h, desc->w, desc->c_in, desc->c_out), 256);
    const bool fused = idx && wgrad_routed_fused(desc->c_in);
    const size_t need = part + (idx && !fused ? round_up((size_t)dense_grad_elems(desc) * 2, 256) : 0) +
                        upsample_bytes(desc);
    if (ws == nullptr || ws_bytes < need) return CF_ERR_WORKSPACE;
    if (stride == 2) {
        uint16_t* buf = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + part);
        cf_status st = launch_upsample2(ctx, desc->n, desc->d, desc->h, desc->w, desc->c_out, dz, buf);
        if (st != CF_OK) return st;
        return launch_wgrad(ctx, desc->n, desc->d, desc->h, desc->w, desc->c_in, desc->c_out, x, buf, nullptr, dw,
                            accumulate, ws, part);
    }
    if (fused)
        return launch_wgrad(ctx, desc->n, desc->d, desc->h, desc->w, desc->c_in, desc->c_out, x, dz, idx, dw,
                            accumulate, ws, part);
    const uint16_t* dz_dense = dz;
    if (idx) {
        uint16_t* buf = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + part);
        cf_status st = launch_pool_bwd(ctx, desc->n, desc->d, desc->h, desc->w, desc->c_out, dz, nullptr, idx, 1.f,
                                       buf, nullptr, nullptr, nullptr, 0);
        if (st != CF_OK) return st;
        dz_dense = buf;
    }
    return launch_wgrad(ctx, desc->n, desc->d, desc->h, desc->w, desc->c_in, desc->c_out, x, dz_dense, nullptr, dw,
                        accumulate, ws, part);
}

cf_status cf_bias_lrelu_pool_fwd(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c, const uint16_t* z,
                                 const float* bias, float slope, uint16_t* y, uint8_t* idx, void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || z == nullptr || y == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(y) || (bias && !aligned16(bias)) || (idx && !aligned16(idx)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || ((d | h | w) & 1)) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_pool_fwd(ctx, n, d, h, w, c, z, bias, slope, y, idx);
}

cf_status cf_bias_lrelu_pool_bwd(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c, const uint16_t* dy,
                                 const uint16_t* y, const uint8_t* idx, float slope, uint16_t* dz, uint16_t* dy_pre,
                                 float* dbias, void* ws, size_t ws_bytes, void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || dy == nullptr) return CF_ERR_INVALID_ARG;
    if (dz != nullptr && idx == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(dy) || (y && !aligned16(y)) || (idx && !aligned16(idx)) || (dz && !aligned16(dz)) ||
        (dy_pre && !aligned16(dy_pre)) || (dbias && !aligned16(dbias)) || (ws && !aligned16(ws)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048 || ((d | h | w) & 1)) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_pool_bwd(ctx, n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, dbias, ws, ws_bytes);
}

cf_status cf_bias_lrelu_pool_bwd_partials(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c, const uint16_t* dy,
                                          const uint16_t* y, const uint8_t* idx, float slope, uint16_t* dz,
                                          uint16_t* dy_pre, float* partial, size_t partial_bytes, void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || dy == nullptr || partial == nullptr)
        return CF_ERR_INVALID_ARG;
    if (dz != nullptr && idx == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(dy) || (y && !aligned16(y)) || (idx && !aligned16(idx)) || (dz && !aligned16(dz)) ||
        (dy_pre && !aligned16(dy_pre)) || !aligned16(partial))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048 || ((d | h | w) & 1)) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_pool_bwd(ctx, n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, partial, partial, partial_bytes, false);
}

int64_t cf_pool_bwd_partial_rows(void) {
    LaunchCtx ctx;
    if (!device_ctx(&ctx, nullptr)) return 0;
    return (int64_t)(pool_bwd_workspace_bytes(ctx.num_sms, 1) / sizeof(float));
}

cf_status cf_column_sums(int64_t rows, int32_t c, const float* partial, float* out, void* stream) {
    if (rows <= 0 || rows > INT32_MAX || c <= 0 || partial == nullptr || out == nullptr) return CF_ERR_INVALID_ARG;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_colsum(ctx, partial, (int)rows, c, out);
}

cf_status cf_block_epilogue_fwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* aux,
                                void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || z == nullptr || y == nullptr) return CF_ERR_INVALID_ARG;
    if (pool < CF_POOL_MAX || pool > CF_POOL_NONE) return CF_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(y) || (bias && !aligned16(bias)) || (aux && !aligned16(aux)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || (pool != CF_POOL_NONE && ((d | h | w) & 1))) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    if (pool == CF_POOL_MAX) return launch_pool_fwd(ctx, n, d, h, w, c, z, bias, slope, y, aux);
    if (pool == CF_POOL_AVG) return launch_avgpool_fwd(ctx, n, d, h, w, c, z, bias, slope, y, aux);
    return launch_act_fwd(ctx, n * d * h * w * c, c, z, bias, slope, y);
}

cf_status cf_block_epilogue_bwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                const uint16_t* dy, const uint16_t* y, const uint8_t* aux, float slope,
                                uint16_t* dz, uint16_t* dy_pre, float* dbias, void* ws, size_t ws_bytes,
                                void* stream) {
    if (pool == CF_POOL_MAX)
        return cf_bias_lrelu_pool_bwd(n, d, h, w, c, dy, y, aux, slope, dz, dy_pre, dbias, ws, ws_bytes, stream);
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || dy == nullptr) return CF_ERR_INVALID_ARG;
    if (pool != CF_POOL_AVG && pool != CF_POOL_NONE) return CF_ERR_INVALID_ARG;
    if (dy_pre != nullptr) return CF_ERR_INVALID_ARG;  // max pooling only
    if (pool == CF_POOL_AVG && aux == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(dy) || (y && !aligned16(y)) || (aux && !aligned16(aux)) || (dz && !aligned16(dz)) ||
        (dbias && !aligned16(dbias)) || (ws && !aligned16(ws)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048 || (pool == CF_POOL_AVG && ((d | h | w) & 1))) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    if (pool == CF_POOL_AVG) return launch_avgpool_bwd(ctx, n, d, h, w, c, dy, aux, slope, dz, dbias, ws, ws_bytes);
    return launch_act_bwd(ctx, n * d * h * w * c, c, dy, y, slope, dz, dbias, ws, ws_bytes);
}

cf_status cf_bn_stats(int64_t rows, int32_t c, const uint16_t* z, float* sums, void* ws, size_t ws_bytes,
                      void* stream) {
    if (rows <= 0 || c <= 0 || z == nullptr || sums == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(sums) || (ws && !aligned16(ws))) return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_channel_stats(ctx, rows, c, z, sums, ws, ws_bytes);
}

cf_status cf_bn_act_pool_fwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c, const uint16_t* z,
                             const float* sums, const float* gamma, const float* beta, float eps, float slope,
                             uint16_t* y, uint8_t* aux, void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || !z || !sums || !gamma || !beta || !y)
        return CF_ERR_INVALID_ARG;
    if (pool < CF_POOL_MAX || pool > CF_POOL_NONE || !(eps >= 0.f)) return CF_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(y) || !aligned16(sums) || (aux && !aligned16(aux))) return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || (pool != CF_POOL_NONE && ((d | h | w) & 1))) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_bn_act_pool_fwd(ctx, pool, n, d, h, w, c, z, sums, gamma, beta, eps, slope, y, aux);
}

cf_status cf_bn_act_pool_bwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                             const uint16_t* dy, const uint16_t* y, const uint8_t* aux, const uint16_t* z,
                             const float* sums, const float* gamma, float eps, float slope, uint16_t* dz,
                             float* dsums, void* ws, size_t ws_bytes, void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || !dy || !z || !sums || !gamma || !dz || !dsums)
        return CF_ERR_INVALID_ARG;
    if (pool < CF_POOL_MAX || pool > CF_POOL_NONE || !(eps >= 0.f)) return CF_ERR_INVALID_ARG;
    if (pool != CF_POOL_NONE && aux == nullptr) return CF_ERR_INVALID_ARG;
    if (!aligned16(dy) || (y && !aligned16(y)) || (aux && !aligned16(aux)) || !aligned16(z) || !aligned16(dz) ||
        !aligned16(dsums) || (ws && !aligned16(ws)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048 || (pool != CF_POOL_NONE && ((d | h | w) & 1))) return CF_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_bn_act_pool_bwd(ctx, pool, n, d, h, w, c, dy, y, aux, z, sums, gamma, eps, slope, dz, dsums, ws,
                                  ws_bytes);
}

}  // extern "C"
