// head.cu -- the rest of the CosmoFlow network around the conv stack: fully
// connected layers with leaky ReLU and dropout, the mean squared error, and the
// Adam update (hybrid-parallelism page, section IV and Table I: fc1 2048 ->
// fc2 256 -> fc3 4, leaky ReLU except after the last layer, dropout with keep
// probability 0.8, MSE loss, Adam with beta1 0.9, beta2 0.999, eps 1e-8).
//
// At the pages' batch sizes these layers are matrix-vector shaped (a handful
// of rows against a 2048 x 2048 weight): the weights' bytes, not the MACs,
// set their time, so they are plain SIMT kernels that read each weight once
// per launch, with fixed-order reductions.  Activations and weights are fp32;
// the first layer may read the stack's bf16 output directly and the last
// backward may write the stack's bf16 input gradient.
#include <algorithm>

#include "cf_internal.h"
#include "cf_ptx.cuh"

namespace cf {

__device__ __forceinline__ float load_x(const void* x, int is_bf16, int64_t i) {
    if (is_bf16) return bf16_bits_to_float(static_cast<const uint16_t*>(x)[i]);
    return static_cast<const float*>(x)[i];
}

// One warp per output column j, rows in groups of 8: lanes stride over k
// (fixed order), a butterfly sums the lanes.  y[i][j] = act(x[i] . w[j] + b[j])
// * (mask[i][j] ? 1/keep : 0) (no mask: 1).
__global__ void fc_fwd_kernel(int64_t M, int K, int N, const void* __restrict__ x, int x_bf16,
                              const float* __restrict__ w, const float* __restrict__ b, int act, float slope,
                              const uint8_t* __restrict__ mask, float keep, float* __restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t j = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); j < N; j += warps) {
        const float* wr = w + j * (int64_t)K;
        for (int64_t i0 = 0; i0 < M; i0 += 8) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k = lane; k < K; k += 32) {
                const float wv = wr[k];
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (i0 + r < M) acc[r] = fmaf(wv, load_x(x, x_bf16, (i0 + r) * K + k), acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
            if (lane < 8 && i0 + lane < M) {
                float v = 0.f;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r == lane) v = acc[r];
                v += b ? b[j] : 0.f;
                if (act) v = v > 0.f ? v : slope * v;
                if (mask) v = mask[(i0 + lane) * N + j] ? v / keep : 0.f;
                y[(i0 + lane) * N + j] = v;
            }
        }
    }
}

// Gradient at the pre-activation of output (i, j): dy * mask/keep * LReLU'(h)
// for a hidden layer (h its stored output, after dropout), dy for a linear one.
__device__ __forceinline__ float fc_dpre(const float* __restrict__ dy, const float* __restrict__ h,
                                         const uint8_t* __restrict__ mask, float keep, float slope, int64_t o) {
    float g = dy[o];
    if (mask) g = mask[o] ? g / keep : 0.f;
    if (h) g *= h[o] > 0.f ? 1.f : slope;
    return g;
}

// dW[j][k] = sum_i dpre[i][j] x[i][k] (rows in order), db[j] = sum_i dpre[i][j].
__global__ void fc_bwd_w_kernel(int64_t M, int K, int N, const void* __restrict__ x, int x_bf16,
                                const float* __restrict__ dy, const float* __restrict__ h,
                                const uint8_t* __restrict__ mask, float keep, float slope, float* __restrict__ dw,
                                float* __restrict__ db) {
    const int64_t total = (int64_t)N * K;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = e / K, k = e - j * K;
        float acc = 0.f, sb = 0.f;
        for (int64_t i = 0; i < M; ++i) {
            const float g = fc_dpre(dy, h, mask, keep, slope, i * N + j);
            acc = fmaf(g, load_x(x, x_bf16, i * K + k), acc);
            sb += g;
        }
        dw[e] = acc;
        if (db && k == 0) db[j] = sb;
    }
}

// dx[i][k] = sum_j dpre[i][j] w[j][k] (columns in order), fp32 or bf16.
__global__ void fc_bwd_x_kernel(int64_t M, int K, int N, const float* __restrict__ w, const float* __restrict__ dy,
                                const float* __restrict__ h, const uint8_t* __restrict__ mask, float keep, float slope,
                                void* __restrict__ dx, int dx_bf16) {
    const int64_t total = M * K;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / K, k = e - i * K;
        float acc = 0.f;
        for (int j = 0; j < N; ++j) acc = fmaf(fc_dpre(dy, h, mask, keep, slope, i * N + j), w[(int64_t)j * K + k], acc);
        if (dx_bf16)
            static_cast<uint16_t*>(dx)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        else
            static_cast<float*>(dx)[e] = acc;
    }
}

// loss = mean of (pred - target)^2 over `count` values, dpred = 2 (pred - target)
// / count; one block, fixed-shape tree.
__global__ void mse_kernel(int64_t count, const float* __restrict__ pred, const float* __restrict__ target,
                           float* __restrict__ loss, float* __restrict__ dpred) {
    __shared__ float red[256];
    float s = 0.f;
    for (int64_t i = threadIdx.x; i < count; i += blockDim.x) {
        const float d = pred[i] - target[i];
        s = fmaf(d, d, s);
        if (dpred) dpred[i] = 2.f * d / (float)count;
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int k = blockDim.x / 2; k > 0; k >>= 1) {
        if ((int)threadIdx.x < k) red[threadIdx.x] += red[threadIdx.x + k];
        __syncthreads();
    }
    if (threadIdx.x == 0 && loss) *loss = red[0] / (float)count;
}

// Adam with bias correction (step t >= 1), fp32 master weights; w16, when
// given, receives the updated weights rounded to bf16 (the conv kernels' copy).
__global__ void adam_kernel(int64_t count, float* __restrict__ w, uint16_t* __restrict__ w16,
                            const float* __restrict__ g, float* __restrict__ m, float* __restrict__ v, float lr,
                            float beta1, float beta2, float eps, float c1, float c2) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        const float gi = g[i];
        const float mi = beta1 * m[i] + (1.f - beta1) * gi;
        const float vi = beta2 * v[i] + (1.f - beta2) * gi * gi;
        m[i] = mi;
        v[i] = vi;
        const float wi = w[i] - lr * (mi / c1) / (sqrtf(vi / c2) + eps);
        w[i] = wi;
        if (w16) w16[i] = __bfloat16_as_ushort(__float2bfloat16_rn(wi));
    }
}

static int grid_1d(const LaunchCtx& ctx, int64_t total, int threads) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 16LL * ctx.num_sms));
}

cf_status launch_fc_fwd(const LaunchCtx& ctx, int64_t m, int k, int n, const void* x, int x_bf16, const float* w,
                        const float* b, int act, float slope, const uint8_t* mask, float keep, float* y) {
    const int warps_per_block = 8;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + warps_per_block - 1) / warps_per_block,
                                                                   32LL * ctx.num_sms));
    fc_fwd_kernel<<<blocks, 32 * warps_per_block, 0, ctx.stream>>>(m, k, n, x, x_bf16, w, b, act, slope, mask, keep, y);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_fc_bwd(const LaunchCtx& ctx, int64_t m, int k, int n, const void* x, int x_bf16, const float* w,
                        const float* h, const uint8_t* mask, float keep, float slope, const float* dy, void* dx,
                        int dx_bf16, float* dw, float* db) {
    if (dw) {
        fc_bwd_w_kernel<<<grid_1d(ctx, (int64_t)n * k, 256), 256, 0, ctx.stream>>>(m, k, n, x, x_bf16, dy, h, mask,
                                                                                     keep, slope, dw, db);
        if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    }
    if (dx) {
        fc_bwd_x_kernel<<<grid_1d(ctx, m * k, 256), 256, 0, ctx.stream>>>(m, k, n, w, dy, h, mask, keep, slope, dx,
                                                                           dx_bf16);
        if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    }
    return CF_OK;
}

cf_status launch_mse(const LaunchCtx& ctx, int64_t count, const float* pred, const float* target, float* loss,
                     float* dpred) {
    mse_kernel<<<1, 256, 0, ctx.stream>>>(count, pred, target, loss, dpred);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_adam(const LaunchCtx& ctx, int64_t count, float* w, uint16_t* w16, const float* g, float* m, float* v,
                      float lr, float beta1, float beta2, float eps, int64_t t) {
    const float c1 = (float)(1.0 - pow((double)beta1, (double)t));
    const float c2 = (float)(1.0 - pow((double)beta2, (double)t));
    adam_kernel<<<grid_1d(ctx, count, 256), 256, 0, ctx.stream>>>(count, w, w16, g, m, v, lr, beta1, beta2, eps, c1,
                                                                   c2);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

}  // namespace cf

using namespace cf;

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" {

cf_status cf_fc_fwd(int64_t m, int32_t k, int32_t n, const void* x, int32_t x_is_bf16, const float* w,
                    const float* b, int32_t act, float slope, const uint8_t* keep_mask, float keep, float* y,
                    void* stream) {
    if (m <= 0 || k <= 0 || n <= 0 || !x || !w || !y) return CF_ERR_INVALID_ARG;
    if (!al16(x) || !al16(w) || !al16(y) || (b && !al16(b)) || (keep_mask && !al16(keep_mask)))
        return CF_ERR_INVALID_ARG;
    if (keep_mask && !(keep > 0.f && keep <= 1.f)) return CF_ERR_INVALID_ARG;
    LaunchCtx ctx;
    if (!cf_device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_fc_fwd(ctx, m, k, n, x, x_is_bf16, w, b, act, slope, keep_mask, keep, y);
}

cf_status cf_fc_bwd(int64_t m, int32_t k, int32_t n, const void* x, int32_t x_is_bf16, const float* w, const float* h,
                    float slope, const uint8_t* keep_mask, float keep, const float* dy, void* dx, int32_t dx_is_bf16,
                    float* dw, float* db, void* stream) {
    if (m <= 0 || k <= 0 || n <= 0 || !x || !w || !dy) return CF_ERR_INVALID_ARG;
    if (!al16(x) || !al16(w) || !al16(dy) || (h && !al16(h)) || (keep_mask && !al16(keep_mask)) ||
        (dx && !al16(dx)) || (dw && !al16(dw)) || (db && !al16(db)))
        return CF_ERR_INVALID_ARG;
    if (keep_mask && !(keep > 0.f && keep <= 1.f)) return CF_ERR_INVALID_ARG;
    LaunchCtx ctx;
    if (!cf_device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_fc_bwd(ctx, m, k, n, x, x_is_bf16, w, h, keep_mask, keep, slope, dy, dx, dx_is_bf16, dw, db);
}

cf_status cf_mse(int64_t count, const float* pred, const float* target, float* loss, float* dpred, void* stream) {
    if (count <= 0 || !pred || !target) return CF_ERR_INVALID_ARG;
    LaunchCtx ctx;
    if (!cf_device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_mse(ctx, count, pred, target, loss, dpred);
}

cf_status cf_adam_step(int64_t count, float* w, uint16_t* w_bf16, const float* g, float* m, float* v, float lr,
                       float beta1, float beta2, float eps, int64_t t, void* stream) {
    if (count <= 0 || !w || !g || !m || !v || t < 1) return CF_ERR_INVALID_ARG;
    if (!(beta1 >= 0.f && beta1 < 1.f && beta2 >= 0.f && beta2 < 1.f)) return CF_ERR_INVALID_ARG;
    LaunchCtx ctx;
    if (!cf_device_ctx(&ctx, stream)) return CF_ERR_CUDA;
    return launch_adam(ctx, count, w, w_bf16, g, m, v, lr, beta1, beta2, eps, t);
}

}  // extern "C"
