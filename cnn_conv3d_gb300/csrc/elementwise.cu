// elementwise.cu -- the HBM-bound pieces of the block: standalone bias +
// leaky ReLU + 2x2x2 max-pool (forward), its argmax-routed backward with the
// bias gradient, the filter flip/transpose that turns backward-data into a
// forward convolution, and the wait-timeout probe.
//
// Pooling (CosmoFlow page, section III-C: pooling works per channel over
// KS^3 windows; hybrid-parallelism page, Table I: stride-2 pooling) is the
// max over each 2x2x2 window; the code of the first maximum in (dd,dh,dw)
// order (dd*4+dh*2+dw) is kept for the backward pass.
#include <algorithm>

#include "cf_internal.h"
#include "cf_ptx.cuh"
#include "fastdiv.cuh"

namespace cf {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// Pooled voxel index -> (n, pd, ph, pw) of the pooled grid [N][D2][H2][W2]:
// multiply-shift division by the launch-time extents while the index fits 32
// bits (every realistic case), 64-bit division beyond.
struct PoolGrid {
    FastDiv w2, h2, d2;
};
__device__ __forceinline__ void pool_decode(const PoolGrid& g, int64_t pvox, int64_t& n, int& pd, int& ph, int& pw) {
    if (pvox < (int64_t)0xFFFFFFFF) {
        uint32_t m = (uint32_t)pvox, q = g.w2.div(m);
        pw = (int)(m - q * g.w2.d);
        m = q;
        q = g.h2.div(m);
        ph = (int)(m - q * g.h2.d);
        m = q;
        q = g.d2.div(m);
        pd = (int)(m - q * g.d2.d);
        n = q;
    } else {
        pw = (int)(pvox % g.w2.d);
        int64_t r = pvox / g.w2.d;
        ph = (int)(r % g.h2.d);
        r /= g.h2.d;
        pd = (int)(r % g.d2.d);
        n = r / g.d2.d;
    }
}

static PoolGrid pool_grid(int64_t d, int64_t h, int64_t w) {
    return PoolGrid{FastDiv::make((uint32_t)(w / 2)), FastDiv::make((uint32_t)(h / 2)), FastDiv::make((uint32_t)(d / 2))};
}

// one thread = one pooled voxel x 8 channels
__global__ void pool_fwd_kernel(const uint16_t* __restrict__ z, const float* __restrict__ bias, float slope,
                                uint16_t* __restrict__ y, uint8_t* __restrict__ idx, int64_t N, int D, int H, int W,
                                int C, PoolGrid pg) {
    const int C8 = C / 8, D2 = D / 2, H2 = H / 2, W2 = W / 2;
    const int64_t total = N * D2 * H2 * W2 * C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % C8);
        int64_t pvox = i / C8;
        int64_t n;
        int pd, ph, pw;
        pool_decode(pg, pvox, n, pd, ph, pw);
        float m[8];
        uint32_t code[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            const int64_t o = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z + o)), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                if (k == 0 || f[c] > m[c]) {
                    m[c] = f[c];
                    code[c] = k;
                }
            }
        }
        float out[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float s = m[c] + (bias ? bias[8 * c8 + c] : 0.f);
            out[c] = s > 0.f ? s : slope * s;
        }
        const int64_t po = pvox * C + 8 * c8;
        *reinterpret_cast<uint4*>(y + po) = pack8(out);
        if (idx) {
            uint2 cv;
            cv.x = code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24);
            cv.y = code[4] | (code[5] << 8) | (code[6] << 16) | (code[7] << 24);
            *reinterpret_cast<uint2*>(idx + po) = cv;
        }
    }
}

// one thread = one pooled voxel x 8 channels; the thread's channel group is
// fixed (blockDim and the grid stride are multiples of C/8) so it can keep
// the bias-gradient partial sums in registers.  partial[block][C] receives the
// per-block sums, added in ascending thread order.
__global__ void pool_bwd_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y,
                                const uint8_t* __restrict__ idx, float slope, uint16_t* __restrict__ dz,
                                uint16_t* __restrict__ dy_pre, float* __restrict__ partial, int64_t N, int D, int H,
                                int W, int C, PoolGrid pg) {
    extern __shared__ float red[];  // [blockDim][8]
    const int C8 = C / 8, D2 = D / 2, H2 = H / 2, W2 = W / 2;
    const int64_t total = N * D2 * H2 * W2 * C8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // blockDim and the grid stride are multiples of C8: the thread's channel
    // group is fixed and its pooled voxel advances by a fixed step
    const int c8 = (int)(threadIdx.x % C8);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t pstep = stride / C8;
    int64_t pvox = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += stride, pvox += pstep) {
        const int64_t po = pvox * C + 8 * c8;
        float g[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dy + po)), g);
        if (y) {
            float yy[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(y + po)), yy);
#pragma unroll
            for (int c = 0; c < 8; ++c) g[c] *= (yy[c] > 0.f ? 1.f : slope);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += g[c];
        // dy_pre and dz store g rounded to bf16
        const uint4 gp = pack8(g);
        unpack8(gp, g);
        if (dy_pre) *reinterpret_cast<uint4*>(dy_pre + po) = gp;
        if (dz) {
            const uint2 cv = __ldg(reinterpret_cast<const uint2*>(idx + po));
            const uint32_t codes[2] = {cv.x, cv.y};
            int64_t n;
            int pd, ph, pw;
            pool_decode(pg, pvox, n, pd, ph, pw);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
                float o[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) o[c] = ((codes[c >> 2] >> (8 * (c & 3))) & 0xFF) == (uint32_t)k ? g[c] : 0.f;
                const int64_t zo = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
                *reinterpret_cast<uint4*>(dz + zo) = pack8(o);
            }
        }
    }
    if (partial) {
#pragma unroll
        for (int c = 0; c < 8; ++c) red[threadIdx.x * 8 + c] = acc[c];
        __syncthreads();
        for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
            const int c8 = ch / 8, c = ch % 8;
            float s = 0.f;
            for (int t = c8; t < (int)blockDim.x; t += C8) s += red[t * 8 + c];
            partial[(int64_t)blockIdx.x * C + ch] = s;
        }
    }
}

// out[ch] = sum over rows of partial[row][ch]; one block per channel, each
// thread sums a strided subset of rows, then a fixed-shape tree (deterministic).
__global__ void colsum_kernel(const float* __restrict__ partial, int rows, int C, float* __restrict__ out) {
    __shared__ float red[256];
    const int ch = blockIdx.x;
    float s = 0.f;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) s += partial[(int64_t)r * C + ch];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int k = blockDim.x / 2; k > 0; k >>= 1) {
        if ((int)threadIdx.x < k) red[threadIdx.x] += red[threadIdx.x + k];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[ch] = red[0];
}

// W'[ci][t'][co] = W[co][26 - t'][ci]: the filter of the backward-data
// convolution written as a forward convolution.  One 32 x 32 (co, ci) tile
// of one tap per block iteration, transposed through shared memory so both
// the reads (ci contiguous) and the writes (co contiguous) are coalesced.
__global__ void flip_transpose_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ wt, int Cout, int Cin) {
    __shared__ uint16_t tile[32][33];
    const int tiles_co = (Cout + 31) / 32, tiles_ci = (Cin + 31) / 32;
    const int ntiles = 27 * tiles_co * tiles_ci;
    for (int b = blockIdx.x; b < ntiles; b += gridDim.x) {
        const int tci = b % tiles_ci;
        const int r = b / tiles_ci;
        const int tco = r % tiles_co;
        const int tp = r / tiles_co;  // output tap t'
        for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
            const int co = tco * 32 + ty, ci = tci * 32 + threadIdx.x;
            tile[ty][threadIdx.x] = (co < Cout && ci < Cin) ? w[((int64_t)co * 27 + (26 - tp)) * Cin + ci] : 0;
        }
        __syncthreads();
        for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
            const int ci = tci * 32 + ty, co = tco * 32 + threadIdx.x;
            if (ci < Cin && co < Cout) wt[((int64_t)ci * 27 + tp) * Cout + co] = tile[threadIdx.x][ty];
        }
        __syncthreads();
    }
}

// Bias gradient alone (no dZ, no dYpre, dy already the pre-activation
// gradient): per-thread sums of one 8-channel group over the rows i, i +
// stride, ... in increasing order -- the order pool_bwd_kernel uses -- with
// four rows loaded per iteration; partial[block][C] as pool_bwd_kernel.
__global__ void pool_bwd_dbias_kernel(const uint16_t* __restrict__ dy, float* __restrict__ partial, int64_t total8,
                                      int C) {
    extern __shared__ float red[];  // [blockDim][8]
    const int C8 = C / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < total8; i0 += 4 * stride) {
        uint4 gv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            gv[u] = i < total8 ? __ldg(reinterpret_cast<const uint4*>(dy) + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float g[8];
            unpack8(gv[u], g);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] += g[c];
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) red[threadIdx.x * 8 + c] = acc[c];
    __syncthreads();
    for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
        const int c8 = ch / 8, c = ch % 8;
        float s = 0.f;
        for (int t = c8; t < (int)blockDim.x; t += C8) s += red[t * 8 + c];
        partial[(int64_t)blockIdx.x * C + ch] = s;
    }
}

// Average pooling of the activated window (CosmoFlow page, section III-C:
// constant weights 1/8 for a 2x2x2 window), one thread per pooled voxel x 8
// channels: y = (1/8) sum LReLU(z + b), mask bit dd*4+dh*2+dw = (z + b > 0).
__global__ void avgpool_fwd_kernel(const uint16_t* __restrict__ z, const float* __restrict__ bias, float slope,
                                   uint16_t* __restrict__ y, uint8_t* __restrict__ mask, int64_t N, int D, int H,
                                   int W, int C, PoolGrid pg) {
    const int C8 = C / 8, D2 = D / 2, H2 = H / 2, W2 = W / 2;
    const int64_t total = N * D2 * H2 * W2 * C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % C8);
        const int64_t pvox = i / C8;
        int64_t n;
        int pd, ph, pw;
        pool_decode(pg, pvox, n, pd, ph, pw);
        float b[8], sum[8];
        uint32_t m[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            b[c] = bias ? bias[8 * c8 + c] : 0.f;
            sum[c] = 0.f;
            m[c] = 0u;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            const int64_t o = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z + o)), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float v = f[c] + b[c];
                m[c] |= (v > 0.f ? 1u : 0u) << k;
                sum[c] += v > 0.f ? v : slope * v;
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) sum[c] *= 0.125f;
        const int64_t po = pvox * C + 8 * c8;
        *reinterpret_cast<uint4*>(y + po) = pack8(sum);
        if (mask)
            *reinterpret_cast<uint2*>(mask + po) =
                make_uint2(m[0] | (m[1] << 8) | (m[2] << 16) | (m[3] << 24), m[4] | (m[5] << 8) | (m[6] << 16) | (m[7] << 24));
    }
}

// Backward of the average pool: dz[v] = dy[p] / 8 * LReLU'(z[v] + b) from the
// sign mask, all eight voxels of each window written; the bias gradient sums
// the fp32 dz values per thread (fixed channel group, as pool_bwd_kernel).
__global__ void avgpool_bwd_kernel(const uint16_t* __restrict__ dy, const uint8_t* __restrict__ mask, float slope,
                                   uint16_t* __restrict__ dz, float* __restrict__ partial, int64_t N, int D, int H,
                                   int W, int C, PoolGrid pg) {
    extern __shared__ float red[];  // [blockDim][8]
    const int C8 = C / 8, D2 = D / 2, H2 = H / 2, W2 = W / 2;
    const int64_t total = N * D2 * H2 * W2 * C8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int c8 = (int)(threadIdx.x % C8);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t pstep = stride / C8;
    int64_t pvox = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += stride, pvox += pstep) {
        const int64_t po = pvox * C + 8 * c8;
        float g[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dy + po)), g);
        const uint2 mv = __ldg(reinterpret_cast<const uint2*>(mask + po));
        const uint32_t mw[2] = {mv.x, mv.y};
        int64_t n;
        int pd, ph, pw;
        pool_decode(pg, pvox, n, pd, ph, pw);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            float o[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const bool pos = (mw[c >> 2] >> (8 * (c & 3) + k)) & 1u;
                o[c] = g[c] * 0.125f * (pos ? 1.f : slope);
                acc[c] += o[c];
            }
            if (dz) {
                const int64_t zo = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
                *reinterpret_cast<uint4*>(dz + zo) = pack8(o);
            }
        }
    }
    if (partial) {
#pragma unroll
        for (int c = 0; c < 8; ++c) red[threadIdx.x * 8 + c] = acc[c];
        __syncthreads();
        for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
            const int cg = ch / 8, c = ch % 8;
            float sum = 0.f;
            for (int t = cg; t < (int)blockDim.x; t += C8) sum += red[t * 8 + c];
            partial[(int64_t)blockIdx.x * C + ch] = sum;
        }
    }
}

// Unpooled block: y = LReLU(z + b), 8 channels per thread.
__global__ void act_fwd_kernel(const uint16_t* __restrict__ z, const float* __restrict__ bias, float slope,
                               uint16_t* __restrict__ y, int64_t total8, int C) {
    const int C8 = C / 8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % C8);
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(z) + i), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float v = f[c] + (bias ? bias[8 * c8 + c] : 0.f);
            f[c] = v > 0.f ? v : slope * v;
        }
        reinterpret_cast<uint4*>(y)[i] = pack8(f);
    }
}

// Its backward: dz = dy * LReLU'(y) (dy as is when y is NULL), bias-gradient
// partials of the fp32 dz per thread (fixed channel group).
__global__ void act_bwd_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y, float slope,
                               uint16_t* __restrict__ dz, float* __restrict__ partial, int64_t total8, int C) {
    extern __shared__ float red[];  // [blockDim][8]
    const int C8 = C / 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total8;
         i += (int64_t)gridDim.x * blockDim.x) {
        float g[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dy) + i), g);
        if (y) {
            float yy[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(y) + i), yy);
#pragma unroll
            for (int c = 0; c < 8; ++c) g[c] *= (yy[c] > 0.f ? 1.f : slope);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += g[c];
        if (dz) reinterpret_cast<uint4*>(dz)[i] = pack8(g);
    }
    if (partial) {
#pragma unroll
        for (int c = 0; c < 8; ++c) red[threadIdx.x * 8 + c] = acc[c];
        __syncthreads();
        for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
            const int cg = ch / 8, c = ch % 8;
            float sum = 0.f;
            for (int t = cg; t < (int)blockDim.x; t += C8) sum += red[t * 8 + c];
            partial[(int64_t)blockIdx.x * C + ch] = sum;
        }
    }
}

// Zero insertion for the stride-2 backward, 8 channels per thread: out voxel
// (d, h, w) takes dz (d/2, h/2, w/2) when all three are even, else zero.
__global__ void upsample2_kernel(const uint16_t* __restrict__ dz, uint16_t* __restrict__ out, int64_t N, int D,
                                 int H, int W, int C) {
    const int C8 = C / 8;
    const int Do = (D + 1) / 2, Ho = (H + 1) / 2, Wo = (W + 1) / 2;
    const int64_t total = N * D * H * W * C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % C8);
        int64_t r = i / C8;
        const int w = (int)(r % W);
        r /= W;
        const int h = (int)(r % H);
        r /= H;
        const int d = (int)(r % D);
        const int64_t n = r / D;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (((d | h | w) & 1) == 0)
            v = __ldg(reinterpret_cast<const uint4*>(dz + ((((n * Do + d / 2) * Ho + h / 2) * Wo + w / 2) * C + 8 * c8)));
        reinterpret_cast<uint4*>(out)[i] = v;
    }
}

// ---------------------------------------------------------------------------
// Batch normalisation after the conv (hybrid-parallelism page, section IV),
// training mode: per-channel statistics of the stored conv output z over all
// n and voxels.

// Per-thread sums of one 8-channel group of z and of its squares over the rows
// i, i + stride, ... (fixed order); partial[block][2C]: sums, then squares.
__global__ void channel_stats_kernel(const uint16_t* __restrict__ z, float* __restrict__ partial, int64_t total8,
                                     int C) {
    extern __shared__ float red[];  // [blockDim][16]
    const int C8 = C / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total8; i += stride) {
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(z) + i), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            s[c] += f[c];
            q[c] = fmaf(f[c], f[c], q[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        red[threadIdx.x * 16 + c] = s[c];
        red[threadIdx.x * 16 + 8 + c] = q[c];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 2 * C; e += blockDim.x) {
        const int which = e / C, ch = e % C, cg = ch / 8, c = ch % 8;
        float acc = 0.f;
        for (int t = cg; t < (int)blockDim.x; t += C8) acc += red[t * 16 + 8 * which + c];
        partial[(int64_t)blockIdx.x * 2 * C + e] = acc;
    }
}

// Batch statistics of channel ch from the sums: mean and 1 / sqrt(var + eps),
// var = E[z^2] - mean^2 (in fp64 from the fp32 channel sums).
__device__ __forceinline__ void bn_stats(const float* __restrict__ sums, int C, int ch, double count, float eps,
                                         double& mean, double& inv) {
    mean = (double)sums[ch] / count;
    const double var = fmax((double)sums[C + ch] / count - mean * mean, 0.0);
    inv = 1.0 / sqrt(var + (double)eps);
}

// Normalisation coefficients: u = a * z + b, a = gamma * inv, b = beta - mean * a.
__device__ __forceinline__ void bn_coef(const float* __restrict__ sums, int C, int ch, double count,
                                        const float* __restrict__ gamma, const float* __restrict__ beta, float eps,
                                        float& a, float& b) {
    double m, iv;
    bn_stats(sums, C, ch, count, eps, m, iv);
    a = (float)((double)gamma[ch] * iv);
    b = (float)((double)beta[ch] - m * (double)gamma[ch] * iv);
}

// u = a*z + b, then the block's activation and pooling (POOL: 0 max with
// codes, 1 average with sign masks, 2 none), one thread per output voxel x 8
// channels.  sums: [2C] (channel sums, sums of squares).
template <int POOL>
__global__ void bn_act_pool_fwd_kernel(const uint16_t* __restrict__ z, const float* __restrict__ sums,
                                       const float* __restrict__ gamma, const float* __restrict__ beta, float eps,
                                       float slope, uint16_t* __restrict__ y, uint8_t* __restrict__ aux, int64_t N,
                                       int D, int H, int W, int C, PoolGrid pg) {
    const int C8 = C / 8;
    const double count = (double)N * D * H * W;
    const int64_t total = POOL == 2 ? N * D * H * W * C8 : N * (D / 2) * (H / 2) * (W / 2) * C8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % C8);
        const int64_t vox = i / C8;
        float a[8], b[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) bn_coef(sums, C, 8 * c8 + c, count, gamma, beta, eps, a[c], b[c]);
        if (POOL == 2) {
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z) + i), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float u = fmaf(a[c], f[c], b[c]);
                f[c] = u > 0.f ? u : slope * u;
            }
            reinterpret_cast<uint4*>(y)[i] = pack8(f);
            continue;
        }
        int64_t n;
        int pd, ph, pw;
        pool_decode(pg, vox, n, pd, ph, pw);
        float m[8];
        uint32_t code[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            m[c] = 0.f;
            code[c] = 0u;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            const int64_t o = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z + o)), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float u = fmaf(a[c], f[c], b[c]);
                if (POOL == 0) {
                    if (k == 0 || u > m[c]) {
                        m[c] = u;
                        code[c] = k;
                    }
                } else {
                    code[c] |= (u > 0.f ? 1u : 0u) << k;
                    m[c] += u > 0.f ? u : slope * u;
                }
            }
        }
        float out[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) out[c] = POOL == 0 ? (m[c] > 0.f ? m[c] : slope * m[c]) : m[c] * 0.125f;
        const int64_t po = vox * C + 8 * c8;
        *reinterpret_cast<uint4*>(y + po) = pack8(out);
        if (aux)
            *reinterpret_cast<uint2*>(aux + po) =
                make_uint2(code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24),
                           code[4] | (code[5] << 8) | (code[6] << 16) | (code[7] << 24));
    }
}

// The activation/pooling backward folded into the batch-norm backward: du at
// full resolution is implicit (POOL 0: g = dy * LReLU'(y) at the argmax voxel,
// else 0; 1: dy / 8 * LReLU'(u) from the mask; 2: dy * LReLU'(y)), with y
// NULL meaning dy already carries LReLU'.  PASS 0: per-thread sums of du and
// du * zh over its 8-channel group (partial[block][2C]: dbeta, then dgamma);
// PASS 1: dz = a * (du - dbeta/count - zh * dgamma/count) for every voxel of
// the thread's window(s), written dense.  red: [2C] reduced dbeta, dgamma.
template <int POOL, int PASS>
__global__ void bn_act_pool_bwd_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y,
                                       const uint8_t* __restrict__ aux, const uint16_t* __restrict__ z,
                                       const float* __restrict__ sums, const float* __restrict__ gamma, float eps,
                                       float slope, const float* __restrict__ dsums, uint16_t* __restrict__ dz,
                                       float* __restrict__ partial, int64_t N, int D, int H, int W, int C,
                                       PoolGrid pg) {
    extern __shared__ float red[];  // [blockDim][16]
    const int C8 = C / 8;
    const double count = (double)N * D * H * W;
    const int64_t total = POOL == 2 ? N * D * H * W * C8 : N * (D / 2) * (H / 2) * (W / 2) * C8;
    const int c8 = (int)(threadIdx.x % C8);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float a[8], mean[8], inv[8], m1[8], m2[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        double m, iv;
        bn_stats(sums, C, 8 * c8 + c, count, eps, m, iv);
        mean[c] = (float)m;
        inv[c] = (float)iv;
        a[c] = (float)((double)gamma[8 * c8 + c] * iv);
        if (PASS == 1) {
            m1[c] = (float)((double)dsums[8 * c8 + c] / count);
            m2[c] = (float)((double)dsums[C + 8 * c8 + c] / count);
        }
    }
    float sb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, sg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t vox = i / C8;
        float g[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dy) + i), g);
        if (y && POOL != 1) {
            float yy[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(y) + i), yy);
#pragma unroll
            for (int c = 0; c < 8; ++c) g[c] *= (yy[c] > 0.f ? 1.f : slope);
        }
        if (POOL == 2) {
            float f[8], o[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z) + i), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float zh = (f[c] - mean[c]) * inv[c];
                if (PASS == 0) {
                    sb[c] += g[c];
                    sg[c] = fmaf(g[c], zh, sg[c]);
                } else {
                    o[c] = a[c] * (g[c] - m1[c] - zh * m2[c]);
                }
            }
            if (PASS == 1) reinterpret_cast<uint4*>(dz)[i] = pack8(o);
            continue;
        }
        uint32_t cw[2] = {0u, 0u};
        const uint2 cv = __ldg(reinterpret_cast<const uint2*>(aux) + i);
        cw[0] = cv.x;
        cw[1] = cv.y;
        int64_t n;
        int pd, ph, pw;
        pool_decode(pg, vox, n, pd, ph, pw);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            const int64_t o = ((((n * D + 2 * pd + dd) * H + 2 * ph + dh) * W) + 2 * pw + dw) * C + 8 * c8;
            float f[8], out[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(z + o)), f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t byte = (cw[c >> 2] >> (8 * (c & 3))) & 0xFFu;
                float du;
                if (POOL == 0) {
                    du = byte == (uint32_t)k ? g[c] : 0.f;
                } else {
                    du = g[c] * 0.125f * (((byte >> k) & 1u) ? 1.f : slope);
                }
                const float zh = (f[c] - mean[c]) * inv[c];
                if (PASS == 0) {
                    sb[c] += du;
                    sg[c] = fmaf(du, zh, sg[c]);
                } else {
                    out[c] = a[c] * (du - m1[c] - zh * m2[c]);
                }
            }
            if (PASS == 1) *reinterpret_cast<uint4*>(dz + o) = pack8(out);
        }
    }
    if (PASS == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            red[threadIdx.x * 16 + c] = sb[c];
            red[threadIdx.x * 16 + 8 + c] = sg[c];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < 2 * C; e += blockDim.x) {
            const int which = e / C, ch = e % C, cg = ch / 8, c = ch % 8;
            float acc = 0.f;
            for (int t = cg; t < (int)blockDim.x; t += C8) acc += red[t * 16 + 8 * which + c];
            partial[(int64_t)blockIdx.x * 2 * C + e] = acc;
        }
    }
}

__global__ void timeout_probe_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, limit_ns, status, WAIT_PROBE);
}

// ---------------------------------------------------------------------------

static int pool_bwd_block(int c) {
    const int c8 = c / 8;
    return (256 / c8) * c8;
}
static int pool_bwd_grid(int num_sms) { return 4 * num_sms; }

size_t pool_bwd_workspace_bytes(int num_sms, int c) {
    return (size_t)pool_bwd_grid(num_sms) * c * sizeof(float);
}

cf_status launch_pool_fwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                          const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* idx) {
    const int64_t total = n * (d / 2) * (h / 2) * (w / 2) * (c / 8);
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 16LL * ctx.num_sms));
    pool_fwd_kernel<<<blocks, threads, 0, ctx.stream>>>(z, bias, slope, y, idx, n, (int)d, (int)h, (int)w, c,
                                                        pool_grid(d, h, w));
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_pool_bwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                          const uint16_t* dy, const uint16_t* y, const uint8_t* idx, float slope, uint16_t* dz,
                          uint16_t* dy_pre, float* dbias, void* ws, size_t ws_bytes, bool reduce) {
    if (c / 8 > 256) return CF_ERR_UNSUPPORTED;
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    float* partial = nullptr;
    if (dbias) {
        if (ws == nullptr || ws_bytes < pool_bwd_workspace_bytes(ctx.num_sms, c)) return CF_ERR_WORKSPACE;
        partial = static_cast<float*>(ws);
    }
    if (y == nullptr && dz == nullptr && dy_pre == nullptr) {
        if (partial == nullptr) return CF_OK;  // nothing requested
        pool_bwd_dbias_kernel<<<blocks, threads, threads * 8 * sizeof(float), ctx.stream>>>(
            dy, partial, n * (d / 2) * (h / 2) * (w / 2) * (c / 8), c);
    } else {
        pool_bwd_kernel<<<blocks, threads, threads * 8 * sizeof(float), ctx.stream>>>(
            dy, y, idx, slope, dz, dy_pre, partial, n, (int)d, (int)h, (int)w, c, pool_grid(d, h, w));
    }
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    if (dbias && reduce) {
        colsum_kernel<<<c, 256, 0, ctx.stream>>>(partial, blocks, c, dbias);
        if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    }
    return CF_OK;
}

size_t channel_sums_workspace_bytes(int num_sms, int c) { return pool_bwd_workspace_bytes(num_sms, c); }

cf_status launch_colsum(const LaunchCtx& ctx, const float* partial, int rows, int c, float* out);

cf_status launch_channel_sums(const LaunchCtx& ctx, const uint16_t* x, int64_t rows, int c, float* partial,
                              float* out) {
    if (c % 8 != 0 || c / 8 > 256) return CF_ERR_UNSUPPORTED;
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    pool_bwd_dbias_kernel<<<blocks, threads, threads * 8 * sizeof(float), ctx.stream>>>(x, partial, rows * (c / 8),
                                                                                         c);
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    return launch_colsum(ctx, partial, blocks, c, out);
}

cf_status launch_colsum(const LaunchCtx& ctx, const float* partial, int rows, int c, float* out) {
    colsum_kernel<<<c, 256, 0, ctx.stream>>>(partial, rows, c, out);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_flip_transpose(const LaunchCtx& ctx, int c_out, int c_in, const uint16_t* w, uint16_t* wt) {
    const int64_t ntiles = 27LL * ((c_out + 31) / 32) * ((c_in + 31) / 32);
    const int blocks = (int)std::min<int64_t>(ntiles, 8LL * ctx.num_sms);
    flip_transpose_kernel<<<blocks, dim3(32, 8), 0, ctx.stream>>>(w, wt, c_out, c_in);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_avgpool_fwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                             const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* mask) {
    const int64_t total = n * (d / 2) * (h / 2) * (w / 2) * (c / 8);
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 16LL * ctx.num_sms));
    avgpool_fwd_kernel<<<blocks, threads, 0, ctx.stream>>>(z, bias, slope, y, mask, n, (int)d, (int)h, (int)w, c,
                                                           pool_grid(d, h, w));
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_avgpool_bwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                             const uint16_t* dy, const uint8_t* mask, float slope, uint16_t* dz, float* dbias,
                             void* ws, size_t ws_bytes) {
    if (c / 8 > 256) return CF_ERR_UNSUPPORTED;
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    float* partial = nullptr;
    if (dbias) {
        if (ws == nullptr || ws_bytes < pool_bwd_workspace_bytes(ctx.num_sms, c)) return CF_ERR_WORKSPACE;
        partial = static_cast<float*>(ws);
    }
    avgpool_bwd_kernel<<<blocks, threads, threads * 8 * sizeof(float), ctx.stream>>>(
        dy, mask, slope, dz, partial, n, (int)d, (int)h, (int)w, c, pool_grid(d, h, w));
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    return dbias ? launch_colsum(ctx, partial, blocks, c, dbias) : CF_OK;
}

cf_status launch_act_fwd(const LaunchCtx& ctx, int64_t count, int c, const uint16_t* z, const float* bias,
                         float slope, uint16_t* y) {
    const int64_t total8 = count / 8;
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total8 + threads - 1) / threads, 16LL * ctx.num_sms));
    act_fwd_kernel<<<blocks, threads, 0, ctx.stream>>>(z, bias, slope, y, total8, c);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_act_bwd(const LaunchCtx& ctx, int64_t count, int c, const uint16_t* dy, const uint16_t* y,
                         float slope, uint16_t* dz, float* dbias, void* ws, size_t ws_bytes) {
    if (c / 8 > 256) return CF_ERR_UNSUPPORTED;
    // blockDim and the grid stride are multiples of c/8: each thread keeps one
    // channel group
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    float* partial = nullptr;
    if (dbias) {
        if (ws == nullptr || ws_bytes < pool_bwd_workspace_bytes(ctx.num_sms, c)) return CF_ERR_WORKSPACE;
        partial = static_cast<float*>(ws);
    }
    act_bwd_kernel<<<blocks, threads, threads * 8 * sizeof(float), ctx.stream>>>(dy, y, slope, dz, partial,
                                                                                   count / 8, c);
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    return dbias ? launch_colsum(ctx, partial, blocks, c, dbias) : CF_OK;
}

cf_status launch_upsample2(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                           const uint16_t* dz, uint16_t* out) {
    const int64_t total = n * d * h * w * (c / 8);
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 16LL * ctx.num_sms));
    upsample2_kernel<<<blocks, threads, 0, ctx.stream>>>(dz, out, n, (int)d, (int)h, (int)w, c);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

size_t bn_workspace_bytes(int num_sms, int c) { return (size_t)pool_bwd_grid(num_sms) * 2 * c * sizeof(float); }

cf_status launch_channel_stats(const LaunchCtx& ctx, int64_t rows, int c, const uint16_t* z, float* sums, void* ws,
                               size_t ws_bytes) {
    if (c % 8 != 0 || c / 8 > 256) return CF_ERR_UNSUPPORTED;
    if (ws == nullptr || ws_bytes < bn_workspace_bytes(ctx.num_sms, c)) return CF_ERR_WORKSPACE;
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    float* partial = static_cast<float*>(ws);
    channel_stats_kernel<<<blocks, threads, threads * 16 * sizeof(float), ctx.stream>>>(z, partial, rows * (c / 8), c);
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    return launch_colsum(ctx, partial, blocks, 2 * c, sums);
}

cf_status launch_bn_act_pool_fwd(const LaunchCtx& ctx, int pool, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                                 const uint16_t* z, const float* sums, const float* gamma, const float* beta,
                                 float eps, float slope, uint16_t* y, uint8_t* aux) {
    const int64_t total = (pool == 2 ? n * d * h * w : n * (d / 2) * (h / 2) * (w / 2)) * (c / 8);
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 16LL * ctx.num_sms));
    const PoolGrid pg = pool_grid(std::max<int64_t>(d, 2), std::max<int64_t>(h, 2), std::max<int64_t>(w, 2));
    if (pool == 0)
        bn_act_pool_fwd_kernel<0><<<blocks, threads, 0, ctx.stream>>>(z, sums, gamma, beta, eps, slope, y, aux, n,
                                                                      (int)d, (int)h, (int)w, c, pg);
    else if (pool == 1)
        bn_act_pool_fwd_kernel<1><<<blocks, threads, 0, ctx.stream>>>(z, sums, gamma, beta, eps, slope, y, aux, n,
                                                                      (int)d, (int)h, (int)w, c, pg);
    else
        bn_act_pool_fwd_kernel<2><<<blocks, threads, 0, ctx.stream>>>(z, sums, gamma, beta, eps, slope, y, aux, n,
                                                                      (int)d, (int)h, (int)w, c, pg);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_bn_act_pool_bwd(const LaunchCtx& ctx, int pool, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                                 const uint16_t* dy, const uint16_t* y, const uint8_t* aux, const uint16_t* z,
                                 const float* sums, const float* gamma, float eps, float slope, uint16_t* dz,
                                 float* dsums, void* ws, size_t ws_bytes) {
    if (c % 8 != 0 || c / 8 > 256) return CF_ERR_UNSUPPORTED;
    if (ws == nullptr || ws_bytes < bn_workspace_bytes(ctx.num_sms, c)) return CF_ERR_WORKSPACE;
    const int threads = pool_bwd_block(c);
    const int blocks = pool_bwd_grid(ctx.num_sms);
    float* partial = static_cast<float*>(ws);
    const PoolGrid pg = pool_grid(std::max<int64_t>(d, 2), std::max<int64_t>(h, 2), std::max<int64_t>(w, 2));
    const size_t sh = threads * 16 * sizeof(float);
#define CF_BN_BWD(P, S)                                                                                          \
    bn_act_pool_bwd_kernel<P, S><<<blocks, threads, sh, ctx.stream>>>(dy, y, aux, z, sums, gamma, eps, slope, dsums, \
                                                                     dz, partial, n, (int)d, (int)h, (int)w, c, pg)
    if (pool == 0)
        CF_BN_BWD(0, 0);
    else if (pool == 1)
        CF_BN_BWD(1, 0);
    else
        CF_BN_BWD(2, 0);
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    cf_status st = launch_colsum(ctx, partial, blocks, 2 * c, dsums);
    if (st != CF_OK) return st;
    if (pool == 0)
        CF_BN_BWD(0, 1);
    else if (pool == 1)
        CF_BN_BWD(1, 1);
    else
        CF_BN_BWD(2, 1);
#undef CF_BN_BWD
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_timeout_probe(const LaunchCtx& ctx) {
    timeout_probe_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, ctx.wait_ns);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

}  // namespace cf
