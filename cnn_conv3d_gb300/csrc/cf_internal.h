// cf_internal.h -- host-side declarations shared by the library's translation
// units (launchers implemented in the .cu files, called from cf_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/cf_conv3d.h"

namespace cf {

// Status codes written into the device status word by a bounded wait that gave
// up (any non-zero value maps to CF_ERR_TIMEOUT on the host).
enum : int {
    WAIT_PRODUCER_EMPTY = 0x101,
    WAIT_MMA_TMEM_EMPTY = 0x102,
    WAIT_MMA_FULL = 0x103,
    WAIT_EPI_TMEM_FULL = 0x104,
    WAIT_DRAIN = 0x105,
    WAIT_PROBE = 0x1FF,
};

// Epilogue of a conv kernel (a compile-time mode): plain bf16 store, max-pool
// (+ bias, leaky ReLU, argmax codes), backward-data leaky-ReLU derivative,
// average pool of the activated window (+ sign masks), bias + leaky ReLU
// without pooling.
enum EpiMode : int { EPI_PLAIN = 0, EPI_POOL = 1, EPI_DGRAD = 2, EPI_AVG = 3, EPI_ACT = 4 };

struct LaunchCtx {
    cudaStream_t stream;
    int num_sms;
    int* status;       // device status word
    uint64_t wait_ns;  // bounded-wait limit
};

// Fills ctx for the current device and `stream` (cf_api.cu); false on a CUDA error.
bool cf_device_ctx(LaunchCtx* ctx, void* stream);

// Geometry of the 128-voxel output tile of the implicit GEMM: a box of
// td x th x tw voxels (td = 2 so that pooled tiles hold whole windows).
struct TileGeom {
    int tw, th, td;
};
TileGeom choose_tile(int64_t d, int64_t h, int64_t w);

// Encodes a tiled TMA descriptor; returns false on failure.  elem_strides:
// traversal stride per dimension (NULL = 1 everywhere); along a dimension with
// stride s the box loads ceil(box / s) elements, every s-th one.
bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz,
                 const uint32_t* elem_strides = nullptr);

// conv_fwd.cu ---------------------------------------------------------------
// Generic implicit-GEMM conv (c_in a multiple of 16): out = conv(x, wk) where
// wk is [c_out][27][c_in] (K-major GEMM B operand).  EPI_POOL writes the pooled
// block output and argmax codes (pool_kind 0) or the average of the activated
// window and its sign masks (pool_kind 1); EPI_PLAIN stores z, or LReLU(z + b)
// with act = 1; EPI_DGRAD multiplies by LReLU'(x_act).  n, d, h, w are the
// input sizes; stride 2 computes the output at the even input positions,
// (d + 1) / 2 ... per dimension.
cf_status launch_conv_igemm(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                            int c_out, const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y,
                            uint8_t* idx, const float* bias, const uint16_t* x_act, float slope,
                            int pool_kind = 0, int act = 0, int stride = 1, uint16_t* route_dz = nullptr,
                            const uint8_t* route_idx = nullptr);

// conv_halo.cu: same contract as launch_conv_igemm (stride 1) for c_in % 16 == 0
// and c_out in {32, 64, 128}, reading A from one halo tile per channel chunk.
bool halo_path_supported(int c_in, int c_out);
// colsum_part (unpooled epilogues, c_out <= 32): [grid][c_out] channel sums of
// the stored outputs, one row per CTA (grid <= SM count), or NULL.
cf_status launch_conv_halo(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                           int c_out, const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y,
                           uint8_t* idx, const float* bias, const uint16_t* x_act, float slope,
                           float* colsum_part = nullptr, int pool_kind = 0, int act = 0,
                           uint16_t* route_dz = nullptr, const uint8_t* route_idx = nullptr);

// conv_quad.cu -------------------------------------------------------------
// First-layer forward (c_in 4, c_out 16 or 32) with the max-pool epilogue,
// A read straight from the input tile: d even, h a multiple of 16, w of 32.
bool quad_path_supported(int64_t d, int64_t h, int64_t w, int c_in, int c_out);
cf_status launch_conv_quad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_out,
                           const uint16_t* x, const uint16_t* wk, uint16_t* y, uint8_t* idx, const float* bias,
                           float slope);

// conv_smallc.cu: forward conv for c_in in {1,4} (im2col operand in tensor memory).
cf_status launch_conv_smallc(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                             int c_out, const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y,
                             uint8_t* idx, const float* bias, float slope, int pool_kind = 0, int act = 0);

// conv_wgrad_halo.cu: backward weight reading the input once per K block as a
// halo tile (c_in 32 with c_out 32/64/128, c_in 64 with c_out 64/128); writes
// split-K partials [n_splits][c_out][27*c_in].
bool wgrad_halo_supported(int c_in, int c_out);
size_t wgrad_halo_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out);
cf_status launch_wgrad_halo(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                            int c_out, const uint16_t* x, const uint16_t* dz, float* part, int* n_splits);

// conv_wgrad.cu -------------------------------------------------------------
size_t wgrad_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out);
// the (c_in, c_out) pairs launch_wgrad implements
// conv_wgrad_quad.cu: first-layer weight gradient (c_in 4, c_out 32) with the
// max-pool backward fused, d even, h a multiple of 16, w of 32; writes
// *n_splits phase-major split-K partials of 32 x 108 floats.
bool wgrad_quad_supported(int64_t d, int64_t h, int64_t w, int c_in, int c_out);
size_t wgrad_quad_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w);
cf_status launch_wgrad_quad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, const uint16_t* x,
                            const uint16_t* g, const uint8_t* idx, float* part, int* n_splits);
bool wgrad_shape_supported(int c_in, int c_out);
// true when launch_wgrad takes the routed form (idx != NULL: dz pooled, the
// dense dZ expanded on chip) for this c_in
bool wgrad_routed_fused(int c_in);
cf_status launch_wgrad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                       const uint16_t* x, const uint16_t* dz, const uint8_t* idx, float* dw, int accumulate,
                       void* ws, size_t ws_bytes);

// elementwise.cu ------------------------------------------------------------
cf_status launch_pool_fwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                          const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* idx);
size_t pool_bwd_workspace_bytes(int num_sms, int c);
// reduce = false: the bias gradient is left as the per-block partial sums in ws
// ([pool_bwd_workspace_bytes / (4 c)][c]); dbias must then be non-NULL (it only
// requests the partials).
cf_status launch_pool_bwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                          const uint16_t* dy, const uint16_t* y, const uint8_t* idx, float slope, uint16_t* dz,
                          uint16_t* dy_pre, float* dbias, void* ws, size_t ws_bytes, bool reduce = true);
cf_status launch_flip_transpose(const LaunchCtx& ctx, int c_out, int c_in, const uint16_t* w, uint16_t* wt);
// Page variants of the block epilogue as standalone kernels: average pooling
// of the activated window (y and sign masks), the unpooled activation, and
// their backward passes (dz from dy and the masks / the output, bias-gradient
// partials [blocks][c] in `partial`, reduced by colsum).
cf_status launch_avgpool_fwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                             const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* mask);
cf_status launch_avgpool_bwd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                             const uint16_t* dy, const uint8_t* mask, float slope, uint16_t* dz, float* dbias,
                             void* ws, size_t ws_bytes);
cf_status launch_act_fwd(const LaunchCtx& ctx, int64_t count, int c, const uint16_t* z, const float* bias,
                         float slope, uint16_t* y);
cf_status launch_act_bwd(const LaunchCtx& ctx, int64_t count, int c, const uint16_t* dy, const uint16_t* y,
                         float slope, uint16_t* dz, float* dbias, void* ws, size_t ws_bytes);
// Zero insertion for the stride-2 backward: out [n][d][h][w][c] holds
// dz [n][(d+1)/2][(h+1)/2][(w+1)/2][c] at the even positions, zeros elsewhere.
cf_status launch_upsample2(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                           const uint16_t* dz, uint16_t* out);
// out[ch] = sum over `rows` of partial[row][ch] (fixed order)
cf_status launch_colsum(const LaunchCtx& ctx, const float* partial, int rows, int c, float* out);
// out[ch] = sum over the rows of x [rows][c] bf16 (fixed order); partial holds
// channel_sums_workspace_bytes
size_t channel_sums_workspace_bytes(int num_sms, int c);
cf_status launch_channel_sums(const LaunchCtx& ctx, const uint16_t* x, int64_t rows, int c, float* partial,
                              float* out);
// Batch normalisation (training mode): the per-channel sums of z and z^2
// ([2c] fp32, fixed order) of rows x c bf16; the normalisation + leaky ReLU +
// pooling (pool 0 max, 1 average, 2 none) from those sums; and the backward,
// du implicit from the pooling backward, dsums = [dbeta, dgamma] ([2c]), dz
// written dense.  Workspace: bn_workspace_bytes.
size_t bn_workspace_bytes(int num_sms, int c);
cf_status launch_channel_stats(const LaunchCtx& ctx, int64_t rows, int c, const uint16_t* z, float* sums, void* ws,
                               size_t ws_bytes);
cf_status launch_bn_act_pool_fwd(const LaunchCtx& ctx, int pool, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                                 const uint16_t* z, const float* sums, const float* gamma, const float* beta,
                                 float eps, float slope, uint16_t* y, uint8_t* aux);
cf_status launch_bn_act_pool_bwd(const LaunchCtx& ctx, int pool, int64_t n, int64_t d, int64_t h, int64_t w, int c,
                                 const uint16_t* dy, const uint16_t* y, const uint8_t* aux, const uint16_t* z,
                                 const float* sums, const float* gamma, float eps, float slope, uint16_t* dz,
                                 float* dsums, void* ws, size_t ws_bytes);
cf_status launch_timeout_probe(const LaunchCtx& ctx);

}  // namespace cf
