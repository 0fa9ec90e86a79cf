/*
 * cf_conv3d.h -- C ABI of libcfconv3d.so, the GB300 (sm_103a) conv3d block of
 * a CosmoFlow-style volumetric CNN.
 *
 * What is computed (sources: "CosmoFlow: Using Deep Learning to Learn the
 * Universe at Scale", section III-A (3D conv layers followed by leaky ReLU and
 * pooling) and III-C (forward data, backward data, backward weight operators);
 * "The Case for Strong Scaling in Deep Learning: Training Large 3D CNNs with
 * Hybrid Parallelism", section IV, Table I (3^3 filters, stride-1 "same"
 * convolution, stride-2 pooling)):
 *
 *   Z[n,d,h,w,co] = sum_{kd,kh,kw,ci} W[co,kd,kh,kw,ci] * X[n,d+kd-1,h+kh-1,w+kw-1,ci]
 *                   (cross-correlation, zero padding 1, stride 1)
 *   m   = max of Z over each 2x2x2 window (stride 2), I = its code dd*4+dh*2+dw
 *         (first maximum in that order), taken on the fp32 accumulator
 *   Y   = LReLU(m + b[co]),  LReLU(s) = s > 0 ? s : slope*s
 *
 * Conventions for every entry point:
 *  - tensors are device pointers the caller owns; the library never allocates
 *    or frees device memory and never synchronises the stream (except
 *    cf_last_device_status, which says so);
 *  - activations are NDHWC, bf16 stored as uint16_t bit patterns;
 *    filters are [C_out][3][3][3][C_in] bf16; biases and weight gradients fp32;
 *    argmax codes uint8 in the pooled NDHWC shape;
 *  - every pointer must be 16-byte aligned;
 *  - work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream);
 *  - argument or precondition errors return before anything is launched;
 *    a kernel that gives up on a bounded wait records CF_ERR_TIMEOUT in a
 *    device status word read by cf_last_device_status;
 *  - sizes use 64-bit arithmetic throughout (tensors may exceed 2^31 elements).
 */
#ifndef CF_CONV3D_H
#define CF_CONV3D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CF_OK = 0,
    CF_ERR_INVALID_ARG = 1,  /* NULL where a tensor is required, bad sizes, misaligned pointer */
    CF_ERR_UNSUPPORTED = 2,  /* valid request outside the shapes the kernels implement */
    CF_ERR_WORKSPACE = 3,    /* ws_bytes smaller than cf_workspace_size() */
    CF_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, tensor map) */
    CF_ERR_TIMEOUT = 5       /* a kernel abandoned a bounded wait (device status word) */
} cf_status;

/* Geometry of one k=3, pad-1 convolution.  n, d, h, w are the sizes of its
 * input.  stride 0 or 1: the conv output has the same sizes; stride 2 (the
 * hybrid-parallelism page's Table I, layer c4, "stride of 2"): the output is
 *   Z[n,o,co] = sum_{t,ci} W[co,t,ci] * X[n, 2*o + t - 1, ci]
 * with (d+1)/2, (h+1)/2, (w+1)/2 voxels (padding 1 on every face).  A
 * descriptor initialised without the stride member (zero) is stride 1. */
typedef struct {
    int64_t n, d, h, w;
    int32_t c_in, c_out;
    int32_t stride;
} cf_conv_desc;

/* Pooling of the block epilogue. */
enum {
    CF_POOL_MAX = 0,  /* the CosmoFlow block of this library: max over each 2x2x2 window */
    CF_POOL_AVG = 1,  /* average of the activated window (CosmoFlow page, section III-C:
                         constant weights 1/KS^3) */
    CF_POOL_NONE = 2  /* no pooling: y = LReLU(z + b) at the conv output's size
                         (Table I layers after the last pooling) */
};

/* Fused epilogue of the forward conv.  A struct initialised without the pool
 * member (zero) is the max-pool epilogue. */
typedef struct {
    const float* bias; /* [c_out] fp32 device, or NULL for zero bias */
    float slope;       /* leaky-ReLU negative slope (0.3 in the CosmoFlow block) */
    uint8_t* argmax;   /* pooled shape [n][d'/2][h'/2][w'/2][c_out], device, or NULL (inference):
                          CF_POOL_MAX: first-maximum codes dd*4+dh*2+dw;
                          CF_POOL_AVG: sign masks, bit dd*4+dh*2+dw set where z + b > 0
                          (the backward's leaky-ReLU derivatives); CF_POOL_NONE: unused */
    int32_t pool;      /* CF_POOL_MAX, CF_POOL_AVG or CF_POOL_NONE */
} cf_pool_epi;

/* Operation ids for cf_workspace_size. */
enum { CF_OP_FWD = 0, CF_OP_DGRAD = 1, CF_OP_WGRAD = 2, CF_OP_DGRAD_ROUTED = 3,
       CF_OP_WGRAD_ROUTED = 4, CF_OP_POOL_BWD = 5, CF_OP_BN = 6 };

/*
 * Forward convolution (CosmoFlow page, section III-A/III-C "forward data";
 * hybrid-parallelism page, Table I: 3^3 filters, "same" padding).
 *   x  : [n][d][h][w][c_in] bf16
 *   w  : [c_out][3][3][3][c_in] bf16
 *   epi: NULL -> y is the plain conv output Z rounded to bf16, [n][d'][h'][w'][c_out]
 *        (d', h', w' the conv output sizes, see cf_conv_desc);
 *        pool CF_POOL_MAX / CF_POOL_AVG -> y is the pooled block output Y,
 *        [n][d'/2][h'/2][w'/2][c_out], and epi->argmax (if not NULL) receives the
 *        window codes / sign masks; CF_POOL_NONE -> y = LReLU(Z + b), [n][d'][h'][w'][c_out].
 *        Average pooling: Y = (1/8) * sum over the window of LReLU(Z + b).
 *   ws : unused (pass NULL, 0).
 * Supported: c_in in {1, 4} or a multiple of 16 (the CosmoFlow page's rule of
 * channel counts in multiples of 16, section III-A); c_out a multiple of 16, or
 * a multiple of 8 (<= 256) when c_in is 1 or 4; w * c_in a multiple of 8 when c_in is 1 or 4;
 * d', h', w' even when pooling; stride 2 only for c_in a multiple of 16.
 */
cf_status cf_conv3d_fwd(const cf_conv_desc* desc, const uint16_t* x, const uint16_t* w,
                        const cf_pool_epi* epi, uint16_t* y, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * Backward data (CosmoFlow page, section III-C "backward data"):
 *   dX[n,u,ci] = sum_{t,co} W[co,t,ci] * dZ[n, u-(t-1), co]   (dZ = 0 outside)
 * then, if x_act is not NULL, dX *= (x_act > 0 ? 1 : slope): the leaky-ReLU
 * derivative of the previous block, whose pooled output x_act is this conv's
 * input.  The result is stored bf16 in dx [n][d][h][w][c_in].
 *   dz : idx == NULL -> dense dZ [n][d][h][w][c_out] bf16;
 *        idx != NULL -> dz is the pooled pre-activation gradient
 *        [n][d/2][h/2][w/2][c_out] and dZ is its argmax-routed expansion
 *        (written to the workspace first; needs cf_workspace_size(CF_OP_DGRAD_ROUTED)).
 *   w  : the forward filter [c_out][3][3][3][c_in] (flipped and transposed
 *        internally into the workspace).
 *   dsum : NULL, or [c_in] fp32 receiving sum over n and all voxels of the
 *        stored dx (fixed order).  In a block stack dx is the previous block's
 *        pooled pre-activation gradient and dsum its bias gradient (fused into
 *        the epilogue for c_in <= 32, a separate pass over dx otherwise).
 *   stride 2: dz has the conv output's sizes ((d+1)/2 ...); it is written with
 *        zeros at the odd positions into the workspace and the stride-1
 *        backward runs on that (the index map 2*o + t - 1 = u of the forward);
 *        idx must be NULL.
 * Supported: c_out and c_in multiples of 16.
 */
cf_status cf_conv3d_dgrad(const cf_conv_desc* desc, const uint16_t* dz, const uint8_t* idx,
                          const uint16_t* w, const uint16_t* x_act, float slope, uint16_t* dx,
                          float* dsum, void* ws, size_t ws_bytes, void* stream);

/*
 * The filter of the backward-data convolution written as a forward filter
 * (CosmoFlow page, section III-C "backward data": dX is the convolution of dZ
 * with the flipped, transposed filter):
 *   wt[ci][t][co] = w[co][26 - t][ci],  t = 9*kd + 3*kh + kw
 * w: [c_out][27][c_in] bf16; wt: [c_in][27][c_out] bf16; both device,
 * caller-owned, 16-byte aligned.  cf_conv3d_dgrad computes this into its
 * workspace on every call; a caller that reuses one filter, or wants the flip
 * off its critical path (on another stream, before the backward), computes
 * it once here and calls cf_conv3d_dgrad_flipped.
 * Supported: c_out and c_in multiples of 16.
 */
cf_status cf_filter_flip(int32_t c_out, int32_t c_in, const uint16_t* w, uint16_t* wt, void* stream);

/*
 * cf_conv3d_dgrad with the filter given already flipped (wt from
 * cf_filter_flip for this desc's c_out, c_in).  Same arguments, results and
 * workspace size otherwise; bit-identical to cf_conv3d_dgrad.
 */
cf_status cf_conv3d_dgrad_flipped(const cf_conv_desc* desc, const uint16_t* dz, const uint8_t* idx,
                                  const uint16_t* wt, const uint16_t* x_act, float slope, uint16_t* dx,
                                  float* dsum, void* ws, size_t ws_bytes, void* stream);

/*
 * Backward data fused with the previous block's max-pool backward (CosmoFlow
 * page, section III-C "backward data"; the block's pool backward as in
 * cf_bias_lrelu_pool_bwd): everything cf_conv3d_dgrad computes for a dense dz
 * (idx NULL, stride 1) -- dx = the previous block's pooled pre-activation
 * gradient g (x_act given) and optionally its channel sums dsum = that
 * block's bias gradient -- and in the same epilogue
 *   prev_dz [n][2d][2h][2w][c_in] bf16: g routed to the voxel of each 2x2x2
 *           window that prev_idx ([n][d][h][w][c_in], the previous block's
 *           argmax codes) names, zero at the other seven
 * (the previous block's dense dZ, which its weight gradient and backward data
 * read), so that no separate pool-backward pass re-reads g.  Same values, bit
 * for bit, as cf_conv3d_dgrad followed by cf_bias_lrelu_pool_bwd(g, NULL, prev_idx).
 * Supported: as cf_conv3d_dgrad; prev_idx and prev_dz required.
 */
cf_status cf_conv3d_dgrad_pool_bwd(const cf_conv_desc* desc, const uint16_t* dz, const uint16_t* w,
                                   const uint16_t* x_act, float slope, uint16_t* dx, float* dsum,
                                   const uint8_t* prev_idx, uint16_t* prev_dz, void* ws, size_t ws_bytes,
                                   void* stream);

/*
 * Backward weight (CosmoFlow page, section III-C "backward weights", work
 * split over voxels):
 *   dW[co,t,ci] = sum_{n,v} dZ[n,v,co] * X[n, v+(t-1), ci]   (X zero-padded)
 * accumulated in fp32 (split-K over n*d*h*w with a fixed-order reduction).
 *   dz/idx : as in cf_conv3d_dgrad.  For c_in 1 or 4 the routed form is fused:
 *        the kernel expands each K block of dZ in shared memory from the pooled
 *        gradient and the codes (no dense dZ, no workspace beyond the split-K
 *        partials); d, h, w must be even.  Other c_in expand dZ into the
 *        workspace first.  cf_workspace_size(CF_OP_WGRAD_ROUTED) covers both.
 *   dw : [c_out][3][3][3][c_in] fp32; accumulate != 0 adds to it, else overwrites.
 *   stride 2: as in cf_conv3d_dgrad (dz zero-inserted into the workspace; idx NULL).
 * Supported: c_in in {1, 4} (w * c_in a multiple of 8) or a multiple of 16;
 * c_out a multiple of 16 (at most 256 when c_in is 1 or 4).
 */
cf_status cf_conv3d_wgrad(const cf_conv_desc* desc, const uint16_t* x, const uint16_t* dz,
                          const uint8_t* idx, float* dw, int accumulate, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * Standalone bias + leaky ReLU + 2x2x2 max-pool (the fused epilogue of
 * cf_conv3d_fwd as its own HBM-bound kernel).
 *   z   : [n][d][h][w][c] bf16 pre-activation; bias [c] fp32 or NULL
 *   y   : [n][d/2][h/2][w/2][c] bf16;  idx: same shape uint8, or NULL
 * The argmax is taken on the bf16 values of z.  Supported: c a multiple of 8,
 * d, h, w even.
 */
cf_status cf_bias_lrelu_pool_fwd(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                 const uint16_t* z, const float* bias, float slope, uint16_t* y,
                                 uint8_t* idx, void* stream);

/*
 * Pool/LReLU backward.  With g = dy * (y > 0 ? 1 : slope)  (or g = dy when
 * y is NULL, i.e. dy is already the pre-activation gradient):
 *   dz     : [n][d][h][w][c] bf16, g at each window's argmax voxel, 0 at the
 *            other seven; may be NULL
 *   dy_pre : g, pooled shape, bf16; may be NULL
 *   dbias  : [c] fp32, sum of g over n and pooled voxels (fixed-order
 *            reduction through the workspace, cf_workspace_size(CF_OP_POOL_BWD));
 *            may be NULL
 * n,d,h,w are the full-resolution sizes.  Supported: c a multiple of 8.
 */
cf_status cf_bias_lrelu_pool_bwd(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                 const uint16_t* dy, const uint16_t* y, const uint8_t* idx,
                                 float slope, uint16_t* dz, uint16_t* dy_pre, float* dbias,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * cf_bias_lrelu_pool_bwd with its bias-gradient reduction left to the caller,
 * so that it can run on another stream (nothing downstream of the pool
 * backward reads the bias gradient): dz and dy_pre as there; the bias gradient
 * is left as per-block partial sums
 *   partial : [R][c] fp32, R = cf_pool_bwd_partial_rows(), partial_bytes >= 4*R*c
 * and cf_column_sums(R, c, partial, dbias) turns them into the same dbias, bit
 * for bit, as cf_bias_lrelu_pool_bwd.  Supported: as cf_bias_lrelu_pool_bwd.
 */
cf_status cf_bias_lrelu_pool_bwd_partials(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                          const uint16_t* dy, const uint16_t* y, const uint8_t* idx,
                                          float slope, uint16_t* dz, uint16_t* dy_pre, float* partial,
                                          size_t partial_bytes, void* stream);

/* Rows R of the partial sums of cf_bias_lrelu_pool_bwd_partials on the current
 * device (0 on a CUDA error). */
int64_t cf_pool_bwd_partial_rows(void);

/*
 * out[j] = sum over r = 0 .. rows-1, in that order, of partial[r][j]; partial
 * [rows][c] fp32 and out [c] fp32 device pointers.  The fixed-order column
 * reduction of the library's bias gradients.
 */
cf_status cf_column_sums(int64_t rows, int32_t c, const float* partial, float* out, void* stream);

/*
 * The block epilogue of any pooling kind (CF_POOL_*) as standalone kernels:
 * the unfused counterpart of the fused epilogues of cf_conv3d_fwd and the
 * backward that feeds cf_conv3d_dgrad / cf_conv3d_wgrad with a dense dZ.
 * Sources: CosmoFlow page, section III-A (every conv layer followed by leaky
 * ReLU) and III-C (average pooling, constant weights 1/KS^3); hybrid-
 * parallelism page, Table I (stride-2 pooling; layers without pooling).
 *   n, d, h, w : sizes of z / dz (full resolution); d, h, w even when pooling.
 *   forward  : z [n][d][h][w][c] bf16 -> y (pooled shape, or z's for NONE) and
 *              aux (pooled shape uint8: MAX codes, AVG sign masks, NONE unused).
 *   backward : g = dy * LReLU'(y) (MAX with y given; NONE: y given, or dy
 *              itself when y is NULL); MAX routes g to the window's argmax,
 *              AVG writes dz = dy / 8 * LReLU'(z + b) from the masks, NONE
 *              writes dz = g.  dy_pre (MAX only, pooled shape): g.  dbias [c]:
 *              sum of dz over n and voxels (fixed order, workspace of
 *              cf_workspace_size(CF_OP_POOL_BWD)).  Outputs may be NULL.
 * Supported: c a multiple of 8 (at most 2048 in the backward).
 */
cf_status cf_block_epilogue_fwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                const uint16_t* z, const float* bias, float slope, uint16_t* y, uint8_t* aux,
                                void* stream);
cf_status cf_block_epilogue_bwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                const uint16_t* dy, const uint16_t* y, const uint8_t* aux, float slope,
                                uint16_t* dz, uint16_t* dy_pre, float* dbias, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * Batch normalisation between the conv and the activation (the
 * hybrid-parallelism page, section IV: a batch normalization layer after
 * every convolutional layer), training mode with the batch's statistics, per
 * channel over all n and voxels (count = n*d*h*w; biased variance):
 *   u = gamma * (z - mean) / sqrt(var + eps) + beta,  then LReLU and pooling
 * The conv output z is stored (cf_conv3d_fwd with epi NULL), because the
 * statistics need all of it before any voxel can be normalised.
 *   cf_bn_stats        : sums [2c] fp32 = (sum of z, sum of z^2) per channel over
 *                        `rows` voxels of z [rows][c] bf16 (fixed order).
 *   cf_bn_act_pool_fwd : y, aux from z and the sums, as cf_block_epilogue_fwd
 *                        with u in place of z + b (max-pool codes are taken on u).
 *   cf_bn_act_pool_bwd : from dy (pooled shape, or z's for CF_POOL_NONE; with y
 *                        given, dy is the gradient at the block output and the
 *                        leaky-ReLU derivative is applied; with y NULL, dy already
 *                        carries it), du is the pooling backward (max: routed to
 *                        the argmax; avg: dy/8 * LReLU'(u) from the masks; none:
 *                        dy), and
 *                          dgamma = sum du * zh,  dbeta = sum du,
 *                          dz = gamma / sqrt(var + eps) * (du - dbeta/count - zh * dgamma/count)
 *                        written dense to dz [n][d][h][w][c]; dsums [2c] = (dbeta, dgamma).
 * Workspace: cf_workspace_size(CF_OP_BN, desc with c_out = c).  Supported: c a
 * multiple of 8 (<= 2048); d, h, w even when pooling.
 */
cf_status cf_bn_stats(int64_t rows, int32_t c, const uint16_t* z, float* sums, void* ws, size_t ws_bytes,
                      void* stream);
cf_status cf_bn_act_pool_fwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c, const uint16_t* z,
                             const float* sums, const float* gamma, const float* beta, float eps, float slope,
                             uint16_t* y, uint8_t* aux, void* stream);
cf_status cf_bn_act_pool_bwd(int32_t pool, int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                             const uint16_t* dy, const uint16_t* y, const uint8_t* aux, const uint16_t* z,
                             const float* sums, const float* gamma, float eps, float slope, uint16_t* dz,
                             float* dsums, void* ws, size_t ws_bytes, void* stream);

/*
 * The rest of the network around the conv stack (the hybrid-parallelism
 * page, section IV and Table I: fc1 2048 -> fc2 256 -> fc3 4 outputs, leaky
 * ReLU after every layer but the last, dropout with keep probability 0.8
 * after the hidden fully connected layers, mean squared error; Adam with
 * beta1 0.9, beta2 0.999, eps 1e-8).  Activations and weights fp32, row-major;
 * m rows (samples).  Dropout draws are inputs: keep_mask [m][n] uint8 (1 =
 * kept), kept values scaled by 1/keep.
 *   cf_fc_fwd : y [m][n] = act(x [m][k] . w[j] (w [n][k]) + b[j]) masked; act 0 =
 *               linear, 1 = leaky ReLU(slope); x bf16 when x_is_bf16 (e.g. the
 *               flattened NDHWC stack output), else fp32.
 *   cf_fc_bwd : from dy [m][n] (gradient at y), with h = this layer's stored y
 *               (NULL for a linear layer: no leaky-ReLU derivative) and the same
 *               keep_mask / keep: dw [n][k] = sum_i g[i][j] x[i][k], db [n] = sum_i
 *               g[i][j], dx [m][k] = sum_j g[i][j] w[j][k] (bf16 when dx_is_bf16),
 *               g = dy * mask/keep * LReLU'(h); dx, dw, db may be NULL.
 *   cf_mse    : loss [1] = mean of (pred - target)^2 over count values,
 *               dpred = 2 (pred - target) / count (either may be NULL).
 *   cf_adam_step : m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2,
 *               w -= lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), step t >= 1;
 *               w_bf16 (may be NULL) receives w rounded to bf16.
 * Reductions have a fixed order.  Pointers 16-byte aligned.
 */
cf_status cf_fc_fwd(int64_t m, int32_t k, int32_t n, const void* x, int32_t x_is_bf16, const float* w,
                    const float* b, int32_t act, float slope, const uint8_t* keep_mask, float keep, float* y,
                    void* stream);
cf_status cf_fc_bwd(int64_t m, int32_t k, int32_t n, const void* x, int32_t x_is_bf16, const float* w, const float* h,
                    float slope, const uint8_t* keep_mask, float keep, const float* dy, void* dx, int32_t dx_is_bf16,
                    float* dw, float* db, void* stream);
cf_status cf_mse(int64_t count, const float* pred, const float* target, float* loss, float* dpred, void* stream);
cf_status cf_adam_step(int64_t count, float* w, uint16_t* w_bf16, const float* g, float* m, float* v, float lr,
                       float beta1, float beta2, float eps, int64_t t, void* stream);

/*
 * cf_bias_lrelu_pool_bwd without a workspace argument, for callers that
 * cannot allocate device memory (for example an operator plugged into a host
 * framework that owns all device allocations and hands its plug-ins neither
 * an allocator nor a workspace).  The CosmoFlow pages have no counterpart:
 * this is an interface variant, not part of the method.
 *   Arguments, layouts and results: as cf_bias_lrelu_pool_bwd.
 *   Scratch: the bias-gradient partial sums live in a 1 MiB array inside the
 *   library (one per device, held until the process exits).  It holds
 *   4 * SM-count * c floats, so when dbias is requested c may be at most the
 *   largest multiple of 8 not above 65536 / SM-count (424 on a 152-SM GB300,
 *   440 on a 148-SM GPU); a larger c returns CF_ERR_WORKSPACE before anything
 *   is launched.
 *   The first call on a device looks up the array's device address with that
 *   device current; make that first call before any stream capture.  The
 *   address is kept for the life of the process (as is the device status
 *   word's, for every entry point): after a cudaDeviceReset the kept
 *   addresses are stale, so the library must not be used across a device
 *   reset.
 *   Every call shares the array (it keeps the last call's contents; this
 *   operation overwrites every partial it reads, so nothing needs clearing):
 *   calls whose work overlaps on the GPU race on it.
 *   Calls no allocating routine.
 */
cf_status cf_bias_lrelu_pool_bwd_noalloc(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                         const uint16_t* dy, const uint16_t* y, const uint8_t* idx,
                                         float slope, uint16_t* dz, uint16_t* dy_pre, float* dbias,
                                         void* stream);

/* Workspace bytes the operation `op` (CF_OP_*) needs for `desc` (for
 * CF_OP_POOL_BWD desc->c_out is the channel count).  0 if none. */
size_t cf_workspace_size(int op, const cf_conv_desc* desc);

/* Static description of a status code. */
const char* cf_status_string(cf_status s);

/* Synchronises `stream`, then reads and clears the device status word that
 * kernels set when they abandon a bounded wait.  Returns CF_OK or
 * CF_ERR_TIMEOUT (or CF_ERR_CUDA if the synchronisation itself failed). */
cf_status cf_last_device_status(void* stream);

/* Sets the limit, in nanoseconds, after which a kernel abandons a wait on an
 * on-chip barrier (default 2e9).  Affects launches issued afterwards. */
cf_status cf_set_wait_limit_ns(uint64_t ns);

/* Launches a one-CTA kernel that waits on a barrier nothing will ever signal,
 * under the current wait limit; it must come back with the device status word
 * set to CF_ERR_TIMEOUT.  Exercises the timeout path without a GPU fault. */
cf_status cf_debug_wait_timeout_probe(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CF_CONV3D_H */
