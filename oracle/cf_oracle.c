/*
 * cf_oracle.c -- plain, slow, fp64 CPU oracle for the CosmoFlow conv3d block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the bench's
 * CPU-baseline leg load it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Every routine is the textbook definition written out as direct nested loops
 * in double precision (OpenMP only splits independent outputs across threads;
 * each output is summed in the same order as the single-threaded loop).
 *
 * Sources for what is computed (page title, section):
 *  - "CosmoFlow: Using Deep Learning to Learn the Universe at Scale" (summary
 *    of arXiv 1808.04728v2), section III-A: 3D convolution layers, every conv
 *    layer followed by leaky ReLU; section III-C: forward data, backward data
 *    and backward weight operators of the convolution; pooling averages or
 *    selects per channel.
 *  - "The Case for Strong Scaling in Deep Learning: Training Large 3D CNNs
 *    with Hybrid Parallelism", section IV, Table I: 3^3 filters, stride-1
 *    convolution with "same" padding, stride-2 pooling.
 *  - The block studied here: conv3d k=3 stride 1 pad 1, + bias, leaky ReLU with
 *    slope 0.3, 2x2x2 max-pool stride 2.  The pages do not state the slope;
 *    0.3 and max-pooling are the readings this build fixes.
 *
 * Conventions (readings of points the pages leave open):
 *  - "convolution" is cross-correlation (no filter flip in the forward pass),
 *    zero padding of one voxel on every face;
 *  - layouts are NDHWC for activations and [C_out][3][3][3][C_in] for filters;
 *  - max-pool picks the FIRST maximum in (dd,dh,dw) lexicographic order using a
 *    strict '>' scan, and records it as code dd*4+dh*2+dw;
 *  - the pool is taken on the pre-bias value m; y = LReLU(m + b).  Adding a
 *    constant and applying LReLU are both monotone non-decreasing, so this
 *    equals pooling after the activation;
 *  - LReLU'(z) = 1 if z > 0 else slope (so slope at exactly zero).
 *
 * Parity: every function here is pinned by tests that do not call it twice
 * (dense-operator brute force, a library correlation routine, shift and
 * constant-input identities, adjoint identities, finite differences, pooling
 * closed forms).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#define I5(n, d, h, w, c, D, H, W, C) \
    (((((int64_t)(n) * (D) + (d)) * (H) + (h)) * (W) + (w)) * (int64_t)(C) + (c))
/* filter element W[co][kd][kh][kw][ci] */
#define IW(co, kd, kh, kw, ci, Ci) \
    (((((int64_t)(co) * 3 + (kd)) * 3 + (kh)) * 3 + (kw)) * (int64_t)(Ci) + (ci))

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dabs(double v) { return v < 0 ? -v : v; }

/* ------------------------------------------------------------------------ */
/* Forward: z[n,d,h,w,co] = sum_{kd,kh,kw,ci} W[co,kd,kh,kw,ci] *
 *                          x[n, d+kd-1, h+kh-1, w+kw-1, ci]   (x = 0 outside). */
void oracle_conv3d_fwd(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                       const double* x, const double* wt, double* z)
{
    int64_t planes = N * D;
#pragma omp parallel for schedule(static)
    for (int64_t nd = 0; nd < planes; ++nd) {
        int64_t n = nd / D, d = nd % D;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t w = 0; w < W; ++w)
                for (int32_t co = 0; co < Co; ++co) {
                    double acc = 0.0;
                    for (int kd = 0; kd < 3; ++kd) {
                        int64_t id = d + kd - 1;
                        if (id < 0 || id >= D) continue;
                        for (int kh = 0; kh < 3; ++kh) {
                            int64_t ih = h + kh - 1;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < 3; ++kw) {
                                int64_t iw = w + kw - 1;
                                if (iw < 0 || iw >= W) continue;
                                const double* xp = x + I5(n, id, ih, iw, 0, D, H, W, Ci);
                                const double* wp = wt + IW(co, kd, kh, kw, 0, Ci);
                                for (int32_t ci = 0; ci < Ci; ++ci) acc += wp[ci] * xp[ci];
                            }
                        }
                    }
                    z[I5(n, d, h, w, co, D, H, W, Co)] = acc;
                }
    }
}

/* Backward data: dx[n,u,ci] = sum_{t,co} W[co,t,ci] * dz[n, u-(t-1), co]
 * (dz = 0 outside the volume).  Written as the gather over the taps that
 * reach voxel u. */
void oracle_conv3d_dgrad(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                         const double* dz, const double* wt, double* dx)
{
    int64_t planes = N * D;
#pragma omp parallel for schedule(static)
    for (int64_t nd = 0; nd < planes; ++nd) {
        int64_t n = nd / D, d = nd % D;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t w = 0; w < W; ++w)
                for (int32_t ci = 0; ci < Ci; ++ci) {
                    double acc = 0.0;
                    for (int kd = 0; kd < 3; ++kd) {
                        int64_t od = d - (kd - 1);
                        if (od < 0 || od >= D) continue;
                        for (int kh = 0; kh < 3; ++kh) {
                            int64_t oh = h - (kh - 1);
                            if (oh < 0 || oh >= H) continue;
                            for (int kw = 0; kw < 3; ++kw) {
                                int64_t ow = w - (kw - 1);
                                if (ow < 0 || ow >= W) continue;
                                const double* gp = dz + I5(n, od, oh, ow, 0, D, H, W, Co);
                                for (int32_t co = 0; co < Co; ++co)
                                    acc += wt[IW(co, kd, kh, kw, ci, Ci)] * gp[co];
                            }
                        }
                    }
                    dx[I5(n, d, h, w, ci, D, H, W, Ci)] = acc;
                }
    }
}

/* Backward weight: dW[co,t,ci] = sum_{n,v} dz[n,v,co] * x[n, v+(t-1), ci]. */
void oracle_conv3d_wgrad(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                         const double* x, const double* dz, double* dw)
{
    int64_t items = (int64_t)Co * 27;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < items; ++it) {
        int32_t co = (int32_t)(it / 27);
        int t = (int)(it % 27), kd = t / 9, kh = (t / 3) % 3, kw = t % 3;
        for (int32_t ci = 0; ci < Ci; ++ci) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                for (int64_t d = 0; d < D; ++d) {
                    int64_t id = d + kd - 1;
                    if (id < 0 || id >= D) continue;
                    for (int64_t h = 0; h < H; ++h) {
                        int64_t ih = h + kh - 1;
                        if (ih < 0 || ih >= H) continue;
                        for (int64_t w = 0; w < W; ++w) {
                            int64_t iw = w + kw - 1;
                            if (iw < 0 || iw >= W) continue;
                            acc += dz[I5(n, d, h, w, co, D, H, W, Co)] *
                                   x[I5(n, id, ih, iw, ci, D, H, W, Ci)];
                        }
                    }
                }
            dw[IW(co, kd, kh, kw, ci, Ci)] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Bias + leaky ReLU + 2x2x2 max-pool, stride 2.  z is the full-resolution conv
 * output [N][D][H][W][C]; y and idx are [N][D/2][H/2][W/2][C]. */
void oracle_pool_fwd(int64_t N, int64_t D, int64_t H, int64_t W, int32_t C,
                     const double* z, const double* bias, double slope,
                     double* y, uint8_t* idx)
{
    int64_t D2 = D / 2, H2 = H / 2, W2 = W / 2;
    int64_t planes = N * D2;
#pragma omp parallel for schedule(static)
    for (int64_t np = 0; np < planes; ++np) {
        int64_t n = np / D2, pd = np % D2;
        for (int64_t ph = 0; ph < H2; ++ph)
            for (int64_t pw = 0; pw < W2; ++pw)
                for (int32_t c = 0; c < C; ++c) {
                    double m = 0.0;
                    int code = -1;
                    for (int dd = 0; dd < 2; ++dd)
                        for (int dh = 0; dh < 2; ++dh)
                            for (int dw = 0; dw < 2; ++dw) {
                                double v = z[I5(n, 2 * pd + dd, 2 * ph + dh, 2 * pw + dw, c, D, H, W, C)];
                                if (code < 0 || v > m) {
                                    m = v;
                                    code = dd * 4 + dh * 2 + dw;
                                }
                            }
                    double s = m + (bias ? bias[c] : 0.0);
                    int64_t o = I5(n, pd, ph, pw, c, D2, H2, W2, C);
                    y[o] = s > 0 ? s : slope * s;
                    if (idx) idx[o] = (uint8_t)code;
                }
    }
}

/* Pool/LReLU backward.
 *  dy      : gradient w.r.t. the pooled output y            [N][D/2][H/2][W/2][C]
 *  y       : the pooled output (for LReLU'), or NULL when dy is already the
 *            gradient w.r.t. the pooled pre-activation m+b
 *  idx     : argmax codes from the forward pass
 *  dz      : (out, optional) full-resolution gradient w.r.t. z: g at the argmax
 *            voxel of each window, 0 at the other seven  [N][D][H][W][C]
 *  dy_pre  : (out, optional) g itself, pooled shape
 *  db      : (out, optional) [C]: sum over n and pooled voxels of g
 * with g = dy * (y > 0 ? 1 : slope). */
void oracle_pool_bwd(int64_t N, int64_t D, int64_t H, int64_t W, int32_t C,
                     const double* dy, const double* y, const uint8_t* idx, double slope,
                     double* dz, double* dy_pre, double* db)
{
    int64_t D2 = D / 2, H2 = H / 2, W2 = W / 2;
    if (dz) memset(dz, 0, sizeof(double) * (size_t)(N * D * H * W * C));
    if (db)
        for (int32_t c = 0; c < C; ++c) db[c] = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t pd = 0; pd < D2; ++pd)
            for (int64_t ph = 0; ph < H2; ++ph)
                for (int64_t pw = 0; pw < W2; ++pw)
                    for (int32_t c = 0; c < C; ++c) {
                        int64_t o = I5(n, pd, ph, pw, c, D2, H2, W2, C);
                        double g = dy[o];
                        if (y) g *= (y[o] > 0 ? 1.0 : slope);
                        if (dy_pre) dy_pre[o] = g;
                        if (db) db[c] += g;
                        if (dz) {
                            int code = idx[o];
                            int dd = (code >> 2) & 1, dh = (code >> 1) & 1, dw = code & 1;
                            dz[I5(n, 2 * pd + dd, 2 * ph + dh, 2 * pw + dw, c, D, H, W, C)] = g;
                        }
                    }
}

/* ------------------------------------------------------------------------ */
/* Sampled versions on bf16 inputs, for sizes where the full tensors are too
 * large to evaluate in fp64 on the host.  Each returns the exact fp64 value of
 * the requested output elements and S = the sum of |product| terms of that
 * element (the scale of its rounding error). */

/* pts: npts x (n,d,h,w,co) */
void oracle_conv3d_fwd_pts_bf16(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                                const uint16_t* x, const uint16_t* wt,
                                int64_t npts, const int64_t* pts, double* out, double* sabs)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t p = 0; p < npts; ++p) {
        int64_t n = pts[5 * p], d = pts[5 * p + 1], h = pts[5 * p + 2], w = pts[5 * p + 3];
        int32_t co = (int32_t)pts[5 * p + 4];
        double acc = 0.0, sa = 0.0;
        for (int kd = 0; kd < 3; ++kd) {
            int64_t id = d + kd - 1;
            if (id < 0 || id >= D) continue;
            for (int kh = 0; kh < 3; ++kh) {
                int64_t ih = h + kh - 1;
                if (ih < 0 || ih >= H) continue;
                for (int kw = 0; kw < 3; ++kw) {
                    int64_t iw = w + kw - 1;
                    if (iw < 0 || iw >= W) continue;
                    for (int32_t ci = 0; ci < Ci; ++ci) {
                        double t = bf16_to_double(wt[IW(co, kd, kh, kw, ci, Ci)]) *
                                   bf16_to_double(x[I5(n, id, ih, iw, ci, D, H, W, Ci)]);
                        acc += t;
                        sa += dabs(t);
                    }
                }
            }
        }
        out[p] = acc;
        if (sabs) sabs[p] = sa;
    }
}

/* pts: npts x (n,d,h,w,ci) */
void oracle_conv3d_dgrad_pts_bf16(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                                  const uint16_t* dz, const uint16_t* wt,
                                  int64_t npts, const int64_t* pts, double* out, double* sabs)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t p = 0; p < npts; ++p) {
        int64_t n = pts[5 * p], d = pts[5 * p + 1], h = pts[5 * p + 2], w = pts[5 * p + 3];
        int32_t ci = (int32_t)pts[5 * p + 4];
        double acc = 0.0, sa = 0.0;
        for (int kd = 0; kd < 3; ++kd) {
            int64_t od = d - (kd - 1);
            if (od < 0 || od >= D) continue;
            for (int kh = 0; kh < 3; ++kh) {
                int64_t oh = h - (kh - 1);
                if (oh < 0 || oh >= H) continue;
                for (int kw = 0; kw < 3; ++kw) {
                    int64_t ow = w - (kw - 1);
                    if (ow < 0 || ow >= W) continue;
                    for (int32_t co = 0; co < Co; ++co) {
                        double t = bf16_to_double(wt[IW(co, kd, kh, kw, ci, Ci)]) *
                                   bf16_to_double(dz[I5(n, od, oh, ow, co, D, H, W, Co)]);
                        acc += t;
                        sa += dabs(t);
                    }
                }
            }
        }
        out[p] = acc;
        if (sabs) sabs[p] = sa;
    }
}

/* pts: npts x (co,kd,kh,kw,ci); sums over every sample and voxel. */
void oracle_conv3d_wgrad_pts_bf16(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                                  const uint16_t* x, const uint16_t* dz,
                                  int64_t npts, const int64_t* pts, double* out, double* sabs)
{
    for (int64_t p = 0; p < npts; ++p) {
        int32_t co = (int32_t)pts[5 * p];
        int kd = (int)pts[5 * p + 1], kh = (int)pts[5 * p + 2], kw = (int)pts[5 * p + 3];
        int32_t ci = (int32_t)pts[5 * p + 4];
        double acc = 0.0, sa = 0.0;
        int64_t planes = N * D;
#pragma omp parallel for schedule(static) reduction(+ : acc, sa)
        for (int64_t nd = 0; nd < planes; ++nd) {
            int64_t n = nd / D, d = nd % D;
            int64_t id = d + kd - 1;
            if (id < 0 || id >= D) continue;
            for (int64_t h = 0; h < H; ++h) {
                int64_t ih = h + kh - 1;
                if (ih < 0 || ih >= H) continue;
                for (int64_t w = 0; w < W; ++w) {
                    int64_t iw = w + kw - 1;
                    if (iw < 0 || iw >= W) continue;
                    double t = bf16_to_double(dz[I5(n, d, h, w, co, D, H, W, Co)]) *
                               bf16_to_double(x[I5(n, id, ih, iw, ci, D, H, W, Ci)]);
                    acc += t;
                    sa += dabs(t);
                }
            }
        }
        out[p] = acc;
        if (sabs) sabs[p] = sa;
    }
}

/* Fused block at sampled pooled outputs: for each (n,pd,ph,pw,co) evaluates
 * the eight conv outputs of its window (bf16 inputs, fp64 sums), the first
 * maximum m and its code, y = LReLU(m + b), S at the argmax voxel, and the gap
 * between the largest and second-largest of the eight values. */
void oracle_block_fwd_pts_bf16(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                               const uint16_t* x, const uint16_t* wt, const float* bias, double slope,
                               int64_t npts, const int64_t* pts,
                               double* y, uint8_t* idx, double* sabs, double* gap)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t p = 0; p < npts; ++p) {
        int64_t q[5 * 8];
        double zv[8], zs[8];
        for (int k = 0; k < 8; ++k) {
            int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
            q[5 * k + 0] = pts[5 * p];
            q[5 * k + 1] = 2 * pts[5 * p + 1] + dd;
            q[5 * k + 2] = 2 * pts[5 * p + 2] + dh;
            q[5 * k + 3] = 2 * pts[5 * p + 3] + dw;
            q[5 * k + 4] = pts[5 * p + 4];
        }
        /* serial evaluation of the eight window voxels */
        for (int k = 0; k < 8; ++k) {
            int64_t n = q[5 * k], d = q[5 * k + 1], h = q[5 * k + 2], w = q[5 * k + 3];
            int32_t co = (int32_t)q[5 * k + 4];
            double acc = 0.0, sa = 0.0;
            for (int kd = 0; kd < 3; ++kd) {
                int64_t id = d + kd - 1;
                if (id < 0 || id >= D) continue;
                for (int kh = 0; kh < 3; ++kh) {
                    int64_t ih = h + kh - 1;
                    if (ih < 0 || ih >= H) continue;
                    for (int kw = 0; kw < 3; ++kw) {
                        int64_t iw = w + kw - 1;
                        if (iw < 0 || iw >= W) continue;
                        for (int32_t ci = 0; ci < Ci; ++ci) {
                            double t = bf16_to_double(wt[IW(co, kd, kh, kw, ci, Ci)]) *
                                       bf16_to_double(x[I5(n, id, ih, iw, ci, D, H, W, Ci)]);
                            acc += t;
                            sa += dabs(t);
                        }
                    }
                }
            }
            zv[k] = acc;
            zs[k] = sa;
        }
        int code = 0;
        for (int k = 1; k < 8; ++k)
            if (zv[k] > zv[code]) code = k;
        double second = -1e300;
        for (int k = 0; k < 8; ++k)
            if (k != code && zv[k] > second) second = zv[k];
        double b = bias ? (double)bias[pts[5 * p + 4]] : 0.0;
        double s = zv[code] + b;
        y[p] = s > 0 ? s : slope * s;
        idx[p] = (uint8_t)code;
        sabs[p] = zs[code] + dabs(b);
        gap[p] = zv[code] - second;
    }
    (void)N;
    (void)Co;
}

/* Backward weight at sampled filter elements when dZ is the argmax-routed
 * expansion of a pooled gradient (the max-pool backward): dz[n,v,co] equals
 * g[n,p,co] at the voxel v = 2p + (dd,dh,dw) whose code dd*4+dh*2+dw is
 * idx[n,p,co], and 0 at the other seven voxels of the window.  The sum
 *   dW[co,t,ci] = sum_{n,v} dz[n,v,co] * x[n, v+(t-1), ci]
 * therefore runs over the pooled voxels p, one routed voxel each.
 * g, idx: [N][D/2][H/2][W/2][Co]; x: [N][D][H][W][Ci]; D, H, W even.
 * pts: npts x (co,kd,kh,kw,ci). */
void oracle_conv3d_wgrad_routed_pts_bf16(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                                         const uint16_t* x, const uint16_t* g, const uint8_t* idx,
                                         int64_t npts, const int64_t* pts, double* out, double* sabs)
{
    int64_t D2 = D / 2, H2 = H / 2, W2 = W / 2;
    for (int64_t p = 0; p < npts; ++p) {
        int32_t co = (int32_t)pts[5 * p];
        int kd = (int)pts[5 * p + 1], kh = (int)pts[5 * p + 2], kw = (int)pts[5 * p + 3];
        int32_t ci = (int32_t)pts[5 * p + 4];
        double acc = 0.0, sa = 0.0;
        int64_t planes = N * D2;
#pragma omp parallel for schedule(static) reduction(+ : acc, sa)
        for (int64_t np = 0; np < planes; ++np) {
            int64_t n = np / D2, pd = np % D2;
            for (int64_t ph = 0; ph < H2; ++ph)
                for (int64_t pw = 0; pw < W2; ++pw) {
                    int64_t o = I5(n, pd, ph, pw, co, D2, H2, W2, Co);
                    int code = idx[o];
                    int64_t d = 2 * pd + ((code >> 2) & 1), h = 2 * ph + ((code >> 1) & 1), w = 2 * pw + (code & 1);
                    int64_t id = d + kd - 1, ih = h + kh - 1, iw = w + kw - 1;
                    if (id < 0 || id >= D || ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
                    double t = bf16_to_double(g[o]) * bf16_to_double(x[I5(n, id, ih, iw, ci, D, H, W, Ci)]);
                    acc += t;
                    sa += dabs(t);
                }
        }
        out[p] = acc;
        if (sabs) sabs[p] = sa;
    }
}

/* ------------------------------------------------------------------------ */
/* Page variants ("next" rows).
 *
 * Average pooling (CosmoFlow page, section III-C: pooling averages each
 * channel separately with constant weights 1/KS^3; section III-A: every conv
 * layer is followed by leaky ReLU): the block is conv -> + bias -> leaky ReLU
 * -> 2x2x2 average, so
 *   y[p] = (1/8) * sum_{v in window(p)} LReLU(z[v] + b)
 * and its backward
 *   dz[v] = dy[p] / 8 * LReLU'(z[v] + b),   db = sum over v of dz[v].
 * Unlike the max-pool, pooling does not commute with the activation here, so
 * the backward needs the sign of every pre-activation of the window; mask[p]
 * records it (bit dd*4+dh*2+dw set where z + b > 0). */
void oracle_avgpool_fwd(int64_t N, int64_t D, int64_t H, int64_t W, int32_t C,
                        const double* z, const double* bias, double slope, double* y, uint8_t* mask)
{
    int64_t D2 = D / 2, H2 = H / 2, W2 = W / 2;
    int64_t planes = N * D2;
#pragma omp parallel for schedule(static)
    for (int64_t np = 0; np < planes; ++np) {
        int64_t n = np / D2, pd = np % D2;
        for (int64_t ph = 0; ph < H2; ++ph)
            for (int64_t pw = 0; pw < W2; ++pw)
                for (int32_t c = 0; c < C; ++c) {
                    double sum = 0.0;
                    int m = 0;
                    for (int dd = 0; dd < 2; ++dd)
                        for (int dh = 0; dh < 2; ++dh)
                            for (int dw = 0; dw < 2; ++dw) {
                                double s = z[I5(n, 2 * pd + dd, 2 * ph + dh, 2 * pw + dw, c, D, H, W, C)] +
                                           (bias ? bias[c] : 0.0);
                                if (s > 0) m |= 1 << (dd * 4 + dh * 2 + dw);
                                sum += s > 0 ? s : slope * s;
                            }
                    int64_t o = I5(n, pd, ph, pw, c, D2, H2, W2, C);
                    y[o] = sum / 8.0;
                    if (mask) mask[o] = (uint8_t)m;
                }
    }
}

/* dz (full resolution) and db from dy (pooled) and the pre-activation signs. */
void oracle_avgpool_bwd(int64_t N, int64_t D, int64_t H, int64_t W, int32_t C,
                        const double* dy, const uint8_t* mask, double slope, double* dz, double* db)
{
    int64_t D2 = D / 2, H2 = H / 2, W2 = W / 2;
    if (db)
        for (int32_t c = 0; c < C; ++c) db[c] = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t pd = 0; pd < D2; ++pd)
            for (int64_t ph = 0; ph < H2; ++ph)
                for (int64_t pw = 0; pw < W2; ++pw)
                    for (int32_t c = 0; c < C; ++c) {
                        int64_t o = I5(n, pd, ph, pw, c, D2, H2, W2, C);
                        for (int k = 0; k < 8; ++k) {
                            int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
                            double g = dy[o] / 8.0 * (((mask[o] >> k) & 1) ? 1.0 : slope);
                            if (dz) dz[I5(n, 2 * pd + dd, 2 * ph + dh, 2 * pw + dw, c, D, H, W, C)] = g;
                            if (db) db[c] += g;
                        }
                    }
}

/* Unpooled block (layers of the hybrid-parallelism page's Table I after the
 * last pooling: convolution followed by leaky ReLU only):
 *   y = LReLU(z + b);  backward dz = dy * LReLU'(y), db = sum of dz
 * (y > 0 exactly where z + b > 0). */
void oracle_act_fwd(int64_t count, int32_t C, const double* z, const double* bias, double slope, double* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        double s = z[i] + (bias ? bias[i % C] : 0.0);
        y[i] = s > 0 ? s : slope * s;
    }
}

void oracle_act_bwd(int64_t count, int32_t C, const double* dy, const double* y, double slope, double* dz,
                    double* db)
{
    if (db)
        for (int32_t c = 0; c < C; ++c) db[c] = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        double g = dy[i] * (y[i] > 0 ? 1.0 : slope);
        if (dz) dz[i] = g;
        if (db) db[i % C] += g;
    }
}

/* Stride-2 convolution (Table I, layer c4: "stride of 2"), padding 1 on
 * every face ("same" padding), output [N][Do][Ho][Wo] with Do = (D + 1) / 2:
 *   z[n,o,co] = sum_{t,ci} W[co,t,ci] * x[n, 2*o + t - 1, ci]    (o = (od,oh,ow))
 * backward data and weight by the same index map:
 *   dx[n,u,ci] = sum over (t, o) with 2*o + t - 1 = u of W[co,t,ci] * dz[n,o,co]
 *   dW[co,t,ci] = sum_{n,o} dz[n,o,co] * x[n, 2*o + t - 1, ci]. */
void oracle_conv3d_fwd_s2(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                          const double* x, const double* wt, double* z)
{
    int64_t Do = (D + 1) / 2, Ho = (H + 1) / 2, Wo = (W + 1) / 2;
    int64_t planes = N * Do;
#pragma omp parallel for schedule(static)
    for (int64_t np = 0; np < planes; ++np) {
        int64_t n = np / Do, od = np % Do;
        for (int64_t oh = 0; oh < Ho; ++oh)
            for (int64_t ow = 0; ow < Wo; ++ow)
                for (int32_t co = 0; co < Co; ++co) {
                    double acc = 0.0;
                    for (int kd = 0; kd < 3; ++kd) {
                        int64_t id = 2 * od + kd - 1;
                        if (id < 0 || id >= D) continue;
                        for (int kh = 0; kh < 3; ++kh) {
                            int64_t ih = 2 * oh + kh - 1;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < 3; ++kw) {
                                int64_t iw = 2 * ow + kw - 1;
                                if (iw < 0 || iw >= W) continue;
                                for (int32_t ci = 0; ci < Ci; ++ci)
                                    acc += wt[IW(co, kd, kh, kw, ci, Ci)] * x[I5(n, id, ih, iw, ci, D, H, W, Ci)];
                            }
                        }
                    }
                    z[I5(n, od, oh, ow, co, Do, Ho, Wo, Co)] = acc;
                }
    }
}

/* dz: [N][Do][Ho][Wo][Co]; dx: [N][D][H][W][Ci].  Scatter form over (o, t). */
void oracle_conv3d_dgrad_s2(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                            const double* dz, const double* wt, double* dx)
{
    int64_t Do = (D + 1) / 2, Ho = (H + 1) / 2, Wo = (W + 1) / 2;
    memset(dx, 0, sizeof(double) * (size_t)(N * D * H * W * Ci));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t od = 0; od < Do; ++od)
            for (int64_t oh = 0; oh < Ho; ++oh)
                for (int64_t ow = 0; ow < Wo; ++ow)
                    for (int kd = 0; kd < 3; ++kd) {
                        int64_t id = 2 * od + kd - 1;
                        if (id < 0 || id >= D) continue;
                        for (int kh = 0; kh < 3; ++kh) {
                            int64_t ih = 2 * oh + kh - 1;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < 3; ++kw) {
                                int64_t iw = 2 * ow + kw - 1;
                                if (iw < 0 || iw >= W) continue;
                                for (int32_t co = 0; co < Co; ++co) {
                                    double g = dz[I5(n, od, oh, ow, co, Do, Ho, Wo, Co)];
                                    for (int32_t ci = 0; ci < Ci; ++ci)
                                        dx[I5(n, id, ih, iw, ci, D, H, W, Ci)] += wt[IW(co, kd, kh, kw, ci, Ci)] * g;
                                }
                            }
                        }
                    }
}

void oracle_conv3d_wgrad_s2(int64_t N, int64_t D, int64_t H, int64_t W, int32_t Ci, int32_t Co,
                            const double* x, const double* dz, double* dw)
{
    int64_t Do = (D + 1) / 2, Ho = (H + 1) / 2, Wo = (W + 1) / 2;
    int64_t items = (int64_t)Co * 27;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < items; ++it) {
        int32_t co = (int32_t)(it / 27);
        int t = (int)(it % 27), kd = t / 9, kh = (t / 3) % 3, kw = t % 3;
        for (int32_t ci = 0; ci < Ci; ++ci) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                for (int64_t od = 0; od < Do; ++od) {
                    int64_t id = 2 * od + kd - 1;
                    if (id < 0 || id >= D) continue;
                    for (int64_t oh = 0; oh < Ho; ++oh) {
                        int64_t ih = 2 * oh + kh - 1;
                        if (ih < 0 || ih >= H) continue;
                        for (int64_t ow = 0; ow < Wo; ++ow) {
                            int64_t iw = 2 * ow + kw - 1;
                            if (iw < 0 || iw >= W) continue;
                            acc += dz[I5(n, od, oh, ow, co, Do, Ho, Wo, Co)] * x[I5(n, id, ih, iw, ci, D, H, W, Ci)];
                        }
                    }
                }
            dw[IW(co, kd, kh, kw, ci, Ci)] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Batch normalisation after the convolution (the hybrid-parallelism page,
 * section IV: "a batch normalization layer after every convolutional layer"),
 * in training mode with the statistics of the batch, per channel c over all
 * n and voxels (count = N*D*H*W):
 *   mu = mean(z),  var = mean((z - mu)^2)  (biased),  zh = (z - mu) / sqrt(var + eps)
 *   u = gamma * zh + beta
 * followed by the block's leaky ReLU and pooling.  Backward, from du:
 *   dgamma = sum(du * zh),  dbeta = sum(du)
 *   dz = gamma / sqrt(var + eps) * (du - dbeta / count - zh * dgamma / count).
 * z, u, du, dz: [count][C]; mean, var, dgamma, dbeta: [C]. */
void oracle_bn_fwd(int64_t count, int32_t C, const double* z, const double* gamma, const double* beta, double eps,
                   double* u, double* mean, double* var)
{
    for (int32_t c = 0; c < C; ++c) {
        double s = 0.0;
        for (int64_t i = 0; i < count; ++i) s += z[i * C + c];
        double mu = s / (double)count;
        double q = 0.0;
        for (int64_t i = 0; i < count; ++i) {
            double t = z[i * C + c] - mu;
            q += t * t;
        }
        double v = q / (double)count;
        double inv = 1.0 / sqrt(v + eps);
        for (int64_t i = 0; i < count; ++i) u[i * C + c] = gamma[c] * (z[i * C + c] - mu) * inv + beta[c];
        if (mean) mean[c] = mu;
        if (var) var[c] = v;
    }
}

void oracle_bn_bwd(int64_t count, int32_t C, const double* z, const double* du, const double* gamma, double eps,
                   double* dz, double* dgamma, double* dbeta)
{
    for (int32_t c = 0; c < C; ++c) {
        double s = 0.0;
        for (int64_t i = 0; i < count; ++i) s += z[i * C + c];
        double mu = s / (double)count;
        double q = 0.0;
        for (int64_t i = 0; i < count; ++i) {
            double t = z[i * C + c] - mu;
            q += t * t;
        }
        double inv = 1.0 / sqrt(q / (double)count + eps);
        double sg = 0.0, sb = 0.0;
        for (int64_t i = 0; i < count; ++i) {
            double zh = (z[i * C + c] - mu) * inv;
            sg += du[i * C + c] * zh;
            sb += du[i * C + c];
        }
        for (int64_t i = 0; i < count; ++i) {
            double zh = (z[i * C + c] - mu) * inv;
            dz[i * C + c] = gamma[c] * inv * (du[i * C + c] - sb / (double)count - zh * sg / (double)count);
        }
        if (dgamma) dgamma[c] = sg;
        if (dbeta) dbeta[c] = sb;
    }
}
