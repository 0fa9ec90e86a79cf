// wgrad_common.cuh -- split-K bookkeeping shared by the backward-weight
// kernels that walk voxel boxes (conv_wgrad.cu, conv_wgrad_smallc.cu): the box
// geometry, a division-free box cursor, and the store of a unit's fp32
// accumulator into the partial buffer that the fixed-order reduction sums.
#pragma once

#include "conv_common.cuh"

namespace cf {

struct WgradGeom {
    int N, D, H, W, Cin, Cout;
    int vw, vh, vd;           // voxel box (K block)
    int nb_w, nb_h, nb_d;     // boxes per dimension
    int64_t total_boxes;      // N * nb_d * nb_h * nb_w
    int n_mblocks;            // ceil(27*Cin / 128)
    int n_ntiles;             // output-channel tiles of bn channels (the last may be partly beyond Cout)
    int bn;                   // channels per N tile
    int n_splits;
    int64_t boxes_per_split;
    int num_units;            // n_mblocks * n_ntiles * n_splits
};

// Box cursor: decodes a linear box index once, then steps through the boxes
// with carries (no divisions on the per-stage path).
struct BoxCursor {
    int n, bd, bh, bw;
    __device__ __forceinline__ void init(const WgradGeom& g, int64_t b) {
        bw = (int)(b % g.nb_w);
        b /= g.nb_w;
        bh = (int)(b % g.nb_h);
        b /= g.nb_h;
        bd = (int)(b % g.nb_d);
        n = (int)(b / g.nb_d);
    }
    __device__ __forceinline__ void next(const WgradGeom& g) {
        if (++bw == g.nb_w) {
            bw = 0;
            if (++bh == g.nb_h) {
                bh = 0;
                if (++bd == g.nb_d) {
                    bd = 0;
                    ++n;
                }
            }
        }
    }
};

// Writes the unit's accumulator rows (t,ci) < 27*Cin, channels co0 + c < Cout,
// into part[split][co][row].
template <int BN>
__device__ __forceinline__ void wgrad_store_partial(const WgradGeom& g, float* part, int mb, int split, int co0,
                                                    uint32_t tmem_base, int q, int lane) {
    const int row = q * 32 + lane;
    const int mrow = mb * 128 + row;
    const int KK = 27 * g.Cin;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
    float* base = part + ((int64_t)split * g.Cout + co0) * KK + mrow;
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
        uint32_t r[32];
        tmem_ld16(lane_addr + c, r);
        tmem_ld_wait();
        if (mrow < KK) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (co0 + c + k < g.Cout) base[(int64_t)(c + k) * KK] = __uint_as_float(r[k]);
        }
    }
}

// conv_wgrad_smallc.cu: the small-channel (c_in 1 or 4) kernel writing the
// unit partials for geometry g (voxel box 16 x 4 x 2).  idx != NULL: dz is the
// pooled pre-activation gradient [n][d/2][h/2][w/2][c_out] and idx its argmax
// codes; the dense dZ is expanded in shared memory.
cf_status launch_wgrad_smallc(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                              const uint8_t* idx, float* part);

}  // namespace cf
