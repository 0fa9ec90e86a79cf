// halo_common.cuh -- output-tile shape and epilogue shared by the kernels
// that compute a 2 x 16 x 8 voxel tile as two M=128 accumulators (one per
// plane, row r = 8*line + voxel): the halo-tile implicit GEMM (conv_halo.cu).
// The small-channel first layer (conv_smallc.cu) shares the parameter block.
#pragma once

#include "conv_common.cuh"

namespace cf {

constexpr int HT_W = 8, HT_H = 16, HT_D = 2;                 // output tile
constexpr int HH_W = HT_W + 2, HH_H = HT_H + 2, HH_D = HT_D + 2;  // halo box
constexpr int H_ROWS = HH_W * HH_H * HH_D;                   // 720

struct HaloParams {
    int N, D, H, W, Cin, Cout;
    int tiles_w, tiles_h, tiles_d, n_ntiles, num_tiles, n_chunks;
    FastDiv fd_nt, fd_w, fd_h, fd_d;  // dividers by n_ntiles, tiles_w, tiles_h, tiles_d
    EpiArgs ea;
    int* status;
    uint64_t wait_ns;
};

// Host: the tile-decode dividers of p (after its tile counts are set).
inline void set_tile_dividers(HaloParams& p) {
    p.fd_nt = FastDiv::make((uint32_t)p.n_ntiles);
    p.fd_w = FastDiv::make((uint32_t)p.tiles_w);
    p.fd_h = FastDiv::make((uint32_t)p.tiles_h);
    p.fd_d = FastDiv::make((uint32_t)p.tiles_d);
}

// Tile index -> (N tile, w, h, d, n) tile coordinates, N tile fastest.
struct TileIdx {
    int nt, tw, th, td, n;
};
__device__ __forceinline__ TileIdx tile_index(const HaloParams& p, int tile) {
    TileIdx r;
    uint32_t m = (uint32_t)tile, q = p.fd_nt.div(m);
    r.nt = (int)(m - q * p.fd_nt.d);
    m = q;
    q = p.fd_w.div(m);
    r.tw = (int)(m - q * p.fd_w.d);
    m = q;
    q = p.fd_h.div(m);
    r.th = (int)(m - q * p.fd_h.d);
    m = q;
    q = p.fd_d.div(m);
    r.td = (int)(m - q * p.fd_d.d);
    r.n = (int)q;
    return r;
}

struct HTile {
    int n, d0, h0, w0, co0;
};

__device__ __forceinline__ HTile halo_decode(const HaloParams& p, int tile, int bn) {
    HTile t;
    const TileIdx r = tile_index(p, tile);
    const int nt = r.nt, tw = r.tw, th = r.th;
    t.n = r.n;
    const int td = r.td;
    t.w0 = tw * HT_W;
    t.h0 = th * HT_H;
    t.d0 = td * HT_D;
    t.co0 = nt * bn;
    return t;
}

// (value, code) pair of the first maximum: larger value wins, equal values
// keep the smaller code.
__device__ __forceinline__ void pool_combine(float& v, int& k, float v2, int k2) {
    if (v2 > v || (v2 == v && k2 < k)) {
        v = v2;
        k = k2;
    }
}

// Epilogue of one tile for the accumulator columns c_begin, c_begin + step,
// ... (CH columns per pass); CH = 0 picks min(BN, 32) and step CH.  Several
// warps per TMEM lane quarter can thus split the channels of a tile.
// dsum (backward-data, BN <= 32): per-channel running sums of the stored
// bf16 outputs of this thread's voxels, or NULL.
// add0 / add1: accumulator columns added to plane 0 / plane 1 (partial sums of
// a second issuer), or 0xFFFFFFFF for none.
template <int BN, int EPI, int CH_ = 0>
__device__ __forceinline__ void halo_epilogue(const HaloParams& p, const HTile& t, uint32_t tmem_base,
                                              uint32_t acc_col, int q, int lane, int c_begin = 0,
                                              int c_step = 0, float* dsum = nullptr,
                                              uint32_t add0 = 0xFFFFFFFFu, uint32_t add1 = 0xFFFFFFFFu) {
    constexpr int CH = CH_ != 0 ? CH_ : (BN >= 32 ? 32 : 16);  // accumulator columns per pass
    const int r = q * 32 + lane;
    const int j = r >> 3, l = r & 7;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + acc_col;
    const uint32_t lane_q = tmem_base + ((uint32_t)(q * 32) << 16);
    const int h = t.h0 + j, w = t.w0 + l;
    const int step = c_step != 0 ? c_step : CH;
#pragma unroll 1
    for (int c = c_begin; c < BN; c += step) {
        uint32_t a0[32], a1[32];
        if (CH == 32) {
            tmem_ld32(lane_addr + c, a0);
            tmem_ld32(lane_addr + BN + c, a1);
        } else {
            tmem_ld16(lane_addr + c, a0);
            tmem_ld16(lane_addr + BN + c, a1);
        }
        if (add0 != 0xFFFFFFFFu || add1 != 0xFFFFFFFFu) {  // warp-uniform
            uint32_t b0[32], b1[32];
            if (add0 != 0xFFFFFFFFu) {
                if (CH == 32)
                    tmem_ld32(lane_q + add0 + c, b0);
                else
                    tmem_ld16(lane_q + add0 + c, b0);
            }
            if (add1 != 0xFFFFFFFFu) {
                if (CH == 32)
                    tmem_ld32(lane_q + add1 + c, b1);
                else
                    tmem_ld16(lane_q + add1 + c, b1);
            }
            tmem_ld_wait();
            if (add0 != 0xFFFFFFFFu) {
#pragma unroll
                for (int k = 0; k < CH; ++k) a0[k] = __float_as_uint(__uint_as_float(a0[k]) + __uint_as_float(b0[k]));
            }
            if (add1 != 0xFFFFFFFFu) {
#pragma unroll
                for (int k = 0; k < CH; ++k) a1[k] = __float_as_uint(__uint_as_float(a1[k]) + __uint_as_float(b1[k]));
            }
        }
        tmem_ld_wait();
        // channels of this pass that exist (c_out is a multiple of 8)
        const int nvalid = min(CH, p.Cout - (t.co0 + c));
        if (EPI == EPI_POOL || EPI == EPI_AVG) {
            float bias[CH];  // the pass's bias values, loaded before the reduction chain
#pragma unroll
            for (int cc = 0; cc < CH; ++cc) {
                const int co = t.co0 + c + cc;
                bias[cc] = (p.ea.bias != nullptr && co < p.Cout) ? __ldg(p.ea.bias + co) : 0.f;
            }
            const int D2 = p.D >> 1, H2 = p.H >> 1, W2 = p.W >> 1;
            const int pd = t.d0 >> 1, ph = h >> 1, pw = w >> 1;
            const bool writer = ((j | l) & 1) == 0 && pd < D2 && ph < H2 && pw < W2;
            const int kbase = (j & 1) * 2 + (l & 1);
            uint32_t ybits[CH / 2];
            uint32_t codes[CH / 4];
            constexpr bool avg = EPI == EPI_AVG;
#pragma unroll
            for (int cc = 0; cc < CH; ++cc) {
                float y;
                int k;
                if (avg) {
                    // average of the activated window: this lane's two voxels (planes 0
                    // and 1), then the w and h neighbours; code = the window's sign mask
                    const float s0 = __uint_as_float(a0[cc]) + bias[cc], s1 = __uint_as_float(a1[cc]) + bias[cc];
                    float sum = lrelu(s0, p.ea.slope) + lrelu(s1, p.ea.slope);
                    k = ((s0 > 0.f ? 1 : 0) << kbase) | ((s1 > 0.f ? 1 : 0) << (kbase + 4));
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    k |= __shfl_xor_sync(0xffffffffu, k, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 8);
                    k |= __shfl_xor_sync(0xffffffffu, k, 8);
                    y = sum * 0.125f;
                } else {
                    float v = __uint_as_float(a0[cc]);
                    k = kbase;
                    pool_combine(v, k, __uint_as_float(a1[cc]), kbase + 4);
                    pool_combine(v, k, __shfl_xor_sync(0xffffffffu, v, 1), __shfl_xor_sync(0xffffffffu, k, 1));
                    pool_combine(v, k, __shfl_xor_sync(0xffffffffu, v, 8), __shfl_xor_sync(0xffffffffu, k, 8));
                    y = lrelu(v + bias[cc], p.ea.slope);
                }
                const uint32_t yb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y));
                if (cc & 1)
                    ybits[cc >> 1] |= yb << 16;
                else
                    ybits[cc >> 1] = yb;
                if ((cc & 3) == 0) codes[cc >> 2] = 0;
                codes[cc >> 2] |= (uint32_t)k << (8 * (cc & 3));
            }
            if (writer) {
                const int64_t po = ((((int64_t)t.n * D2 + pd) * H2 + ph) * W2 + pw) * p.Cout + t.co0 + c;
#pragma unroll
                for (int g8 = 0; g8 < CH / 8; ++g8) {
                    if (g8 * 8 >= nvalid) break;
                    *reinterpret_cast<uint4*>(p.ea.y + po + 8 * g8) =
                        make_uint4(ybits[4 * g8], ybits[4 * g8 + 1], ybits[4 * g8 + 2], ybits[4 * g8 + 3]);
                    if (p.ea.idx)
                        *reinterpret_cast<uint2*>(p.ea.idx + po + 8 * g8) = make_uint2(codes[2 * g8], codes[2 * g8 + 1]);
                }
            }
        } else {
            // backward data: the stored activations of this pass's voxels and
            // channels, all loaded before the first store (the stores may alias
            // nothing the compiler can see, so loads inside the store loop would
            // each wait out their latency)
            uint4 xa_all[EPI == EPI_DGRAD ? 2 * (CH / 8) : 1];
            if (EPI == EPI_DGRAD) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int d = t.d0 + i;
                    const bool in = d < p.D && h < p.H && w < p.W;
                    const int64_t o = ((((int64_t)t.n * p.D + d) * p.H + h) * p.W + w) * p.Cout + t.co0 + c;
#pragma unroll
                    for (int q8 = 0; q8 < CH / 8; ++q8)
                        xa_all[i * (CH / 8) + q8] = (in && q8 * 8 < nvalid)
                                                        ? *reinterpret_cast<const uint4*>(p.ea.x_act + o + q8 * 8)
                                                        : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int d = t.d0 + i;
                if (d >= p.D || h >= p.H || w >= p.W) continue;
                const int64_t o = ((((int64_t)t.n * p.D + d) * p.H + h) * p.W + w) * p.Cout + t.co0 + c;
                const uint32_t* a = i == 0 ? a0 : a1;
#pragma unroll
                for (int q8 = 0; q8 < CH / 8; ++q8) {
                    if (q8 * 8 >= nvalid) break;
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(a[q8 * 8 + k]);
                    if (EPI == EPI_ACT) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            v[k] = lrelu(v[k] + (p.ea.bias ? p.ea.bias[t.co0 + c + q8 * 8 + k] : 0.f), p.ea.slope);
                    }
                    if (EPI == EPI_DGRAD) {
                        const uint4 xa = xa_all[EPI == EPI_DGRAD ? i * (CH / 8) + q8 : 0];
                        const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float lo = __uint_as_float(xw[k] << 16);
                            const float hi = __uint_as_float(xw[k] & 0xFFFF0000u);
                            v[2 * k] *= (lo > 0.f ? 1.f : p.ea.slope);
                            v[2 * k + 1] *= (hi > 0.f ? 1.f : p.ea.slope);
                        }
                    }
                    uint4 pk;
                    pk.x = pack_bf16x2(v[0], v[1]);
                    pk.y = pack_bf16x2(v[2], v[3]);
                    pk.z = pack_bf16x2(v[4], v[5]);
                    pk.w = pack_bf16x2(v[6], v[7]);
                    *reinterpret_cast<uint4*>(p.ea.y + o + q8 * 8) = pk;
                    if (EPI == EPI_DGRAD && p.ea.route_dz != nullptr) {
                        const uint2 cv = *reinterpret_cast<const uint2*>(p.ea.route_idx + o + q8 * 8);
                        const int64_t ws = p.Cout, hs = 2 * (int64_t)p.W * p.Cout, ds = 4 * (int64_t)p.H * p.W * p.Cout;
                        uint16_t* dz0 = p.ea.route_dz +
                                        ((((int64_t)t.n * 2 * p.D + 2 * d) * 2 * p.H + 2 * h) * 2 * p.W + 2 * w) * p.Cout +
                                        t.co0 + c + q8 * 8;
                        route_window(dz0, pk, cv, ws, hs, ds);
                    }
                    if (BN <= 32 && dsum != nullptr) {
                        const uint32_t pw[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            dsum[c + q8 * 8 + 2 * k] += __uint_as_float(pw[k] << 16);
                            dsum[c + q8 * 8 + 2 * k + 1] += __uint_as_float(pw[k] & 0xFFFF0000u);
                        }
                    }
                }
            }
        }
    }
}

// The 4-plane tile for c_out 32 (conv_halo4.cu); p carries the problem (sizes,
// epilogue arguments), the tile counts are its own.
bool halo4_path_supported(int c_in, int c_out);
cf_status launch_conv_halo4(const LaunchCtx& ctx, const HaloParams& p, const uint16_t* x, const uint16_t* wk,
                            int epi);

}  // namespace cf
