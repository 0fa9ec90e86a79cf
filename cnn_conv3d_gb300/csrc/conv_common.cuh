// conv_common.cuh -- pieces shared by the forward/backward-data implicit-GEMM
// kernels: tile decoding and the fused epilogues that read the fp32
// accumulator out of tensor memory.
#pragma once

#include <algorithm>

#include "cf_internal.h"
#include "cf_ptx.cuh"
#include "fastdiv.cuh"

namespace cf {

// Output tile of 128 voxels: box (TD=2) x th x tw starting at (d0,h0,w0) of
// sample n, and output channels [co0, co0 + BN).
struct TileCoord {
    int n, d0, h0, w0, co0;
};

struct ConvGeom {
    int N, D, H, W;
    int Cin, Cout;  // GEMM view: K = 27 * Cin, N-dimension = Cout
    int tw, th, td;
    int lw, lh;  // log2(tw), log2(th): the tile extents are powers of two
    int tiles_w, tiles_h, tiles_d;
    int n_ntiles;
    int num_tiles;
    FastDiv fd_nt, fd_w, fd_h, fd_d;  // dividers by n_ntiles, tiles_w, tiles_h, tiles_d
};

__device__ __forceinline__ TileCoord decode_tile(const ConvGeom& g, int tile, int bn) {
    TileCoord c;
    uint32_t m = (uint32_t)tile, q = g.fd_nt.div(m);
    const int nt = (int)(m - q * g.fd_nt.d);
    m = q;
    q = g.fd_w.div(m);
    const int tw = (int)(m - q * g.fd_w.d);
    m = q;
    q = g.fd_h.div(m);
    const int th = (int)(m - q * g.fd_h.d);
    m = q;
    q = g.fd_d.div(m);
    const int td = (int)(m - q * g.fd_d.d);
    c.n = (int)q;
    c.w0 = tw * g.tw;
    c.h0 = th * g.th;
    c.d0 = td * g.td;
    c.co0 = nt * bn;
    return c;
}

// The epilogue warps wait for an accumulator through one leader thread, which
// then releases the other 127 with a named barrier: a wait that gives up is
// thus seen by all of them, and none is left behind at a later named barrier.
__device__ __forceinline__ bool epi_wait(uint64_t* bar, uint32_t parity, int et, volatile int* flag,
                                         volatile int* abort, uint64_t limit_ns, int* status, int nthreads = 128) {
    if (et == 0) *flag = mbar_wait(bar, parity, abort, limit_ns, status, WAIT_EPI_TMEM_FULL) ? 1 : 0;
    named_bar_sync(2, nthreads);
    return *flag != 0;
}

struct EpiArgs {
    uint16_t* y;
    uint8_t* idx;
    const float* bias;
    const uint16_t* x_act;
    float slope;
    // backward-data only: per-CTA channel sums of the stored outputs,
    // [gridDim.x][C] fp32 (rows of CTAs without tiles stay as they were), or NULL
    float* colsum_part = nullptr;
    // EPI_DGRAD, optional: the previous block's max-pool backward fused in.  The
    // stored output (the previous block's pooled pre-activation gradient g, same
    // NDHWC grid as y) is also routed to its window's argmax voxel in route_dz
    // ([n][2d][2h][2w][C] bf16, zero at the other seven voxels), by the codes
    // route_idx (same grid as y).
    uint16_t* route_dz = nullptr;
    const uint8_t* route_idx = nullptr;
};

__device__ __forceinline__ float lrelu(float s, float slope) { return s > 0.f ? s : slope * s; }

// 32-bit masks, all ones where the code byte of a channel differs from `code`
// (channels 2h, 2h+1 of the word: half h).  Bit 7 of each byte of
// ((b ^ code) & 0x7f) + 0x7f, or of b ^ code, is set iff the byte differs; the
// permute replicates that bit over two bytes.
__device__ __forceinline__ void code_mismatch(uint32_t codes4, uint32_t code4, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = codes4 ^ code4;
    const uint32_t nz = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x;
    asm("prmt.b32 %0, %1, 0, 0x9988;" : "=r"(lo) : "r"(nz));
    asm("prmt.b32 %0, %1, 0, 0xBBAA;" : "=r"(hi) : "r"(nz));
}

// Max-pool backward of one pooled voxel x 8 channels: the bf16 values `pk`
// (channels 2i, 2i+1 in word i) written to the window voxel whose code
// dd*4+dh*2+dw the channel's code byte (cv) names, zero to the other seven.
// dz0 points at channel c0 of window voxel (0,0,0); the window's other voxels
// are dw*ws + dh*hs + dd*ds elements away.
__device__ __forceinline__ void route_window(uint16_t* dz0, uint4 pk, uint2 cv, int64_t ws, int64_t hs,
                                             int64_t ds) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t code4 = (uint32_t)k * 0x01010101u;
        uint32_t m0, m1, m2, m3;
        code_mismatch(cv.x, code4, m0, m1);
        code_mismatch(cv.y, code4, m2, m3);
        *reinterpret_cast<uint4*>(dz0 + (k >> 2) * ds + ((k >> 1) & 1) * hs + (k & 1) * ws) =
            make_uint4(pk.x & ~m0, pk.y & ~m1, pk.z & ~m2, pk.w & ~m3);
    }
}

// Epilogue of one tile, executed by the 128 epilogue threads (4 warps whose
// warp index modulo 4 is q; thread row = 32*q + lane is TMEM lane = GEMM row).
//   acc_col : first TMEM column of this tile's accumulator
//   stg     : [128][33] fp32 staging buffer (EPI_POOL only)
//   et      : epilogue thread id 0..127
template <int BN, int EPI>
__device__ __forceinline__ void conv_epilogue(const ConvGeom& g, const TileCoord& tc, const EpiArgs& ea,
                                              uint32_t tmem_base, uint32_t acc_col, int q, int lane, int et,
                                              float* stg) {
    constexpr int CH = BN >= 32 ? 32 : 16;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + acc_col;
    const int l = row & (g.tw - 1), j = (row >> g.lw) & (g.th - 1), i = row >> (g.lw + g.lh);
    const int d = tc.d0 + i, h = tc.h0 + j, w = tc.w0 + l;
    const bool valid = d < g.D && h < g.H && w < g.W;
    const int64_t vox = (((int64_t)tc.n * g.D + d) * g.H + h) * g.W + w;

#pragma unroll 1
    for (int c = 0; c < BN; c += CH) {
        uint32_t r[32];
        if (CH == 32)
            tmem_ld32(lane_addr + c, r);
        else
            tmem_ld16(lane_addr + c, r);
        tmem_ld_wait();
        if (EPI == EPI_POOL || EPI == EPI_AVG) {
#pragma unroll
            for (int k = 0; k < CH; ++k) stg[row * 33 + k] = __uint_as_float(r[k]);
            named_bar_sync(1, 128);
            constexpr int CPT = CH / 8;  // channels per thread
            const int wi = et >> 3;      // 16 windows per tile
            const int tw2 = g.tw >> 1;
            const int pw_l = wi % tw2, ph_l = wi / tw2;
            const int cb = (et & 7) * CPT;
            const int D2 = g.D >> 1, H2 = g.H >> 1, W2 = g.W >> 1;
            const int pd = tc.d0 >> 1, ph = (tc.h0 >> 1) + ph_l, pw = (tc.w0 >> 1) + pw_l;
            if (pd < D2 && ph < H2 && pw < W2) {
                const int64_t po = ((((int64_t)tc.n * D2 + pd) * H2 + ph) * W2 + pw) * g.Cout + tc.co0 + c + cb;
                float yv[CPT];
                uint32_t codes = 0;
#pragma unroll
                for (int cc = 0; cc < CPT; ++cc) {
                    const int co = tc.co0 + c + cb + cc;
                    const float b = (ea.bias != nullptr && co < g.Cout) ? ea.bias[co] : 0.f;
                    if (EPI == EPI_AVG) {
                        // average of the activated window; code = the window's sign mask
                        float sum = 0.f;
                        int mask = 0;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
                            const int rr = (dd * g.th + 2 * ph_l + dh) * g.tw + 2 * pw_l + dw;
                            const float s = stg[rr * 33 + cb + cc] + b;
                            mask |= (s > 0.f ? 1 : 0) << k;
                            sum += lrelu(s, ea.slope);
                        }
                        yv[cc] = sum * 0.125f;
                        codes |= (uint32_t)mask << (8 * cc);
                        continue;
                    }
                    float m = 0.f;
                    int code = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int dd = k >> 2, dh = (k >> 1) & 1, dw = k & 1;
                        const int rr = (dd * g.th + 2 * ph_l + dh) * g.tw + 2 * pw_l + dw;
                        const float v = stg[rr * 33 + cb + cc];
                        if (k == 0 || v > m) {
                            m = v;
                            code = k;
                        }
                    }
                    yv[cc] = lrelu(m + b, ea.slope);
                    codes |= (uint32_t)code << (8 * cc);
                }
                const int co_first = tc.co0 + c + cb;
                if (co_first + CPT <= g.Cout) {
                    if (CPT == 4) {
                        uint2 pk;
                        pk.x = pack_bf16x2(yv[0], yv[1]);
                        pk.y = pack_bf16x2(yv[2 % CPT], yv[3 % CPT]);
                        *reinterpret_cast<uint2*>(ea.y + po) = pk;
                        if (ea.idx) *reinterpret_cast<uint32_t*>(ea.idx + po) = codes;
                    } else {
                        *reinterpret_cast<uint32_t*>(ea.y + po) = pack_bf16x2(yv[0], yv[1 % CPT]);
                        if (ea.idx) *reinterpret_cast<uint16_t*>(ea.idx + po) = (uint16_t)codes;
                    }
                }
            }
            named_bar_sync(1, 128);
        } else if (valid) {
            const int64_t o = vox * g.Cout + tc.co0 + c;
#pragma unroll
            for (int q8 = 0; q8 < CH / 8; ++q8) {
                if (tc.co0 + c + q8 * 8 + 8 > g.Cout) break;
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(r[q8 * 8 + k]);
                if (EPI == EPI_ACT) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        v[k] = lrelu(v[k] + (ea.bias ? ea.bias[tc.co0 + c + q8 * 8 + k] : 0.f), ea.slope);
                }
                if (EPI == EPI_DGRAD) {
                    const uint4 xa = *reinterpret_cast<const uint4*>(ea.x_act + o + q8 * 8);
                    const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = __uint_as_float(xw[k] << 16);
                        const float hi = __uint_as_float(xw[k] & 0xFFFF0000u);
                        v[2 * k] *= (lo > 0.f ? 1.f : ea.slope);
                        v[2 * k + 1] *= (hi > 0.f ? 1.f : ea.slope);
                    }
                }
                uint4 pk;
                pk.x = pack_bf16x2(v[0], v[1]);
                pk.y = pack_bf16x2(v[2], v[3]);
                pk.z = pack_bf16x2(v[4], v[5]);
                pk.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4*>(ea.y + o + q8 * 8) = pk;
                if (EPI == EPI_DGRAD && ea.route_dz != nullptr) {
                    const uint2 cv = *reinterpret_cast<const uint2*>(ea.route_idx + o + q8 * 8);
                    const int64_t ws = g.Cout, hs = 2 * (int64_t)g.W * g.Cout, ds = 4 * (int64_t)g.H * g.W * g.Cout;
                    uint16_t* dz0 = ea.route_dz +
                                    ((((int64_t)tc.n * 2 * g.D + 2 * d) * 2 * g.H + 2 * h) * 2 * g.W + 2 * w) * g.Cout +
                                    tc.co0 + c + q8 * 8;
                    route_window(dz0, pk, cv, ws, hs, ds);
                }
            }
        }
    }
}

// ---- host helpers shared by the conv launchers
inline ConvGeom make_geom(int64_t n, int64_t d, int64_t h, int64_t w, int cin, int cout, int bn) {
    ConvGeom g;
    g.N = (int)n;
    g.D = (int)d;
    g.H = (int)h;
    g.W = (int)w;
    g.Cin = cin;
    g.Cout = cout;
    TileGeom t = choose_tile(d, h, w);
    g.tw = t.tw;
    g.th = t.th;
    g.td = t.td;
    g.lw = 0;
    while ((1 << g.lw) < g.tw) ++g.lw;
    g.lh = 0;
    while ((1 << g.lh) < g.th) ++g.lh;
    g.tiles_w = (int)((w + t.tw - 1) / t.tw);
    g.tiles_h = (int)((h + t.th - 1) / t.th);
    g.tiles_d = (int)((d + t.td - 1) / t.td);
    g.n_ntiles = (cout + bn - 1) / bn;
    g.num_tiles = (int)(n * g.tiles_d * g.tiles_h * g.tiles_w * g.n_ntiles);
    g.fd_nt = FastDiv::make((uint32_t)g.n_ntiles);
    g.fd_w = FastDiv::make((uint32_t)g.tiles_w);
    g.fd_h = FastDiv::make((uint32_t)g.tiles_h);
    g.fd_d = FastDiv::make((uint32_t)g.tiles_d);
    return g;
}

template <typename K>
inline int grid_for(K kernel, uint32_t smem, int threads, int num_sms, int num_tiles, uint32_t tmem_cols) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    per_sm = std::min<int>(per_sm, (int)(512 / tmem_cols));
    return std::max(1, std::min(num_tiles, num_sms * per_sm));
}

}  // namespace cf
