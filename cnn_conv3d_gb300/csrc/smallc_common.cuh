// smallc_common.cuh -- input staging for the small-channel layer (c_in 1 or 4,
// the first CosmoFlow conv): a halo tile of the input loaded by TMA, and the
// per-voxel gather of the 27 taps (im2col row) from it.
//
// The activation is viewed as a 4-D tensor (W*C, H, D, N) so that a TMA box
// can start on a 16-byte boundary although one voxel is only 2 or 8 bytes: the
// box starts HW0 = 16 / (2*C) voxels left of the tile and is TW + 2*HW0 voxels
// wide; out-of-range coordinates read as zero, which is the conv padding.
#pragma once

#include "conv_common.cuh"

namespace cf {

template <int CIN>
struct HaloGeom {
    static constexpr int HW0 = 16 / (2 * CIN);  // voxels of left margin (2 for c=4, 8 for c=1)
};

__host__ __device__ constexpr int halo_line_voxels(int tw, int cin) { return tw + 2 * (16 / (2 * cin)); }
__host__ __device__ constexpr int halo_bytes(int tw, int th, int td, int cin) {
    return (td + 2) * (th + 2) * halo_line_voxels(tw, cin) * cin * 2;
}

// Loads the halo of the tile at (n, d0, h0, w0): box (line, th+2, td+2).
template <int CIN>
__device__ __forceinline__ void load_halo(void* dst, const CUtensorMap* m, uint64_t* bar, int n, int d0, int h0,
                                          int w0) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(m), "r"(smem_u32(bar)), "r"((w0 - HaloGeom<CIN>::HW0) * CIN), "r"(h0 - 1), "r"(d0 - 1), "r"(n)
        : "memory");
}

// Gathers the im2col row of voxel (i, j, l) of the tile -- K index k = 4*t + ci
// for c_in = 4 (54 32-bit words, bf16 pairs, t = 9*kd + 3*kh + kw) -- from the
// halo tile.  The centre voxel of each of the 9 (kd, kh) lines is read from
// shared memory; its w-1 and w+1 neighbours come from the adjacent lanes
// (rows of a line are consecutive lanes), except at the ends of the line.
// Must be called by full warps (shuffles).
__device__ __forceinline__ void gather_row_c4(const uint8_t* halo, int tw, int th, int i, int j, int l,
                                              uint32_t (&wd)[56]) {
    const int pitch = halo_line_voxels(tw, 4) * 8;  // bytes per halo line
#pragma unroll
    for (int kd = 0; kd < 3; ++kd) {
#pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
            const uint8_t* line = halo + ((i + kd) * (th + 2) + (j + kh)) * pitch;
            const uint2 mid = *reinterpret_cast<const uint2*>(line + (l + 2) * 8);
            uint2 left, right;
            left.x = __shfl_up_sync(0xffffffffu, mid.x, 1);
            left.y = __shfl_up_sync(0xffffffffu, mid.y, 1);
            right.x = __shfl_down_sync(0xffffffffu, mid.x, 1);
            right.y = __shfl_down_sync(0xffffffffu, mid.y, 1);
            if (l == 0) left = *reinterpret_cast<const uint2*>(line + (l + 1) * 8);
            if (l == tw - 1) right = *reinterpret_cast<const uint2*>(line + (l + 3) * 8);
            const int t0 = kd * 9 + kh * 3;
            wd[2 * t0 + 0] = left.x;
            wd[2 * t0 + 1] = left.y;
            wd[2 * t0 + 2] = mid.x;
            wd[2 * t0 + 3] = mid.y;
            wd[2 * t0 + 4] = right.x;
            wd[2 * t0 + 5] = right.y;
        }
    }
    wd[54] = 0u;
    wd[55] = 0u;
}

// Same for c_in = 1: K index k = t (27 values padded to 32), 16 words.
__device__ __forceinline__ void gather_row_c1(const uint8_t* halo, int tw, int th, int i, int j, int l,
                                              uint32_t (&wd)[56]) {
    const int pitch = halo_line_voxels(tw, 1) * 2;
    uint32_t v[32];
#pragma unroll
    for (int kd = 0; kd < 3; ++kd)
#pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
            const uint16_t* line = reinterpret_cast<const uint16_t*>(halo + ((i + kd) * (th + 2) + (j + kh)) * pitch);
#pragma unroll
            for (int kw = 0; kw < 3; ++kw) v[kd * 9 + kh * 3 + kw] = line[l + 8 + kw - 1];
        }
#pragma unroll
    for (int t = 27; t < 32; ++t) v[t] = 0u;
#pragma unroll
    for (int q = 0; q < 16; ++q) wd[q] = v[2 * q] | (v[2 * q + 1] << 16);
#pragma unroll
    for (int q = 16; q < 56; ++q) wd[q] = 0u;
}

// Host: the halo tensor map over x viewed as (W*C, H, D, N).
bool make_halo_map(CUtensorMap* m, const uint16_t* x, int n, int d, int h, int w, int cin, int tw, int th, int td);

}  // namespace cf
