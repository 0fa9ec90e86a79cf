// conv_halo4.cu -- the halo-tile forward / backward-data convolution with a
// 4-plane output tile for GEMM N = c_out = 32 (the layer-2 backward data:
// dZ 64 -> dX 32 channels), input channels in chunks of 16, the whole filter
// resident in shared memory.
//
// Output tile: 4 planes x 16 lines x 8 voxels (512 voxels).  With N = 32 the
// MMAs of the 2-plane tile (conv_halo.cu) are bound by the shared-memory reads
// of their operands (128 bytes per cycle; an MMA 128 x N x 16 with A in shared
// memory takes max(N/2, 32 + N/4) cycles).  Halo plane p feeds output planes
// p-2, p-1, p through the filter depth taps kd = 2, 1, 0 with the SAME A
// operand, so one MMA of width up to 3N takes B = the three slabs of one
// (kh, kw) stacked (kd = 2 above 1 above 0) and writes up to three plane
// accumulators N columns apart.  Two issuers split the six halo planes:
//   warp 1: halo planes 0, 1, 2 -> accumulator set A = output planes 0, 1, 2
//           (widths N, 2N, 3N);
//   warp 6: halo planes 3, 4, 5 -> accumulator set B = output planes 1, 2, 3
//           (widths 3N, 2N, N);
// each set is N x 3 columns, and the epilogue adds the two sets' partial sums
// of planes 1 and 2.  Per (kh, kw) and 16-channel K step that is 288 cycles
// of operand reads for 4 output planes, against 2 x 176 for two 2-plane
// tiles; each issuer's three MMAs stay within one thread's issue rate (~55
// cycles per MMA).  The first MMA of a tile in each set (halo plane 2, resp.
// 3: all three of the set's planes) overwrites; the others accumulate.
//
// Halo box per chunk: (16 channels, 10 voxels, 18 lines, 6 planes) with
// 32-byte swizzled rows, three stages in flight; the filter, 27 taps x c_in
// x 32 channels, is loaded once per CTA, slabs in the order (chunk, kh, kw,
// kd = 2, 1, 0).
//
// Warps: 0 TMA producer, 1 and 6 MMA issuers (warp 1 allocates tensor
// memory), 2..5 the epilogue (the 2-plane epilogue run on planes 0, 1 and
// then 2, 3).
#include "halo_common.cuh"

namespace cf {

namespace {

constexpr int H4_PL = 4;          // output planes per tile
constexpr int H4_HD = H4_PL + 2;  // halo planes
constexpr int H4_KC = 16;         // input channels per chunk
constexpr int H4_BN = 32;         // GEMM N (output channels)
constexpr uint32_t H4_ROW = H4_KC * 2;
constexpr uint32_t H4_HALO_BYTES = HH_W * HH_H * H4_HD * H4_ROW;  // 34560
constexpr uint32_t H4_HALO_STRIDE = (H4_HALO_BYTES + 1023) / 1024 * 1024;
constexpr int H4_HS = 3;
constexpr uint32_t H4_W_BYTES = H4_BN * H4_KC * 2;  // one tap's slab: 1 KB
constexpr uint32_t H4_BAR_BYTES = 512;
constexpr uint32_t H4_SBO_A = HH_W * H4_ROW;  // one halo line
constexpr uint32_t H4_SBO_B = 8 * H4_ROW;
constexpr uint32_t H4_SET = 3 * H4_BN;        // columns of one accumulator set
constexpr uint32_t H4_ACC_STRIDE = 2 * H4_SET;  // one tile: set A | set B
constexpr uint32_t H4_TMEM_COLS = 512;          // two tiles (384 columns) in flight
constexpr uint32_t H4_IDESC1 = idesc_bf16(128, H4_BN, 0, 0);
constexpr uint32_t H4_IDESC2 = idesc_bf16(128, 2 * H4_BN, 0, 0);
constexpr uint32_t H4_IDESC3 = idesc_bf16(128, 3 * H4_BN, 0, 0);
static_assert(2 * H4_ACC_STRIDE <= H4_TMEM_COLS, "tensor memory");

uint32_t h4_smem_bytes(int c_in) {
    return 1024 + H4_HS * H4_HALO_STRIDE + (uint32_t)(c_in / H4_KC) * 27 * H4_W_BYTES + H4_BAR_BYTES;
}

__device__ __forceinline__ HTile h4_decode(const HaloParams& p, int tile) {
    const TileIdx r = tile_index(p, tile);
    HTile t;
    t.n = r.n;
    t.w0 = r.tw * HT_W;
    t.h0 = r.th * HT_H;
    t.d0 = r.td * H4_PL;
    t.co0 = 0;
    return t;
}

template <int EPI>
__global__ void __launch_bounds__(224, 1)
    conv_halo4_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const HaloParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* hring = smem;
    uint8_t* wsm = smem + H4_HS * H4_HALO_STRIDE;
    const uint32_t w_region = (uint32_t)p.n_chunks * 27 * H4_W_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + w_region);
    uint64_t* hfull = bars;
    uint64_t* hempty = hfull + H4_HS;
    uint64_t* tfull = hempty + H4_HS;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;  // [2]
    uint64_t* wres = drain + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(wres + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        // halo stages are released and accumulators completed by both issuers
        for (int s = 0; s < H4_HS; ++s) {
            mbar_init(&hfull[s], 1);
            mbar_init(&hempty[s], 2);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 2);
            mbar_init(&tempty[a], 128);
            mbar_init(&drain[a], 1);
        }
        mbar_init(wres, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, H4_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: the filter once, then per tile and chunk one
            // halo box (16, 10, 18, 6)
            int hs = 0;
            uint32_t hph = 0, hiss = 0, hpar = 0;
            bool ok = true, res_issued = false;
            if (blockIdx.x < p.num_tiles) {
                mbar_arrive_expect_tx(wres, w_region);
                for (int ch = 0; ch < p.n_chunks; ++ch)
                    for (int tap = 0; tap < 27; ++tap) {
                        const int kd = tap / 9, r = tap - 9 * kd;  // slot (kh, kw, 2 - kd)
                        tma_load_2d(wsm + (ch * 27 + r * 3 + (2 - kd)) * H4_W_BYTES, &tmW, wres,
                                    tap * p.Cin + ch * H4_KC, 0);
                    }
                res_issued = true;
            }
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                const HTile t = h4_decode(p, tile);
                for (int ch = 0; ch < p.n_chunks; ++ch) {
                    if (!mbar_wait(&hempty[hs], hph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&hfull[hs], H4_HALO_BYTES);
                    tma_load_5d(hring + hs * H4_HALO_STRIDE, &tmX, &hfull[hs], ch * H4_KC, t.w0 - 1, t.h0 - 1,
                                t.d0 - 1, t.n);
                    hiss |= 1u << hs;
                    hpar = (hpar & ~(1u << hs)) | (hph << hs);
                    if (++hs == H4_HS) {
                        hs = 0;
                        hph ^= 1;
                    }
                }
            }
            // copies in flight must land before the CTA exits
            if (res_issued) mbar_wait_timed(wres, 0, p.wait_ns);
            if (!ok) {
                for (int s = 0; s < H4_HS; ++s)
                    if (hiss & (1u << s)) mbar_wait_timed(&hfull[s], (hpar >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 6) {
        if (lane == 0) {
            // ---------------- MMA issuers: warp 1 halo planes 0-2 into set A, warp 6
            // halo planes 3-5 into set B
            const int i = warp == 1 ? 0 : 1;
            int hs = 0;
            uint32_t hph = 0, local = 0;
            bool ok = true;
            const uint64_t adesc0 = sdesc(smem_u32(hring), 16, H4_SBO_A, SWZ_32B);
            const uint64_t bdesc0 = sdesc(smem_u32(wsm), 16, H4_SBO_B, SWZ_32B);
            if (blockIdx.x < p.num_tiles) ok = mbar_wait(wres, 0, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL);
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t acc = local & 1, use = local >> 1;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dset = tmem_base + acc * H4_ACC_STRIDE + i * H4_SET;
                for (int ch = 0; ch < p.n_chunks && ok; ++ch) {
                    if (!mbar_wait(&hfull[hs], hph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ah = adesc0 + ((hs * H4_HALO_STRIDE) >> 4);
#pragma unroll 1
                    for (int g = 0; g < 9; ++g) {
                        const int kh = g / 3, kw = g - 3 * (g / 3);
                        const uint64_t ag = ah + (((uint32_t)(kh * HH_W + kw) * H4_ROW) >> 4);
                        const uint64_t bg = bdesc0 + (((uint32_t)(ch * 27 + g * 3) * H4_W_BYTES) >> 4);
                        const bool first = (ch | g) == 0;
                        // the full-width plane first (it starts all three of the set's sums)
#pragma unroll
                        for (int o = 0; o < 3; ++o) {
                            // set A: halo planes 2, 0, 1; set B: 3, 5, 4
                            const int hp = i == 0 ? (o == 0 ? 2 : o - 1) : (o == 0 ? 3 : (o == 1 ? 5 : 4));
                            const int kdmax = hp < 2 ? hp : 2;
                            const int kdmin = hp - (H4_PL - 1) > 0 ? hp - (H4_PL - 1) : 0;
                            const int span = kdmax - kdmin + 1;
                            const uint32_t idesc = span == 1 ? H4_IDESC1 : (span == 2 ? H4_IDESC2 : H4_IDESC3);
                            // output plane of the first slab (kd = kdmax): j0 = hp - kdmax; set B
                            // holds planes 1..3 from its column 0
                            const int j0 = hp - kdmax - i;
                            const uint64_t a = ag + (((uint32_t)(hp * HH_H * HH_W) * H4_ROW) >> 4);
                            const uint64_t b = bg + (((uint32_t)(2 - kdmax) * H4_W_BYTES) >> 4);
                            umma_bf16(dset + (uint32_t)j0 * H4_BN, a, b, idesc, (first && o == 0) ? 0u : 1u);
                        }
                    }
                    umma_commit(&hempty[hs]);
                    if (++hs == H4_HS) {
                        hs = 0;
                        hph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
            }
            if (!ok) {
                umma_commit(&drain[i]);
                mbar_wait_timed(&drain[i], 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- epilogue warps 2..5: plane 0 = A0, plane 1 = A1 + B0,
        // plane 2 = A2 + B1, plane 3 = B2
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        constexpr bool DSUM = EPI == EPI_PLAIN || EPI == EPI_DGRAD;
        const bool dsum_on = DSUM && p.ea.colsum_part != nullptr;
        float dsum[DSUM ? H4_BN : 1];
#pragma unroll
        for (int c = 0; c < (DSUM ? H4_BN : 1); ++c) dsum[c] = 0.f;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1, use = local >> 1;
            if (!epi_wait(&tfull[acc], use & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            HTile t = h4_decode(p, tile);
            const uint32_t a0 = acc * H4_ACC_STRIDE, b0 = a0 + H4_SET;
            halo_epilogue<H4_BN, EPI>(p, t, tmem_base, a0, q, lane, 0, 0, dsum_on ? dsum : nullptr, 0xFFFFFFFFu, b0);
            t.d0 += 2;
            if (t.d0 < p.D)
                halo_epilogue<H4_BN, EPI>(p, t, tmem_base, b0 + H4_BN, q, lane, 0, 0, dsum_on ? dsum : nullptr,
                                          a0 + 2 * H4_BN, 0xFFFFFFFFu);
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if (dsum_on) {
            // the last tile's MMAs are complete, so the halo ring is idle: reduce
            // the 128 threads' sums through it (thread order, then one row per CTA)
            float* red = reinterpret_cast<float*>(hring);
            named_bar_sync(2, 128);
#pragma unroll
            for (int c = 0; c < (DSUM ? H4_BN : 1); ++c) red[et * (H4_BN + 1) + c] = dsum[c];
            named_bar_sync(2, 128);
            if (et < H4_BN && et < p.Cout) {
                float s = 0.f;
                for (int r = 0; r < 128; ++r) s += red[r * (H4_BN + 1) + et];
                p.ea.colsum_part[(int64_t)blockIdx.x * p.Cout + et] = s;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, H4_TMEM_COLS);
    }
}

template <int EPI>
cf_status run_halo4(const LaunchCtx& ctx, HaloParams p, const uint16_t* x, const uint16_t* wk) {
    CUtensorMap tx, tw;
    const uint64_t dx[5] = {(uint64_t)p.Cin, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.D, (uint64_t)p.N};
    const uint64_t sx[4] = {(uint64_t)p.Cin * 2, (uint64_t)p.W * p.Cin * 2, (uint64_t)p.H * p.W * p.Cin * 2,
                            (uint64_t)p.D * p.H * p.W * p.Cin * 2};
    const uint32_t bx[5] = {(uint32_t)H4_KC, (uint32_t)HH_W, (uint32_t)HH_H, (uint32_t)H4_HD, 1u};
    if (!encode_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dx, sx, bx, CU_TENSOR_MAP_SWIZZLE_32B))
        return CF_ERR_CUDA;
    const uint64_t dw[2] = {(uint64_t)27 * p.Cin, (uint64_t)p.Cout};
    const uint64_t sw[1] = {(uint64_t)27 * p.Cin * 2};
    const uint32_t bw[2] = {(uint32_t)H4_KC, (uint32_t)H4_BN};
    if (!encode_tmap(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wk, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_32B))
        return CF_ERR_CUDA;
    const uint32_t smem = h4_smem_bytes(p.Cin);
    auto kern = conv_halo4_kernel<EPI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = grid_for(kern, smem, 224, ctx.num_sms, p.num_tiles, H4_TMEM_COLS);
    kern<<<grid, 224, smem, ctx.stream>>>(tx, tw, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

}  // namespace

// c_out 32 and a filter (27 x c_in x 32 bf16) that fits beside three halo
// stages: c_in a multiple of 16 up to 64.
bool halo4_path_supported(int c_in, int c_out) {
    return c_out == H4_BN && c_in % H4_KC == 0 && h4_smem_bytes(c_in) <= 227 * 1024;
}

cf_status launch_conv_halo4(const LaunchCtx& ctx, const HaloParams& p0, const uint16_t* x, const uint16_t* wk,
                            int epi) {
    if (!halo4_path_supported(p0.Cin, p0.Cout)) return CF_ERR_UNSUPPORTED;
    HaloParams p = p0;
    p.tiles_d = (p.D + H4_PL - 1) / H4_PL;
    p.n_ntiles = 1;
    p.num_tiles = p.N * p.tiles_d * p.tiles_h * p.tiles_w;
    set_tile_dividers(p);
    p.n_chunks = p.Cin / H4_KC;
    switch (epi) {
        case EPI_PLAIN: return run_halo4<EPI_PLAIN>(ctx, p, x, wk);
        case EPI_POOL: return run_halo4<EPI_POOL>(ctx, p, x, wk);
        case EPI_AVG: return run_halo4<EPI_AVG>(ctx, p, x, wk);
        case EPI_ACT: return run_halo4<EPI_ACT>(ctx, p, x, wk);
        case EPI_DGRAD: return run_halo4<EPI_DGRAD>(ctx, p, x, wk);
    }
    return CF_ERR_INVALID_ARG;
}

}  // namespace cf
