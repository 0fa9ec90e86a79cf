// conv_halo.cu -- forward / backward-data 3x3x3 convolution for narrow GEMM
// N (c_out <= 128): implicit GEMM whose A operand is read from ONE halo tile
// per input-channel chunk instead of one shifted box per tap.
//
// Output tile: 2 planes x 16 lines x 8 voxels (256 voxels) of sample n,
// computed as two M=128 accumulators (plane 0, plane 1); accumulator row
// r = 8*j + l is line j, voxel l.  For each chunk of KC (16 or 32) input channels the
// producer loads the halo box (KC, 10, 18, 4) -- voxels w0-1..w0+8, lines
// h0-1..h0+16, planes d0-1..d0+2, zero outside the volume -- into shared
// memory with TMA (row R = (dd*18 + hh)*10 + ww, KC*2 bytes per row, swizzled).
// The A operand of tap (kd,kh,kw) for plane i is then the sub-matrix starting
// at row ((i+kd)*18 + kh)*10 + kw: eight consecutive rows (one 8-voxel line
// segment) form a core-matrix group, and groups (lines) are 10 rows apart, so
// the shared-memory descriptor only changes its start address (the hardware
// swizzle is a function of the absolute address, so any row offset reads
// back what TMA wrote).  Each halo row is reused by up to 27 taps, cutting
// the L2->SM traffic of A by ~10x against per-tap loads; the filter slab of
// each tap streams through a separate ring.
//
// Plane pairs (GEMM N <= 64): halo plane p feeds output plane 0 through tap
// row kd = p and output plane 1 through kd = p - 1 with the SAME A operand, so
// for p = 1, 2 one MMA of width 2*N takes B = the two filter slabs stacked
// (kd = p above kd = p - 1: the resident filter keeps, per (kh, kw), the slabs
// in the order kd = 2, 1, 0) and writes both planes' accumulators, which lie
// N columns apart.  Per (kh, kw) and k step that is 4 MMAs (two of width 2N,
// two of width N for p = 0, 3) instead of 6, and A is read from shared memory
// 4 times instead of 6.  Issuer warp 1 takes halo planes 0, 1 and warp 6
// planes 2, 3, each into its own pair of plane accumulators; the epilogue
// adds the two.
//
// GEMM N = 32 with a filter that fits in shared memory whole runs the 4-plane
// tile of conv_halo4.cu instead (two issuers on three halo planes each).
//
// Epilogues: plain bf16 store, backward-data leaky-ReLU derivative, or the
// CosmoFlow bias + leaky ReLU + 2x2x2 max-pool: the two planes of a window
// are in the same TMEM lane (two accumulators), the w and h neighbours are
// lanes +1 and +8 of the same warp, so the window max and its first-maximum
// code (dd*4+dh*2+dw) are reduced with warp shuffles.
#include "halo_common.cuh"

namespace cf {

template <int BN, int KC, int EPI, bool RES>
struct HaloCfg {
    static constexpr bool STK = BN <= 64;  // plane pairs stacked into one MMA (see above)
    static constexpr uint32_t ROW = KC * 2;
    static constexpr uint32_t HALO_BYTES = H_ROWS * ROW;  // 23040, 46080 or 92160
    static constexpr uint32_t HALO_STRIDE = (HALO_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t W_BYTES = BN * KC * 2;      // one tap's filter slab
    static constexpr int TPS = 3;                         // taps per streamed filter stage
    static constexpr int HS = 2;
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t BUDGET = 227 * 1024 - 1024 - BAR_BYTES - HS * HALO_STRIDE;
    static constexpr int WS_RAW = (int)(BUDGET / (TPS * W_BYTES));
    static constexpr int WS = WS_RAW > 12 ? 12 : WS_RAW;
    static constexpr uint32_t SWZ = KC == 64 ? SWZ_128B : (KC == 32 ? SWZ_64B : SWZ_32B);
    static constexpr uint32_t SBO_A = HH_W * ROW;  // one halo line
    static constexpr uint32_t SBO_B = 8 * ROW;
    // per tile buffer: plane 0 | plane 1 (BN columns each), one pair per issuer when stacked
    static constexpr uint32_t ACC_STRIDE = STK ? 4 * BN : 2 * BN;
    static constexpr uint32_t TMEM_COLS = 2 * ACC_STRIDE <= 128 ? 128 : (2 * ACC_STRIDE <= 256 ? 256 : 512);
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    static constexpr uint32_t IDESC2 = idesc_bf16(128, STK ? 2 * BN : BN, 0, 0);
    static_assert(RES || WS >= 3, "shared memory");
    static_assert(2 * ACC_STRIDE <= 512, "tensor memory");
    // shared memory: halo ring, then either the resident filter (n_chunks * 27
    // slabs, sized at launch) or the streamed filter ring
    static uint32_t smem_bytes(int n_chunks) {
        const uint32_t w = RES ? (uint32_t)n_chunks * 27 * W_BYTES : (uint32_t)WS * TPS * W_BYTES;
        return 1024 + HS * HALO_STRIDE + w + BAR_BYTES;
    }
};

template <int BN, int KC, int EPI, bool RES>
__global__ void __launch_bounds__(224, 1)
    conv_halo_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const HaloParams p) {
    using C = HaloCfg<BN, KC, EPI, RES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* hring = smem;
    uint8_t* wsm = smem + C::HS * C::HALO_STRIDE;
    const uint32_t w_region = RES ? (uint32_t)p.n_chunks * 27 * C::W_BYTES : (uint32_t)C::WS * C::TPS * C::W_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + w_region);
    uint64_t* hfull = bars;
    uint64_t* hempty = hfull + C::HS;
    uint64_t* wfull = hempty + C::HS;
    uint64_t* wempty = wfull + C::WS;
    uint64_t* tfull = wempty + C::WS;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;  // [2]
    uint64_t* wres = drain + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(wres + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        // stages are released and accumulators completed by both MMA issuers
        for (int s = 0; s < C::HS; ++s) {
            mbar_init(&hfull[s], 1);
            mbar_init(&hempty[s], 2);
        }
        for (int s = 0; s < C::WS; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 2);
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
        tmem_alloc(tmem_holder, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: per chunk one halo box; the filter either
            // once (resident) or TPS taps per ring stage
            int hs = 0, ws = 0;
            uint32_t hph = 0, wph = 0, hiss = 0, hpar = 0, wiss = 0, wpar = 0;
            bool ok = true, res_issued = false;
            if (RES && blockIdx.x < p.num_tiles) {
                mbar_arrive_expect_tx(wres, (uint32_t)p.n_chunks * 27 * C::W_BYTES);
                for (int ch = 0; ch < p.n_chunks; ++ch)
                    for (int tap = 0; tap < 27; ++tap) {
                        // stacked: slot (kh, kw, 2 - kd); else slot = tap
                        const int kd = tap / 9, r = tap - 9 * kd;
                        const int slot = C::STK ? r * 3 + (2 - kd) : tap;
                        tma_load_2d(wsm + (ch * 27 + slot) * C::W_BYTES, &tmW, wres, tap * p.Cin + ch * KC, 0);
                    }
                res_issued = true;
            }
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                const HTile t = halo_decode(p, tile, BN);
                for (int ch = 0; ch < p.n_chunks && ok; ++ch) {
                    if (!mbar_wait(&hempty[hs], hph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&hfull[hs], C::HALO_BYTES);
                    tma_load_5d(hring + hs * C::HALO_STRIDE, &tmX, &hfull[hs], ch * KC, t.w0 - 1, t.h0 - 1, t.d0 - 1,
                                t.n);
                    hiss |= 1u << hs;
                    hpar = (hpar & ~(1u << hs)) | (hph << hs);
                    if (++hs == C::HS) {
                        hs = 0;
                        hph ^= 1;
                    }
                    if (RES) continue;
                    for (int g = 0; g < 27 / C::TPS; ++g) {
                        if (!mbar_wait(&wempty[ws], wph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&wfull[ws], C::TPS * C::W_BYTES);
                        // a stage: stacked, the kd = 2, 1, 0 slabs of (kh, kw) = g; else the
                        // kw = 0, 1, 2 slabs of (kd, kh) = g
                        for (int u = 0; u < C::TPS; ++u)
                            tma_load_2d(wsm + (ws * C::TPS + u) * C::W_BYTES, &tmW, &wfull[ws],
                                        (C::STK ? (2 - u) * 9 + g : g * C::TPS + u) * p.Cin + ch * KC, t.co0);
                        wiss |= 1u << ws;
                        wpar = (wpar & ~(1u << ws)) | (wph << ws);
                        if (++ws == C::WS) {
                            ws = 0;
                            wph ^= 1;
                        }
                    }
                }
            }
            if (!ok || res_issued) {  // copies in flight must land before the CTA exits
                if (res_issued) mbar_wait_timed(wres, 0, p.wait_ns);
                if (!ok) {
                    for (int s = 0; s < C::HS; ++s)
                        if (hiss & (1u << s)) mbar_wait_timed(&hfull[s], (hpar >> s) & 1, p.wait_ns);
                    for (int s = 0; s < C::WS; ++s)
                        if (wiss & (1u << s)) mbar_wait_timed(&wfull[s], (wpar >> s) & 1, p.wait_ns);
                }
            }
        }
    } else if (warp == 1 || warp == 6) {
        if (lane == 0) {
            // ---------------- MMA issuers: warp 1 for plane 0, warp 6 for plane 1 (one
            // thread's issue rate bounds narrow-N MMAs; the planes' accumulators are disjoint)
            const int i = warp == 1 ? 0 : 1;
            int hs = 0, ws = 0;
            uint32_t hph = 0, wph = 0, local = 0;
            bool ok = true;
            const uint64_t adesc0 = sdesc(smem_u32(hring), 16, C::SBO_A, C::SWZ);
            const uint64_t bdesc0 = sdesc(smem_u32(wsm), 16, C::SBO_B, C::SWZ);
            if (RES && blockIdx.x < p.num_tiles)
                ok = mbar_wait(wres, 0, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL);
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t acc = local & 1, use = local >> 1;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * C::ACC_STRIDE;
                for (int ch = 0; ch < p.n_chunks && ok; ++ch) {
                    if (!mbar_wait(&hfull[hs], hph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    const uint64_t ah = adesc0 + ((hs * C::HALO_STRIDE) >> 4);
                    // taps in groups of TPS = 3 (one kw line: kd, kh fixed); inside a group every
                    // descriptor offset is a compile-time constant
#pragma unroll 1
                    for (int g = 0; g < 27 / C::TPS; ++g) {
                        uint64_t bg;
                        if (RES) {
                            bg = bdesc0 + (((ch * 27 + g * C::TPS) * C::W_BYTES) >> 4);
                        } else {
                            if (!mbar_wait(&wfull[ws], wph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                                ok = false;
                                break;
                            }
                            bg = bdesc0 + ((ws * C::TPS * C::W_BYTES) >> 4);
                        }
                        tc_fence_after();
                        constexpr uint32_t plane_rows = HH_H * HH_W;
                        const uint32_t first = (ch | g) != 0;
                        if (C::STK) {
                            // (kh, kw) = g; slabs kd = 2, 1, 0 at bg, +1, +2 slab.  Issuer i
                            // owns halo planes 2i, 2i+1 and accumulator pair i; the wide MMA
                            // goes first (it starts both planes' sums on the first group)
                            const int kh = g / 3, kw = g % 3;
                            const int pw = 1 + i, pn = 3 * i;  // wide / narrow halo plane
                            const uint32_t dp = d0 + i * 2 * BN;
                            const uint64_t aw = ah + (((uint32_t)((pw * HH_H + kh) * HH_W + kw) * C::ROW) >> 4);
                            const uint64_t an = ah + (((uint32_t)((pn * HH_H + kh) * HH_W + kw) * C::ROW) >> 4);
                            const uint64_t bw = bg + (((uint32_t)(1 - i) * C::W_BYTES) >> 4);  // kd = 1 / 2, then kd - 1
                            const uint64_t bn = bg + (((uint32_t)(i == 0 ? 2 : 0) * C::W_BYTES) >> 4);  // kd = 0 / 2
#pragma unroll
                            for (int k = 0; k < KC / 16; ++k)
                                umma_bf16(dp, aw + ((k * 32) >> 4), bw + ((k * 32) >> 4), C::IDESC2, (first | k) != 0);
#pragma unroll
                            for (int k = 0; k < KC / 16; ++k)
                                umma_bf16(dp + i * BN, an + ((k * 32) >> 4), bn + ((k * 32) >> 4), C::IDESC, 1u);
                        } else {
                        const int kd = g / 3, kh = g % 3;
                        const uint64_t ag = ah + (((uint32_t)((kd * HH_H + kh) * HH_W) * C::ROW) >> 4);
#pragma unroll
                        for (int kw = 0; kw < 3; ++kw) {
                            const uint64_t bw = bg + ((kw * C::W_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < KC / 16; ++k) {
                                const uint64_t ad = ag + (((i * plane_rows + kw) * C::ROW + k * 32) >> 4);
                                umma_bf16(d0 + i * BN, ad, bw + ((k * 32) >> 4), C::IDESC, (first | kw | k) != 0);
                            }
                        }
                        }
                        if (!RES) {
                            umma_commit(&wempty[ws]);
                            if (++ws == C::WS) {
                                ws = 0;
                                wph ^= 1;
                            }
                        }
                    }
                    if (!ok) break;
                    umma_commit(&hempty[hs]);
                    if (++hs == C::HS) {
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
        // ---------------- epilogue warps 2..5
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        // unpooled outputs with BN <= 32, on request: channel sums of the stored
        // outputs (in backward data, the bias gradient of the previous block), per
        // thread over its tiles, then over the CTA
        constexpr bool DSUM = (EPI == EPI_PLAIN || EPI == EPI_DGRAD) && BN <= 32;
        const bool dsum_on = DSUM && p.ea.colsum_part != nullptr;
        float dsum[DSUM ? BN : 1];
#pragma unroll
        for (int c = 0; c < (DSUM ? BN : 1); ++c) dsum[c] = 0.f;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1, use = local >> 1;
            if (!epi_wait(&tfull[acc], use & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            const HTile t = halo_decode(p, tile, BN);
            halo_epilogue<BN, EPI>(p, t, tmem_base, acc * C::ACC_STRIDE, q, lane, 0, 0, dsum_on ? dsum : nullptr,
                                   C::STK ? acc * C::ACC_STRIDE + 2 * BN : 0xFFFFFFFFu,
                                   C::STK ? acc * C::ACC_STRIDE + 3 * BN : 0xFFFFFFFFu);
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if (dsum_on) {
            // the last tile's MMAs are complete, so the halo ring is idle: reduce
            // the 128 threads' sums through it (thread order, then one row per CTA)
            float* red = reinterpret_cast<float*>(hring);
            named_bar_sync(2, 128);
#pragma unroll
            for (int c = 0; c < (DSUM ? BN : 1); ++c) red[et * (BN + 1) + c] = dsum[c];
            named_bar_sync(2, 128);
            if (et < BN && et < p.Cout) {
                float s = 0.f;
                for (int r = 0; r < 128; ++r) s += red[r * (BN + 1) + et];
                p.ea.colsum_part[(int64_t)blockIdx.x * p.Cout + et] = s;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

template <int BN, int KC, int EPI, bool RES>
static cf_status run_halo(const LaunchCtx& ctx, HaloParams p, const uint16_t* x, const uint16_t* wk) {
    using C = HaloCfg<BN, KC, EPI, RES>;
    CUtensorMap tx, tw;
    const uint64_t dx[5] = {(uint64_t)p.Cin, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.D, (uint64_t)p.N};
    const uint64_t sx[4] = {(uint64_t)p.Cin * 2, (uint64_t)p.W * p.Cin * 2, (uint64_t)p.H * p.W * p.Cin * 2,
                            (uint64_t)p.D * p.H * p.W * p.Cin * 2};
    const uint32_t bx[5] = {(uint32_t)KC, (uint32_t)HH_W, (uint32_t)HH_H, (uint32_t)HH_D, 1u};
    const CUtensorMapSwizzle swz = KC == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : KC == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!encode_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dx, sx, bx, swz)) return CF_ERR_CUDA;
    const uint64_t dw[2] = {(uint64_t)27 * p.Cin, (uint64_t)p.Cout};
    const uint64_t sw[1] = {(uint64_t)27 * p.Cin * 2};
    const uint32_t bw[2] = {(uint32_t)KC, (uint32_t)BN};
    if (!encode_tmap(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wk, dw, sw, bw, swz)) return CF_ERR_CUDA;
    p.n_chunks = p.Cin / KC;
    const uint32_t smem = C::smem_bytes(p.n_chunks);
    if (smem > 227 * 1024) return CF_ERR_UNSUPPORTED;
    auto kern = conv_halo_kernel<BN, KC, EPI, RES>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = grid_for(kern, smem, 224, ctx.num_sms, p.num_tiles, C::TMEM_COLS);
    kern<<<grid, 224, smem, ctx.stream>>>(tx, tw, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int BN, int KC, bool RES>
static cf_status halo_epi(const LaunchCtx& ctx, const HaloParams& p, const uint16_t* x, const uint16_t* wk, int epi) {
    switch (epi) {
        case EPI_PLAIN: return run_halo<BN, KC, EPI_PLAIN, RES>(ctx, p, x, wk);
        case EPI_POOL: return run_halo<BN, KC, EPI_POOL, RES>(ctx, p, x, wk);
        case EPI_AVG: return run_halo<BN, KC, EPI_AVG, RES>(ctx, p, x, wk);
        case EPI_ACT: return run_halo<BN, KC, EPI_ACT, RES>(ctx, p, x, wk);
        case EPI_DGRAD: return run_halo<BN, KC, EPI_DGRAD, RES>(ctx, p, x, wk);
    }
    return CF_ERR_INVALID_ARG;
}

// The halo tile pays off wherever the per-tap A re-fetch of the per-tap
// kernel would load L2 (it reads each input row once per tap); c_out up to
// 128 fits two double-buffered accumulator pairs in tensor memory.  Input
// channels go in chunks of 32 (64-byte rows), or of 16 (32-byte rows) when
// c_in is an odd multiple of 16.
bool halo_path_supported(int c_in, int c_out) {
    return (c_in % 16 == 0) && (c_out == 32 || c_out == 64 || c_out == 128);
}

cf_status launch_conv_halo(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                           const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y, uint8_t* idx,
                           const float* bias, const uint16_t* x_act, float slope, float* colsum_part, int pool_kind,
                           int act, uint16_t* route_dz, const uint8_t* route_idx) {
    if (!halo_path_supported(c_in, c_out)) return CF_ERR_UNSUPPORTED;
    if (epi == EPI_POOL && pool_kind == 1) epi = EPI_AVG;
    if (epi == EPI_PLAIN && act) epi = EPI_ACT;
    if (colsum_part && (!(epi == EPI_PLAIN || epi == EPI_DGRAD) || c_out > 32)) return CF_ERR_UNSUPPORTED;
    HaloParams p;
    p.N = (int)n;
    p.D = (int)d;
    p.H = (int)h;
    p.W = (int)w;
    p.Cin = c_in;
    p.Cout = c_out;
    p.tiles_w = (int)((w + HT_W - 1) / HT_W);
    p.tiles_h = (int)((h + HT_H - 1) / HT_H);
    p.tiles_d = (int)((d + HT_D - 1) / HT_D);
    p.n_ntiles = 1;
    p.num_tiles = (int)(n * p.tiles_d * p.tiles_h * p.tiles_w);
    set_tile_dividers(p);
    p.n_chunks = 0;
    p.ea = EpiArgs{y, idx, bias, x_act, slope, colsum_part};
    p.ea.route_dz = route_dz;
    p.ea.route_idx = route_idx;
    p.status = ctx.status;
    p.wait_ns = ctx.wait_ns;
    // c_out 32 with a filter that fits whole: the 4-plane tile (measured on the
    // layer-2 backward data, 64 -> 32 channels at 8 x 64^3: 0.220 -> 0.212 ms)
    if (halo4_path_supported(c_in, c_out)) return launch_conv_halo4(ctx, p, x, wk, epi);
    // The whole filter stays in shared memory when it fits beside two halo
    // stages; otherwise it streams 3 taps per stage.
    const int kc = c_in % 32 == 0 ? 32 : 16;
    const bool resident = (size_t)27 * c_in * c_out * 2 + 2 * (size_t)H_ROWS * kc * 2 + 4096 <= (size_t)227 * 1024;
    if (kc == 16) {
        switch (c_out) {
            case 32: return resident ? halo_epi<32, 16, true>(ctx, p, x, wk, epi) : halo_epi<32, 16, false>(ctx, p, x, wk, epi);
            case 64: return resident ? halo_epi<64, 16, true>(ctx, p, x, wk, epi) : halo_epi<64, 16, false>(ctx, p, x, wk, epi);
            case 128: return halo_epi<128, 16, false>(ctx, p, x, wk, epi);
        }
        return CF_ERR_UNSUPPORTED;
    }
    switch (c_out) {
        case 32: return resident ? halo_epi<32, 32, true>(ctx, p, x, wk, epi) : halo_epi<32, 32, false>(ctx, p, x, wk, epi);
        case 64: return resident ? halo_epi<64, 32, true>(ctx, p, x, wk, epi) : halo_epi<64, 32, false>(ctx, p, x, wk, epi);
        case 128: return halo_epi<128, 32, false>(ctx, p, x, wk, epi);
    }
    return CF_ERR_UNSUPPORTED;
}

}  // namespace cf
