// conv_fwd.cu -- forward (and backward-data) 3x3x3 convolution as an implicit
// GEMM on the sm_103a tensor cores.
//
// GEMM view (CosmoFlow page, section III-C "forward data"; hybrid-parallelism
// page, Table I: 3^3 filters, stride 1, "same" padding):
//   D[m, co] = sum_{t, ci} A[m, (t, ci)] * B[co, (t, ci)]
//   m = output voxel of a 128-voxel tile (box 2 x th x tw), t = (kd,kh,kw),
//   A[m,(t,ci)] = X[voxel(m) + t - 1, ci] (zero outside: TMA out-of-bounds fill),
//   B[co,(t,ci)] = W[co][t][ci] (the filter is already K-major).
//
// Kernel structure (one persistent CTA per SM, 6 warps):
//   warp 0      : TMA producer.  For each tap and 16/32/64-channel chunk it loads
//                 the shifted activation box (the A tile, 128 rows) and the
//                 matching filter slab (B tile) into a multi-stage ring.
//   warp 1      : TMEM allocator and single-thread tcgen05.mma issuer, M=128,
//                 N=BN, K=16 per instruction, fp32 accumulator in TMEM.  Two
//                 accumulators alternate so the epilogue of tile i overlaps the
//                 MMAs of tile i+1.
//   warps 2..5  : epilogue: tcgen05.ld of the accumulator, then either a bf16
//                 store of Z, a fused bias + leaky ReLU + 2x2x2 max-pool with
//                 argmax (CosmoFlow block), or the backward-data epilogue that
//                 multiplies by the leaky-ReLU derivative of the previous block.
//
// The small-channel first layer (c_in = 1 or 4) has its own kernel in
// conv_smallc.cu.
#include <algorithm>

#include "conv_common.cuh"

namespace cf {

// ---------------------------------------------------------------------------
// generic kernel: c_in a multiple of KC (16, 32 or 64 channels per K chunk;
// the A and B rows are KC * 2 bytes, swizzled 32, 64 or 128 bytes)

template <int BN, int KC, int EPI>
struct IgemmCfg {
    static constexpr int BM = 128;
    static constexpr uint32_t A_BYTES = BM * KC * 2;
    static constexpr uint32_t B_BYTES = BN * KC * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t STG_BYTES = (EPI == EPI_POOL || EPI == EPI_AVG) ? 128 * 33 * 4 : 0;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t BUDGET = 227 * 1024 - 1024 - STG_BYTES - BAR_BYTES;
    static constexpr int STAGES_RAW = (int)(BUDGET / STAGE_BYTES);
    static constexpr int STAGE_CAP = KC == 16 ? 16 : 8;  // K steps in flight: 16-channel stages are small
    static constexpr int STAGES = STAGES_RAW > STAGE_CAP ? STAGE_CAP : STAGES_RAW;
    static constexpr uint32_t SMEM = 1024 + STAGES * STAGE_BYTES + STG_BYTES + BAR_BYTES;
    static constexpr uint32_t ROW_BYTES = KC * 2;
    static constexpr uint32_t SWZ = KC == 64 ? SWZ_128B : (KC == 32 ? SWZ_64B : SWZ_32B);
    static constexpr uint32_t SBO = 8 * ROW_BYTES;
    static constexpr uint32_t TMEM_COLS = (2 * BN) <= 32 ? 32 : (2 * BN) <= 64 ? 64 : (2 * BN) <= 128 ? 128
                                                                                 : (2 * BN) <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    static_assert(STAGES >= 2, "not enough shared memory for a pipeline");
};

struct IgemmParams {
    ConvGeom g;      // output tiling (output sizes)
    int n_cchunks;
    int stride;      // 1, or 2: tap (kd,kh,kw) of output voxel o reads input voxel 2*o + k - 1
    EpiArgs ea;
    int* status;
    uint64_t wait_ns;
};

template <int BN, int KC, int EPI>
__global__ void __launch_bounds__(192, 1)
    conv_igemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const IgemmParams p) {
    using C = IgemmCfg<BN, KC, EPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;
    float* stg = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::STG_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ConvGeom& g = p.g;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int nk = 27 * p.n_cchunks;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, par = 0;  // per-stage: issued at least once / parity of last issue
            bool ok = true;
            for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x) {
                const TileCoord tc = decode_tile(g, tile, BN);
                int t = 0, cc = 0, kd = 0, kh = 0, kw = 0;
                for (int kb = 0; kb < nk; ++kb) {
                    if (kb > 0 && ++cc == p.n_cchunks) {  // advance (tap, chunk) without divisions
                        cc = 0;
                        ++t;
                        if (++kw == 3) {
                            kw = 0;
                            if (++kh == 3) {
                                kh = 0;
                                ++kd;
                            }
                        }
                    }
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = ring + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_5d(sa, &tmA, &full[stage], cc * KC, p.stride * tc.w0 + kw - 1,
                                p.stride * tc.h0 + kh - 1, p.stride * tc.d0 + kd - 1, tc.n);
                    tma_load_2d(sa + C::A_BYTES, &tmB, &full[stage], t * g.Cin + cc * KC, tc.co0);
                    issued |= 1u << stage;
                    par = (par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {  // let every copy already in flight land before the CTA exits
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&full[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t acc = local & 1, use = local >> 1;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < KC / 16; ++k) {
                        const uint64_t ad = sdesc(a_addr + k * 32, 16, C::SBO, C::SWZ);
                        const uint64_t bd = sdesc(b_addr + k * 32, 16, C::SBO, C::SWZ);
                        umma_bf16(d_tmem, ad, bd, C::IDESC, (kb | k) != 0);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
            }
            if (!ok) {  // wait for the MMAs already issued before leaving
                umma_commit(drain);
                mbar_wait_timed(drain, 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- epilogue warps 2..5
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1, use = local >> 1;
            if (!epi_wait(&tfull[acc], use & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            const TileCoord tc = decode_tile(g, tile, BN);
            conv_epilogue<BN, EPI>(g, tc, p.ea, tmem_base, acc * BN, q, lane, et, stg);
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
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

// Tile extents are powers of two (the epilogue decodes rows with shifts).
TileGeom choose_tile(int64_t d, int64_t h, int64_t w) {
    (void)d;
    TileGeom t;
    t.td = 2;
    if (w >= 32) {
        t.tw = 32;
        t.th = 2;
    } else if (w >= 16) {
        t.tw = 16;
        t.th = 4;
    } else {
        t.tw = 8;
        t.th = 8;
    }
    (void)h;
    return t;
}

// in_d, in_h, in_w: the input sizes (the output's times the stride, rounded
// up).  With stride 2 the A box spans 2*tw x 2*th x 2*td input voxels and the
// tensor map's traversal stride 2 loads every second one: the same dense
// tw x th x td x KC tile as stride 1.
template <int BN, int KC, int EPI>
static cf_status run_igemm(const LaunchCtx& ctx, const ConvGeom& g, const uint16_t* x, const uint16_t* wk,
                           const EpiArgs& ea, int64_t in_d, int64_t in_h, int64_t in_w, int stride) {
    using C = IgemmCfg<BN, KC, EPI>;
    CUtensorMap ta, tb;
    const uint64_t da[5] = {(uint64_t)g.Cin, (uint64_t)in_w, (uint64_t)in_h, (uint64_t)in_d, (uint64_t)g.N};
    const uint64_t sa[4] = {(uint64_t)g.Cin * 2, (uint64_t)in_w * g.Cin * 2, (uint64_t)in_h * in_w * g.Cin * 2,
                            (uint64_t)in_d * in_h * in_w * g.Cin * 2};
    const uint32_t su = (uint32_t)stride;
    const uint32_t ba[5] = {(uint32_t)KC, su * g.tw, su * g.th, su * g.td, 1u};
    const uint32_t es[5] = {1u, su, su, su, 1u};
    const CUtensorMapSwizzle swz = KC == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : KC == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!encode_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, da, sa, ba, swz, es)) return CF_ERR_CUDA;
    const uint64_t db[2] = {(uint64_t)27 * g.Cin, (uint64_t)g.Cout};
    const uint64_t sb[1] = {(uint64_t)27 * g.Cin * 2};
    const uint32_t bb[2] = {(uint32_t)KC, (uint32_t)BN};
    if (!encode_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wk, db, sb, bb, swz)) return CF_ERR_CUDA;

    IgemmParams p;
    p.g = g;
    p.n_cchunks = g.Cin / KC;
    p.stride = stride;
    p.ea = ea;
    p.status = ctx.status;
    p.wait_ns = ctx.wait_ns;
    auto kern = conv_igemm_kernel<BN, KC, EPI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = grid_for(kern, C::SMEM, 192, ctx.num_sms, g.num_tiles, C::TMEM_COLS);
    kern<<<grid, 192, C::SMEM, ctx.stream>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int BN, int KC>
static cf_status dispatch_epi(const LaunchCtx& ctx, const ConvGeom& g, const uint16_t* x, const uint16_t* wk,
                              int epi, const EpiArgs& ea, int64_t in_d, int64_t in_h, int64_t in_w, int stride) {
    switch (epi) {
        case EPI_PLAIN: return run_igemm<BN, KC, EPI_PLAIN>(ctx, g, x, wk, ea, in_d, in_h, in_w, stride);
        case EPI_POOL: return run_igemm<BN, KC, EPI_POOL>(ctx, g, x, wk, ea, in_d, in_h, in_w, stride);
        case EPI_AVG: return run_igemm<BN, KC, EPI_AVG>(ctx, g, x, wk, ea, in_d, in_h, in_w, stride);
        case EPI_ACT: return run_igemm<BN, KC, EPI_ACT>(ctx, g, x, wk, ea, in_d, in_h, in_w, stride);
        case EPI_DGRAD: return run_igemm<BN, KC, EPI_DGRAD>(ctx, g, x, wk, ea, in_d, in_h, in_w, stride);
    }
    return CF_ERR_INVALID_ARG;
}

cf_status launch_conv_igemm(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                            const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y, uint8_t* idx,
                            const float* bias, const uint16_t* x_act, float slope, int pool_kind, int act,
                            int stride, uint16_t* route_dz, const uint8_t* route_idx) {
    if (c_in % 16 != 0 || c_out % 16 != 0) return CF_ERR_UNSUPPORTED;
    if (stride != 1 && (stride != 2 || epi == EPI_DGRAD)) return CF_ERR_UNSUPPORTED;
    const int64_t in_d = d, in_h = h, in_w = w;
    d = (d + stride - 1) / stride;  // from here on: the output sizes
    h = (h + stride - 1) / stride;
    w = (w + stride - 1) / stride;
    // N tile: the narrowest compiled width that holds c_out (at most 256; the
    // filter rows past c_out read as zero, out-of-bounds fill, and the
    // epilogues skip those channels)
    int bn = 256;
    for (int b : {16, 32, 64, 96, 128, 192, 256})
        if (c_out <= b) {
            bn = b;
            break;
        }
    // Small grids: narrower N tiles when that clearly shortens the critical
    // path (by 20%: narrower tiles re-fetch A once more per N tile).  Cost of a
    // CTA's share = waves x cycles per K step of one MMA 128 x bn x 16,
    // max(issue ~52, shared-memory operand reads 32 + bn/4, tensor bn/2).
    if (bn >= 128 && bn % 64 == 0 && c_out % 64 == 0) {
        const int64_t tiles_m = make_geom(n, d, h, w, c_in, c_out, bn).num_tiles / ((c_out + bn - 1) / bn);
        auto cost = [&](int b) {
            const int64_t tiles = tiles_m * ((c_out + b - 1) / b);
            const int64_t waves = (tiles + ctx.num_sms - 1) / ctx.num_sms;
            return waves * std::max<int64_t>(52, std::max<int64_t>(32 + b / 4, b / 2));
        };
        int best = bn;
        for (int b = bn / 2; b >= 64; b /= 2)
            if (c_out % b == 0 && 5 * cost(b) < 4 * cost(best)) best = b;
        bn = best;
    }
    const int kc = (c_in % 64 == 0) ? 64 : (c_in % 32 == 0 ? 32 : 16);
    EpiArgs ea{y, idx, bias, x_act, slope};
    if (epi == EPI_POOL && pool_kind == 1) epi = EPI_AVG;
    if (epi == EPI_PLAIN && act) epi = EPI_ACT;
    ea.route_dz = route_dz;
    ea.route_idx = route_idx;
    ConvGeom g = make_geom(n, d, h, w, c_in, c_out, bn);
#define CF_BN_CASE(B)                                                                              \
    case B:                                                                                        \
        return kc == 64   ? dispatch_epi<B, 64>(ctx, g, x, wk, epi, ea, in_d, in_h, in_w, stride)  \
               : kc == 32 ? dispatch_epi<B, 32>(ctx, g, x, wk, epi, ea, in_d, in_h, in_w, stride)  \
                          : dispatch_epi<B, 16>(ctx, g, x, wk, epi, ea, in_d, in_h, in_w, stride);
    switch (bn) {
        CF_BN_CASE(16)
        CF_BN_CASE(32)
        CF_BN_CASE(64)
        CF_BN_CASE(96)
        CF_BN_CASE(128)
        CF_BN_CASE(192)
        CF_BN_CASE(256)
        default: return CF_ERR_UNSUPPORTED;
    }
#undef CF_BN_CASE
}

}  // namespace cf
