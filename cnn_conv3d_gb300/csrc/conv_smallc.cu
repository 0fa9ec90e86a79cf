// conv_smallc.cu -- forward conv of the small-channel first layer (c_in = 1
// or 4; CosmoFlow input: four redshift channels) as an implicit GEMM whose A
// operand lives in tensor memory.
//
// GEMM view as in conv_fwd.cu: D[m, co] = sum_k A[m, k] * W[co, k] with
// m = voxel of a 128-voxel tile (box 2 x th x tw) and k = 4*t + ci
// (t = 9*kd + 3*kh + kw), K = 27*c_in padded to 112 (c_in 4) or 32 (c_in 1).
//
// With only 8 (or 2) bytes per voxel, an im2col tile in shared memory would
// be written and read once per tap and bound the kernel by shared-memory
// bandwidth.  Instead:
//   warp 0      : TMA of the tile's input halo (one box of the input viewed as
//                 (W*C, H, D, N); 4.6 KB for a 2 x 2 x 32 tile) into a ring;
//   warps 2..5  : builders: each thread gathers the im2col row of its voxel
//                 from the halo (centre voxels from shared memory, w-1 / w+1
//                 neighbours by warp shuffles) and writes it into a tensor-
//                 memory A buffer with tcgen05.st (lane = voxel);
//   warp 1      : tcgen05.mma with A from tensor memory and the filter
//                 (resident in shared memory, K-major SW128) as B;
//   warps 6..9  : the same epilogues as the generic kernel (fused bias +
//                 leaky ReLU + 2x2x2 max-pool with argmax, or plain bf16).
#include "smallc_common.cuh"

namespace cf {

template <int CIN, int BN, int EPI>
struct SmallTmCfg {
    static constexpr int KREAL = 27 * CIN;
    static constexpr int KP = (KREAL + 15) / 16 * 16;  // 112 or 32
    static constexpr int KCOLS = CIN == 4 ? 56 : 16;   // TMEM columns of one A row (bf16 pairs)
    static constexpr int KSTRIDE = CIN == 4 ? 64 : 16; // TMEM columns between A stages
    static constexpr int KSTEPS = KP / 16;
    static constexpr int ATOMS = (KP + 63) / 64;
    static constexpr uint32_t B_BYTES = BN * 128 * ATOMS;
    static constexpr uint32_t HALO_MAX = 4096 + 1024;  // >= halo_bytes() of every tile shape, 1 KB aligned
    static constexpr int HS = 4;                       // halo ring stages
    static constexpr int AST = 4;                      // TMEM A stages
    static constexpr int NACC = (2 * BN + AST * KSTRIDE <= 512) ? 2 : 1;
    static constexpr uint32_t STG_BYTES = EPI == EPI_POOL ? 128 * 33 * 4 : 0;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t SMEM = 1024 + B_BYTES + HS * HALO_MAX + STG_BYTES + BAR_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t ACOL0 = NACC * BN;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    static_assert(NACC * BN + AST * KSTRIDE <= 512, "tensor memory budget");
};

struct SmallTmParams {
    ConvGeom g;
    const uint16_t* w;  // [Cout][27*CIN]
    EpiArgs ea;
    int* status;
    uint64_t wait_ns;
};

template <int CIN, int BN, int EPI>
__global__ void __launch_bounds__(320, 1)
    conv_smallc_kernel(const __grid_constant__ CUtensorMap tmH, const SmallTmParams p) {
    using C = SmallTmCfg<CIN, BN, EPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* bsm = smem;
    uint8_t* hring = smem + C::B_BYTES;
    float* stg = reinterpret_cast<float*>(hring + C::HS * C::HALO_MAX);
    uint64_t* bars = reinterpret_cast<uint64_t*>(hring + C::HS * C::HALO_MAX + C::STG_BYTES);
    uint64_t* hfull = bars;
    uint64_t* hempty = hfull + C::HS;
    uint64_t* afull = hempty + C::HS;
    uint64_t* aempty = afull + C::AST;
    uint64_t* tfull = aempty + C::AST;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ConvGeom& g = p.g;
    const uint32_t halo_tx = (uint32_t)halo_bytes(g.tw, g.th, g.td, CIN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::HS; ++s) {
            mbar_init(&hfull[s], 1);
            mbar_init(&hempty[s], 128);
        }
        for (int s = 0; s < C::AST; ++s) {
            mbar_init(&afull[s], 128);
            mbar_init(&aempty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmH);
    }
    // resident filter: rows co < BN (zero at and above Cout), K padded with zeros,
    // SW128 K-major atoms of 64 K-elements (atom a at a * BN * 128 bytes)
    for (int e = threadIdx.x; e < BN * (C::ATOMS * 8); e += blockDim.x) {
        const int r = e / (C::ATOMS * 8), c = e % (C::ATOMS * 8);
        uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int k = c * 8 + k8;
            uint32_t bits = 0;
            if (r < g.Cout && k < C::KREAL) bits = p.w[(int64_t)r * C::KREAL + k];
            v[k8 >> 1] |= bits << (16 * (k8 & 1));
        }
        const int atom = c >> 3, cin_atom = c & 7;
        *reinterpret_cast<uint4*>(bsm + atom * (BN * 128) + r * 128 + ((cin_atom ^ (r & 7)) << 4)) =
            make_uint4(v[0], v[1], v[2], v[3]);
    }
    fence_proxy_async_smem();
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
            // ---------------- halo producer
            int hs = 0;
            uint32_t hph = 0, issued = 0, par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x) {
                const TileCoord tc = decode_tile(g, tile, BN);
                if (!mbar_wait(&hempty[hs], hph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&hfull[hs], halo_tx);
                load_halo<CIN>(hring + hs * C::HALO_MAX, &tmH, &hfull[hs], tc.n, tc.d0, tc.h0, tc.w0);
                issued |= 1u << hs;
                par = (par & ~(1u << hs)) | (hph << hs);
                if (++hs == C::HS) {
                    hs = 0;
                    hph ^= 1;
                }
            }
            if (!ok) {
                for (int s = 0; s < C::HS; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&hfull[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int as = 0;
            uint32_t aph = 0, local = 0;
            bool ok = true;
            const uint32_t b_addr = smem_u32(bsm);
            for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
                const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&afull[as], aph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const uint32_t a_tmem = tmem_base + C::ACOL0 + as * C::KSTRIDE;
#pragma unroll
                for (int k = 0; k < C::KSTEPS; ++k) {
                    const uint32_t atom = k >> 2, koff = (k & 3) * 32;
                    const uint64_t bd = sdesc(b_addr + atom * (BN * 128) + koff, 16, 1024, SWZ_128B);
                    umma_bf16_tmem_a(d_tmem, a_tmem + 8 * k, bd, C::IDESC, k != 0);
                }
                umma_commit(&aempty[as]);
                umma_commit(&tfull[acc]);
                if (++as == C::AST) {
                    as = 0;
                    aph ^= 1;
                }
            }
            if (!ok) {
                umma_commit(drain);
                mbar_wait_timed(drain, 0, p.wait_ns);
            }
        }
    } else if (warp < 6) {
        // ---------------- builders: one voxel row per thread, TMEM lanes 32*q ..
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int l = row % g.tw, j = (row / g.tw) % g.th, i = row / (g.tw * g.th);
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + C::ACOL0;
        int hs = 0, as = 0;
        uint32_t hph = 0, aph = 0;
        for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x) {
            // every lane waits, and the warp leaves together if any lane gave up, so
            // the shuffles and .sync.aligned tensor-memory stores below always see
            // the full warp
            if (!__all_sync(0xffffffffu, mbar_wait(&hfull[hs], hph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)))
                break;
            uint32_t wd[56];
            if (CIN == 4)
                gather_row_c4(hring + hs * C::HALO_MAX, g.tw, g.th, i, j, l, wd);
            else
                gather_row_c1(hring + hs * C::HALO_MAX, g.tw, g.th, i, j, l, wd);
            mbar_arrive(&hempty[hs]);
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&aempty[as], aph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)))
                break;
            tc_fence_after();
            const uint32_t ta = lane_addr + as * C::KSTRIDE;
            if (CIN == 4) {
                tmem_st32(ta, wd);
                tmem_st16(ta + 32, wd + 32);
                tmem_st8(ta + 48, wd + 48);
            } else {
                tmem_st16(ta, wd);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&afull[as]);
            if (++hs == C::HS) {
                hs = 0;
                hph ^= 1;
            }
            if (++as == C::AST) {
                as = 0;
                aph ^= 1;
            }
        }
    } else {
        // ---------------- epilogue warps 6..9
        const int q = warp & 3;
        const int et = threadIdx.x - 192;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
            const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
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

bool make_halo_map(CUtensorMap* m, const uint16_t* x, int n, int d, int h, int w, int cin, int tw, int th, int td) {
    const uint64_t dims[4] = {(uint64_t)w * cin, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t str[3] = {(uint64_t)w * cin * 2, (uint64_t)h * w * cin * 2, (uint64_t)d * h * w * cin * 2};
    const uint32_t box[4] = {(uint32_t)(halo_line_voxels(tw, cin) * cin), (uint32_t)(th + 2), (uint32_t)(td + 2), 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int CIN, int BN, int EPI>
static cf_status run_smallc(const LaunchCtx& ctx, const ConvGeom& g, const uint16_t* x, const uint16_t* wk,
                            const EpiArgs& ea) {
    using C = SmallTmCfg<CIN, BN, EPI>;
    if (halo_bytes(g.tw, g.th, g.td, CIN) > (int)C::HALO_MAX) return CF_ERR_UNSUPPORTED;
    CUtensorMap th;
    if (!make_halo_map(&th, x, g.N, g.D, g.H, g.W, CIN, g.tw, g.th, g.td)) return CF_ERR_CUDA;
    SmallTmParams p;
    p.g = g;
    p.w = wk;
    p.ea = ea;
    p.status = ctx.status;
    p.wait_ns = ctx.wait_ns;
    auto kern = conv_smallc_kernel<CIN, BN, EPI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = grid_for(kern, C::SMEM, 320, ctx.num_sms, g.num_tiles, C::TMEM_COLS);
    kern<<<grid, 320, C::SMEM, ctx.stream>>>(th, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int CIN, int BN>
static cf_status smallc_epi(const LaunchCtx& ctx, const ConvGeom& g, const uint16_t* x, const uint16_t* wk, int epi,
                            const EpiArgs& ea) {
    if (epi == EPI_POOL) return run_smallc<CIN, BN, EPI_POOL>(ctx, g, x, wk, ea);
    if (epi == EPI_PLAIN) return run_smallc<CIN, BN, EPI_PLAIN>(ctx, g, x, wk, ea);
    return CF_ERR_UNSUPPORTED;
}

cf_status launch_conv_smallc(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                             const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y, uint8_t* idx,
                             const float* bias, float slope) {
    if (c_out % 8 != 0 || c_out > 256) return CF_ERR_UNSUPPORTED;
    if (c_in != 1 && c_in != 4) return CF_ERR_UNSUPPORTED;
    if ((w * c_in) % 8 != 0) return CF_ERR_UNSUPPORTED;  // halo rows must be 16-byte multiples
    const int bn = (c_out + 15) / 16 * 16;
    EpiArgs ea{y, idx, bias, nullptr, slope};
    ConvGeom g = make_geom(n, d, h, w, c_in, c_out, bn);
    g.n_ntiles = 1;
    g.num_tiles = (int)(n * g.tiles_d * g.tiles_h * g.tiles_w);
#define CF_SC_CASE(B)                                                              \
    case B:                                                                        \
        return c_in == 4 ? smallc_epi<4, B>(ctx, g, x, wk, epi, ea)                \
                         : smallc_epi<1, B>(ctx, g, x, wk, epi, ea);
    switch (bn) {
        CF_SC_CASE(16)
        CF_SC_CASE(32)
        CF_SC_CASE(64)
        CF_SC_CASE(128)
        CF_SC_CASE(256)
        default: return CF_ERR_UNSUPPORTED;
    }
#undef CF_SC_CASE
}

}  // namespace cf
