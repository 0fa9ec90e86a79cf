// conv_smallc.cu -- forward conv of the small-channel first layer (c_in = 1
// or 4; CosmoFlow input: four redshift channels) as an implicit GEMM whose A
// operand lives in tensor memory.
//
// GEMM view: D[m, co] = sum_k A[m, k] * W[co, k] with k = 4*t + ci
// (t = 9*kd + 3*kh + kw), K = 27*c_in padded to 112 (c_in 4) or 32 (c_in 1).
// Output tile: 2 planes x 16 lines x 8 voxels, two M=128 accumulators (one
// per plane), as in conv_halo.cu, but with the interleaved row order of
// tile_line() so that the gathers are free of shared-memory bank conflicts.
//
// With only 8 (or 2) bytes per voxel, an im2col tile in shared memory would
// be written and read once per tap and bound the kernel by shared-memory
// bandwidth.  Instead:
//   warp 0      : TMA of the tile's input halo (one box of the input viewed as
//                 (W*C, H, D, N): 4 planes x 18 lines x (8 + 2*margin) voxels,
//                 zero outside the volume) into a ring;
//   warps 2..9  : builders (plane 0: warps 2..5, plane 1: warps 6..9): each
//                 thread gathers the im2col row of its (line, voxel) from the
//                 halo (centre voxels from shared memory, w-1 / w+1 neighbours
//                 by warp shuffles) and writes it into a tensor-memory A
//                 buffer with tcgen05.st;
//   warp 1      : tcgen05.mma with A from tensor memory and the filter
//                 (resident in shared memory, K-major SW128) as B;
//   warps 10..17: the epilogues of halo_common.cuh (fused bias + leaky ReLU +
//                 2x2x2 max-pool with argmax by warp shuffles, or plain bf16),
//                 two warps per TMEM lane quarter splitting the channels.
// Every per-tile chain (gather, pooling) is latency-bound, so each role has
// two warps per SM sub-partition.
#include "halo_common.cuh"
#include "smallc_common.cuh"

namespace cf {

template <int CIN, int BN, int EPI>
struct SmallTmCfg {
    static constexpr int KREAL = 27 * CIN;
    static constexpr int KP = (KREAL + 15) / 16 * 16;  // 112 or 32
    static constexpr int KSTEPS = KP / 16;
    static constexpr int PCOLS = CIN == 4 ? 64 : 16;   // TMEM columns per plane's A rows (56 / 16 used)
    static constexpr int ASTRIDE = 2 * PCOLS;          // TMEM columns per A stage (two planes)
    static constexpr int ATOMS = (KP + 63) / 64;
    static constexpr uint32_t B_BYTES = BN * 128 * ATOMS;
    static constexpr int HALO_BYTES = 4 * 18 * (8 + 2 * (16 / (2 * CIN))) * CIN * 2;  // 6912 or 3456
    static constexpr uint32_t HALO_STRIDE = (HALO_BYTES + 1023) / 1024 * 1024;
    static constexpr int HS = 12;  // halo stages in flight (TMA latency)
    static constexpr int NACC = (4 * BN + 2 * ASTRIDE <= 512) ? 2 : 1;
    static constexpr int AST_RAW = (512 - 2 * NACC * BN) / ASTRIDE;
    static constexpr int AST = AST_RAW > 4 ? 4 : AST_RAW;
    static constexpr uint32_t BAR_BYTES = 8 * (2 * HS + 2 * 4 + 5) + 16;
    static constexpr uint32_t SMEM = 1024 + B_BYTES + HS * HALO_STRIDE + BAR_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t ACOL0 = 2 * NACC * BN;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    static_assert(AST >= 2, "tensor memory budget");
};

struct SmallTmParams {
    HaloParams hp;
    const uint16_t* w;  // [Cout][27*CIN]
};

// Gathers the im2col row of (plane i, line j, voxel l) from the halo tile:
// for c_in = 4 the 9 (kd, kh) halo lines at voxel l-1, l, l+1 (8 bytes each),
// K index k = 4*t + ci, t = 9*kd + 3*kh + kw (54 words + 2 zero words).  The
// 27 shared-memory loads are independent (no shuffles, no divergent edge
// cases), so a warp keeps them all in flight.
__device__ __forceinline__ void gather_plane_c4(const uint8_t* halo, int i, int j, int l, uint32_t (&wd)[56]) {
    constexpr int PITCH = 12 * 8;  // (8 + 2*2) voxels x 8 bytes
    const uint8_t* base = halo + (i * 18 + j) * PITCH + (l + 1) * 8;
#pragma unroll
    for (int kd = 0; kd < 3; ++kd)
#pragma unroll
        for (int kh = 0; kh < 3; ++kh)
#pragma unroll
            for (int kw = 0; kw < 3; ++kw) {
                const uint2 v = *reinterpret_cast<const uint2*>(base + (kd * 18 + kh) * PITCH + kw * 8);
                const int t = kd * 9 + kh * 3 + kw;
                wd[2 * t] = v.x;
                wd[2 * t + 1] = v.y;
            }
    wd[54] = wd[55] = 0u;
}

// c_in = 1: 27 taps padded to 32 (16 words).
__device__ __forceinline__ void gather_plane_c1(const uint8_t* halo, int i, int j, int l, uint32_t (&wd)[56]) {
    constexpr int PITCH = 24 * 2;  // (8 + 2*8) voxels x 2 bytes
    uint32_t v[32];
#pragma unroll
    for (int t = 27; t < 32; ++t) v[t] = 0u;
#pragma unroll
    for (int kd = 0; kd < 3; ++kd)
#pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
            const uint16_t* line = reinterpret_cast<const uint16_t*>(halo + ((i + kd) * 18 + j + kh) * PITCH);
#pragma unroll
            for (int kw = 0; kw < 3; ++kw) v[kd * 9 + kh * 3 + kw] = line[l + 8 + kw - 1];
        }
#pragma unroll
    for (int q = 0; q < 16; ++q) wd[q] = v[2 * q] | (v[2 * q + 1] << 16);
}

template <int CIN, int BN, int EPI>
__global__ void __launch_bounds__(576, 1)
    conv_smallc_kernel(const __grid_constant__ CUtensorMap tmH, const SmallTmParams sp) {
    using C = SmallTmCfg<CIN, BN, EPI>;
    const HaloParams& p = sp.hp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* bsm = smem;
    uint8_t* hring = smem + C::B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(hring + C::HS * C::HALO_STRIDE);
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::HS; ++s) {
            mbar_init(&hfull[s], 1);
            mbar_init(&hempty[s], 256);
        }
        for (int s = 0; s < C::AST; ++s) {
            mbar_init(&afull[s], 256);
            mbar_init(&aempty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 256);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmH);
    }
    // resident filter of the CTA's N tile: rows co0 .. co0+BN-1 (zero at and
    // above Cout), K padded with zeros, SW128 K-major atoms of 64 K-elements.
    // Tiles are dealt with stride gridDim.x and the launch makes gridDim.x a
    // multiple of n_ntiles, so every tile of this CTA has the same N tile.
    {
        const int co0 = (blockIdx.x % p.n_ntiles) * BN;
        for (int e = threadIdx.x; e < BN * (C::ATOMS * 8); e += blockDim.x) {
            const int r = e / (C::ATOMS * 8), c = e % (C::ATOMS * 8);
            uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
                const int k = c * 8 + k8;
                uint32_t bits = 0;
                if (co0 + r < p.Cout && k < C::KREAL) bits = sp.w[(int64_t)(co0 + r) * C::KREAL + k];
                v[k8 >> 1] |= bits << (16 * (k8 & 1));
            }
            const int atom = c >> 3, cin_atom = c & 7;
            *reinterpret_cast<uint4*>(bsm + atom * (BN * 128) + r * 128 + ((cin_atom ^ (r & 7)) << 4)) =
                make_uint4(v[0], v[1], v[2], v[3]);
        }
        fence_proxy_async_smem();
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
            // ---------------- halo producer
            int hs = 0;
            uint32_t hph = 0, issued = 0, par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const HTile t = halo_decode(p, tile, BN);
                if (!mbar_wait(&hempty[hs], hph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&hfull[hs], (uint32_t)C::HALO_BYTES);
                load_halo<CIN>(hring + hs * C::HALO_STRIDE, &tmH, &hfull[hs], t.n, t.d0, t.h0, t.w0);
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
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
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
                const uint32_t d_tmem = tmem_base + acc * 2 * BN;
                const uint32_t a_tmem = tmem_base + C::ACOL0 + as * C::ASTRIDE;
#pragma unroll
                for (int k = 0; k < C::KSTEPS; ++k) {
                    const uint32_t atom = k >> 2, koff = (k & 3) * 32;
                    const uint64_t bd = sdesc(b_addr + atom * (BN * 128) + koff, 16, 1024, SWZ_128B);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        umma_bf16_tmem_a(d_tmem + i * BN, a_tmem + i * C::PCOLS + 8 * k, bd, C::IDESC, k != 0);
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
    } else if (warp < 10) {
        // ---------------- builders: warps 2..5 plane 0, 6..9 plane 1; one row each
        const int q = warp & 3;
        const int plane = (warp - 2) >> 2;
        const int j = tile_line<true>(q, lane), l = lane & 7;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + C::ACOL0 + plane * C::PCOLS;
        int hs = 0, as = 0;
        uint32_t hph = 0, aph = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            // every lane waits, and the warp leaves together if any lane gave up, so
            // the shuffles and .sync.aligned tensor-memory stores below always see
            // the full warp
            if (!__all_sync(0xffffffffu, mbar_wait(&hfull[hs], hph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL, kNapNs)))
                break;
            uint32_t wd[56];
            if (CIN == 4)
                gather_plane_c4(hring + hs * C::HALO_STRIDE, plane, j, l, wd);
            else
                gather_plane_c1(hring + hs * C::HALO_STRIDE, plane, j, l, wd);
            mbar_arrive(&hempty[hs]);
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&aempty[as], aph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY, kNapNs)))
                break;
            tc_fence_after();
            const uint32_t ta = lane_addr + as * C::ASTRIDE;
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
        // ---------------- epilogue warps 10..17: two per lane quarter, each taking
        // half of every 32-channel group (16 channels when BN is 16: one warp idles)
        const int q = warp & 3;
        const int half = (warp - 10) >> 2;
        const int et = threadIdx.x - 320;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
            const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
            if (!epi_wait(&tfull[acc], use & 1, et, epi_flag, abort_flag, p.wait_ns, p.status, 256)) break;
            tc_fence_after();
            const HTile t = halo_decode(p, tile, BN);
            halo_epilogue<BN, EPI, 16, true>(p, t, tmem_base, acc * 2 * BN, q, lane, 16 * half, 32);
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
static cf_status run_smallc(const LaunchCtx& ctx, const HaloParams& hp, const uint16_t* x, const uint16_t* wk) {
    using C = SmallTmCfg<CIN, BN, EPI>;
    CUtensorMap th;
    if (!make_halo_map(&th, x, hp.N, hp.D, hp.H, hp.W, CIN, HT_W, HT_H, HT_D)) return CF_ERR_CUDA;
    SmallTmParams sp{hp, wk};
    auto kern = conv_smallc_kernel<CIN, BN, EPI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    int grid = grid_for(kern, C::SMEM, 576, ctx.num_sms, hp.num_tiles, C::TMEM_COLS);
    grid = std::max(hp.n_ntiles, grid / hp.n_ntiles * hp.n_ntiles);  // each CTA keeps one N tile
    kern<<<grid, 576, C::SMEM, ctx.stream>>>(th, sp);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int CIN, int BN>
static cf_status smallc_epi(const LaunchCtx& ctx, const HaloParams& hp, const uint16_t* x, const uint16_t* wk,
                            int epi) {
    if (epi == EPI_POOL) return run_smallc<CIN, BN, EPI_POOL>(ctx, hp, x, wk);
    if (epi == EPI_PLAIN) return run_smallc<CIN, BN, EPI_PLAIN>(ctx, hp, x, wk);
    return CF_ERR_UNSUPPORTED;
}

cf_status launch_conv_smallc(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                             const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y, uint8_t* idx,
                             const float* bias, float slope) {
    if (c_out % 8 != 0 || c_out > 256) return CF_ERR_UNSUPPORTED;
    if (c_in != 1 && c_in != 4) return CF_ERR_UNSUPPORTED;
    if ((w * c_in) % 8 != 0) return CF_ERR_UNSUPPORTED;  // halo rows must be 16-byte multiples
    // N tile: c_out rounded up to 16, at most 128 (two N tiles above that)
    const int bn = c_out <= 128 ? (c_out + 15) / 16 * 16 : 128;
    HaloParams hp;
    hp.N = (int)n;
    hp.D = (int)d;
    hp.H = (int)h;
    hp.W = (int)w;
    hp.Cin = c_in;
    hp.Cout = c_out;
    hp.tiles_w = (int)((w + HT_W - 1) / HT_W);
    hp.tiles_h = (int)((h + HT_H - 1) / HT_H);
    hp.tiles_d = (int)((d + HT_D - 1) / HT_D);
    hp.n_ntiles = (c_out + bn - 1) / bn;
    hp.num_tiles = (int)(n * hp.tiles_d * hp.tiles_h * hp.tiles_w * hp.n_ntiles);
    hp.n_chunks = 1;
    hp.ea = EpiArgs{y, idx, bias, nullptr, slope};
    hp.status = ctx.status;
    hp.wait_ns = ctx.wait_ns;
#define CF_SC_CASE(B)                                                        \
    case B:                                                                  \
        return c_in == 4 ? smallc_epi<4, B>(ctx, hp, x, wk, epi)             \
                         : smallc_epi<1, B>(ctx, hp, x, wk, epi);
    switch (bn) {
        CF_SC_CASE(16)
        CF_SC_CASE(32)
        CF_SC_CASE(48)
        CF_SC_CASE(64)
        CF_SC_CASE(80)
        CF_SC_CASE(96)
        CF_SC_CASE(112)
        CF_SC_CASE(128)
        default: return CF_ERR_UNSUPPORTED;
    }
#undef CF_SC_CASE
}

}  // namespace cf
