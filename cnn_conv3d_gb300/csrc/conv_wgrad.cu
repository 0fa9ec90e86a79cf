// conv_wgrad.cu -- backward-weight 3x3x3 convolution on the sm_103a tensor
// cores, split-K over samples x voxels with a fixed-order fp32 reduction.
//
// (CosmoFlow page, section III-C "backward weights": the weight-gradient work
// is divided over voxels.)
//   dW[co, t, ci] = sum_{n,v} dZ[n,v,co] * X[n, v + t - 1, ci]
// GEMM view: M = (t, ci) rows (128 per CTA tile), N = co (tiles of BN <= 256
// channels), K = voxels.  Both operands are MN-major in shared memory:
//   A[(t,ci), v] = X[v + t - 1, ci]  -- TMA box of the tap-shifted activation
//                  (zero fill outside the volume), channel rows of 16, 32 or 64
//   B[co, v]     = dZ[v, co]         -- TMA box of the output gradient; channels
//                  at and beyond c_out read as zero (out-of-bounds fill), so an
//                  N tile may be wider than what is left of c_out
// Each CTA unit = one M block x one N tile x one contiguous range of 64-voxel
// boxes; its fp32 accumulator (TMEM) is written to a partial buffer
// [split][co][27*c_in], and a second kernel sums the splits in a fixed order
// into dW.
//
// The small-channel variant (c_in = 1 or 4, conv_wgrad_smallc.cu) builds the
// A tile with builder warps (im2col rows = voxels, 27*c_in columns padded to
// 128) because TMA cannot address 2- or 8-byte channel rows.
#include <algorithm>

#include "smallc_common.cuh"
#include "wgrad_common.cuh"

namespace cf {

// ---------------------------------------------------------------------------
// generic: c_in a multiple of 16

template <int BN, int SUBA, int SUBB>
struct WgCfg {
    static constexpr int KV = 64;  // voxels per K block
    static constexpr uint32_t A_BYTES = 128 * KV * 2;
    static constexpr uint32_t B_BYTES = BN * KV * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t BUDGET = 227 * 1024 - 1024 - BAR_BYTES;
    static constexpr int STAGES_RAW = (int)(BUDGET / STAGE_BYTES);
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr uint32_t SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static constexpr uint32_t A_SUB_BYTES = KV * SUBA * 2;  // one MN atom column (sub-block)
    static constexpr uint32_t B_SUB_BYTES = KV * SUBB * 2;
    static constexpr uint32_t SWZ_A = SUBA == 64 ? SWZ_128B : (SUBA == 32 ? SWZ_64B : SWZ_32B);
    static constexpr uint32_t SWZ_B = SUBB == 64 ? SWZ_128B : (SUBB == 32 ? SWZ_64B : SWZ_32B);
    static constexpr uint32_t SBO_A = 8 * SUBA * 2;  // 8 K-rows
    static constexpr uint32_t SBO_B = 8 * SUBB * 2;
    static constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 1, 1);
};

struct WgradParams {
    WgradGeom g;
    float* part;
    int* status;
    uint64_t wait_ns;
};

template <int BN, int SUBA, int SUBB>
__global__ void __launch_bounds__(192, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                 const WgradParams p) {
    using C = WgCfg<BN, SUBA, SUBB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WgradGeom& g = p.g;
    const int KK = 27 * g.Cin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 128);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmG);
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
            int stage = 0;
            uint32_t phase = 0, issued = 0, par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x) {
                const int mb = u % g.n_mblocks, rest = u / g.n_mblocks;
                const int co0 = (rest % g.n_ntiles) * BN, split = rest / g.n_ntiles;
                const int64_t b0 = (int64_t)split * g.boxes_per_split;
                const int64_t b1 = b0 + g.boxes_per_split < g.total_boxes ? b0 + g.boxes_per_split : g.total_boxes;
                // A sub-blocks of this M block that hold real rows, and their taps
                constexpr int NSUB = 128 / SUBA;
                int nsub = 0;
                int sci[NSUB], sdw[NSUB], sdh[NSUB], sdd[NSUB];
#pragma unroll
                for (int s = 0; s < NSUB; ++s) {
                    const int r0 = mb * 128 + s * SUBA;
                    const int t = r0 / g.Cin;
                    sci[s] = r0 - t * g.Cin;
                    sdd[s] = t / 9 - 1;
                    sdh[s] = (t / 3) % 3 - 1;
                    sdw[s] = t % 3 - 1;
                    if (r0 < KK) ++nsub;
                }
                const uint32_t tx = nsub * C::A_SUB_BYTES + C::B_BYTES;
                BoxCursor cur;
                cur.init(g, b0);
                for (int64_t b = b0; b < b1; ++b, cur.next(g)) {
                    const int n = cur.n, d0 = cur.bd * g.vd, h0 = cur.bh * g.vh, w0 = cur.bw * g.vw;
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = ring + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], tx);
#pragma unroll
                    for (int s = 0; s < NSUB; ++s)
                        if (s < nsub)
                            tma_load_5d(sa + s * C::A_SUB_BYTES, &tmX, &full[stage], sci[s], w0 + sdw[s], h0 + sdh[s],
                                        d0 + sdd[s], n);
#pragma unroll
                    for (int s = 0; s < BN / SUBB; ++s)
                        tma_load_5d(sa + C::A_BYTES + s * C::B_SUB_BYTES, &tmG, &full[stage], co0 + s * SUBB, w0, h0,
                                    d0, n);
                    issued |= 1u << stage;
                    par = (par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&full[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x, ++local) {
                const int split = u / g.n_mblocks / g.n_ntiles;
                const int64_t b0 = (int64_t)split * g.boxes_per_split;
                const int64_t b1 = b0 + g.boxes_per_split < g.total_boxes ? b0 + g.boxes_per_split : g.total_boxes;
                if (!mbar_wait(tempty, (local & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                bool first = true;
                for (int64_t b = b0; b < b1; ++b) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < C::KV / 16; ++k) {
                        // 16 K rows further = 2 groups of 8 rows
                        const uint64_t ad = sdesc(a_addr + k * 16 * SUBA * 2, C::A_SUB_BYTES, C::SBO_A, C::SWZ_A);
                        const uint64_t bd = sdesc(b_addr + k * 16 * SUBB * 2, C::B_SUB_BYTES, C::SBO_B, C::SWZ_B);
                        umma_bf16(tmem_base, ad, bd, C::IDESC, first ? 0u : 1u);
                        first = false;
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(tfull);
            }
            if (!ok) {
                umma_commit(drain);
                mbar_wait_timed(drain, 0, p.wait_ns);
            }
        }
    } else {
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        uint32_t local = 0;
        for (int u = blockIdx.x; u < g.num_units; u += gridDim.x, ++local) {
            const int mb = u % g.n_mblocks, rest = u / g.n_mblocks;
            const int co0 = (rest % g.n_ntiles) * BN, split = rest / g.n_ntiles;
            if (!epi_wait(tfull, local & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            wgrad_store_partial<BN>(g, p.part, mb, split, co0, tmem_base, q, lane);
            tc_fence_before();
            mbar_arrive(tempty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// dW[i] = (accumulate ? dW[i] : 0) + sum over the splits of part[s][i], in a
// fixed order: G groups of consecutive splits per column (each group summed
// ascending in four interleaved partial sums), then the groups in order.
// A block covers 256 / G columns; its threads read a split's columns
// contiguously.
template <int G>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw,
                                                            int64_t count, int splits, int accumulate) {
    constexpr int COLS = 256 / G;
    __shared__ float red[G][COLS];
    const int col = threadIdx.x % COLS, grp = threadIdx.x / COLS;
    const int per = (splits + G - 1) / G;
    const int s0 = min(splits, grp * per), s1 = min(splits, s0 + per);
    for (int64_t c0 = (int64_t)blockIdx.x * COLS; c0 < count; c0 += (int64_t)gridDim.x * COLS) {
        const int64_t i = c0 + col;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < count) {
            int k = s0;
            for (; k + 4 <= s1; k += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) a[u] += __ldg(part + (int64_t)(k + u) * count + i);
            }
            for (; k < s1; ++k) a[0] += __ldg(part + (int64_t)k * count + i);
        }
        red[grp][col] = (a[0] + a[1]) + (a[2] + a[3]);
        __syncthreads();
        if (grp == 0 && i < count) {
            float t = accumulate ? dw[i] : 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) t += red[g][col];
            dw[i] = t;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side

// N tile of the weight-gradient GEMM for c_out (a multiple of 16): the smallest
// of the compiled widths that holds it, 256-wide tiles above that (c_in 1 or 4:
// at most 256 channels, one tile).
static int wgrad_tile_n(int c_in, int c_out) {
    const bool small = c_in == 1 || c_in == 4;
    static const int generic[] = {16, 32, 48, 64, 96, 128, 192, 256};
    static const int smallc[] = {16, 32, 64, 128, 192, 256};
    const int* t = small ? smallc : generic;
    const int nt = small ? 6 : 8;
    for (int i = 0; i < nt; ++i)
        if (c_out <= t[i]) return t[i];
    return 256;
}

static WgradGeom wgrad_geom(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    WgradGeom g;
    g.N = (int)n;
    g.D = (int)d;
    g.H = (int)h;
    g.W = (int)w;
    g.Cin = c_in;
    g.Cout = c_out;
    const bool small = c_in == 1 || c_in == 4;
    g.bn = wgrad_tile_n(c_in, c_out);
    g.n_ntiles = (c_out + g.bn - 1) / g.bn;
    if (small) {
        g.vw = 16;  // the small-channel kernel's box: 2 planes x 4 lines x 16 voxels
        g.vh = 4;
        g.vd = 2;
        g.n_mblocks = 1;
    } else {
        g.vw = w >= 64 ? 64 : (w >= 32 ? 32 : (w >= 16 ? 16 : 8));
        g.vh = 64 / g.vw;
        g.vd = 1;
        g.n_mblocks = (27 * c_in + 127) / 128;
    }
    g.nb_w = (int)((w + g.vw - 1) / g.vw);
    g.nb_h = (int)((h + g.vh - 1) / g.vh);
    g.nb_d = (int)((d + g.vd - 1) / g.vd);
    g.total_boxes = n * g.nb_d * g.nb_h * g.nb_w;
    // at most one unit per SM (one round of CTAs: rounding the split count up
    // would leave a second round of a few units that doubles the kernel's
    // time), each unit at least 8 boxes long (measured in the five-block step:
    // two units per SM, i.e. twice the partial sums to write and reduce, made
    // the step 0.035 ms slower)
    const int tiles = g.n_mblocks * g.n_ntiles;
    int64_t target = std::max<int64_t>(1, (int64_t)num_sms / tiles);
    target = std::min<int64_t>(target, std::max<int64_t>(1, g.total_boxes / 8));
    g.boxes_per_split = (g.total_boxes + target - 1) / target;
    g.n_splits = (int)((g.total_boxes + g.boxes_per_split - 1) / g.boxes_per_split);
    g.num_units = tiles * g.n_splits;
    return g;
}

bool wgrad_routed_fused(int c_in) { return c_in == 1 || c_in == 4; }

bool wgrad_shape_supported(int c_in, int c_out) {
    const bool small = c_in == 1 || c_in == 4;
    if (!small && c_in % 16 != 0) return false;
    return c_out % 16 == 0 && (!small || c_out <= 256);
}

size_t wgrad_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    if (wgrad_halo_supported(c_in, c_out))
        return wgrad_halo_workspace_bytes(num_sms, n, d, h, w, c_in, c_out);
    WgradGeom g = wgrad_geom(num_sms, n, d, h, w, c_in, c_out);
    const size_t generic = (size_t)g.n_splits * c_out * 27 * c_in * sizeof(float);
    if (wgrad_quad_supported(d, h, w, c_in, c_out))
        return std::max(generic, wgrad_quad_workspace_bytes(num_sms, n, d, h, w));
    return generic;
}

template <typename K>
static int wg_grid(K kernel, uint32_t smem, int threads, int num_sms, int units, uint32_t tmem_cols) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    per_sm = std::min<int>(per_sm, (int)(512 / tmem_cols));
    return std::max(1, std::min(units, num_sms * per_sm));
}

static bool make_act_map(CUtensorMap* m, const uint16_t* base, const WgradGeom& g, int c, int box_c) {
    const uint64_t dims[5] = {(uint64_t)c, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.D, (uint64_t)g.N};
    const uint64_t str[4] = {(uint64_t)c * 2, (uint64_t)g.W * c * 2, (uint64_t)g.H * g.W * c * 2,
                             (uint64_t)g.D * g.H * g.W * c * 2};
    const uint32_t box[5] = {(uint32_t)box_c, (uint32_t)g.vw, (uint32_t)g.vh, (uint32_t)g.vd, 1u};
    const CUtensorMapSwizzle swz = box_c == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : box_c == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, str, box, swz);
}

template <int BN, int SUBA, int SUBB>
static cf_status run_wgrad(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                           float* part) {
    using C = WgCfg<BN, SUBA, SUBB>;
    CUtensorMap tx, tg;
    if (!make_act_map(&tx, x, g, g.Cin, SUBA)) return CF_ERR_CUDA;
    if (!make_act_map(&tg, dz, g, g.Cout, SUBB)) return CF_ERR_CUDA;
    WgradParams p{g, part, ctx.status, ctx.wait_ns};
    auto kern = wgrad_kernel<BN, SUBA, SUBB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = wg_grid(kern, C::SMEM, 192, ctx.num_sms, g.num_units, C::TMEM_COLS);
    kern<<<grid, 192, C::SMEM, ctx.stream>>>(tx, tg, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int BN>
static cf_status wgrad_bn(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                          float* part) {
    // dZ sub-blocks: the widest of 64 / 32 / 16 channels that divides the tile
    constexpr int SUBB = BN % 64 == 0 ? 64 : (BN % 32 == 0 ? 32 : 16);
    if (g.Cin % 64 == 0) return run_wgrad<BN, 64, SUBB>(ctx, g, x, dz, part);
    if (g.Cin % 32 == 0) return run_wgrad<BN, 32, SUBB>(ctx, g, x, dz, part);
    return run_wgrad<BN, 16, SUBB>(ctx, g, x, dz, part);
}

static cf_status launch_splitk_reduce(const LaunchCtx& ctx, const float* part, float* dw, int64_t count, int splits,
                                      int accumulate) {
    // many splits of few columns (small-channel layers): split groups per block;
    // few splits of many columns: one group, 256 columns per block
    auto launch = [&](auto kern, int cols) {
        const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((count + cols - 1) / cols, 8LL * ctx.num_sms));
        kern<<<blocks, 256, 0, ctx.stream>>>(part, dw, count, splits, accumulate);
    };
    if (splits >= 256) launch(splitk_reduce_kernel<32>, 8);  // the first layer's per-CTA, per-phase partials
    else if (splits >= 64) launch(splitk_reduce_kernel<8>, 32);
    else if (splits >= 16) launch(splitk_reduce_kernel<4>, 64);
    else launch(splitk_reduce_kernel<1>, 256);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_wgrad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                       const uint16_t* x, const uint16_t* dz, const uint8_t* idx, float* dw, int accumulate, void* ws,
                       size_t ws_bytes) {
    if (!wgrad_shape_supported(c_in, c_out)) return CF_ERR_UNSUPPORTED;
    if (idx && !wgrad_routed_fused(c_in)) return CF_ERR_UNSUPPORTED;
    if ((c_in == 1 || c_in == 4) && (w * c_in) % 8 != 0) return CF_ERR_UNSUPPORTED;
    const size_t need = wgrad_workspace_bytes(ctx.num_sms, n, d, h, w, c_in, c_out);
    if (ws == nullptr || ws_bytes < need) return CF_ERR_WORKSPACE;
    float* part = static_cast<float*>(ws);
    int n_splits = 0;
    cf_status st;
    if (wgrad_halo_supported(c_in, c_out)) {
        st = launch_wgrad_halo(ctx, n, d, h, w, c_in, c_out, x, dz, part, &n_splits);
        if (st != CF_OK) return st;
        return launch_splitk_reduce(ctx, part, dw, (int64_t)c_out * 27 * c_in, n_splits, accumulate);
    }
    if (idx && wgrad_quad_supported(d, h, w, c_in, c_out)) {
        st = launch_wgrad_quad(ctx, n, d, h, w, x, dz, idx, part, &n_splits);
        if (st != CF_OK) return st;
        return launch_splitk_reduce(ctx, part, dw, (int64_t)c_out * 27 * c_in, n_splits, accumulate);
    }
    WgradGeom g = wgrad_geom(ctx.num_sms, n, d, h, w, c_in, c_out);
    n_splits = g.n_splits;
    if (c_in == 1 || c_in == 4) {
        st = launch_wgrad_smallc(ctx, g, x, dz, idx, part);
        if (st != CF_OK) return st;
        return launch_splitk_reduce(ctx, part, dw, (int64_t)c_out * 27 * c_in, n_splits, accumulate);
    }
    switch (g.bn) {
        case 16: st = wgrad_bn<16>(ctx, g, x, dz, part); break;
        case 32: st = wgrad_bn<32>(ctx, g, x, dz, part); break;
        case 48: st = wgrad_bn<48>(ctx, g, x, dz, part); break;
        case 64: st = wgrad_bn<64>(ctx, g, x, dz, part); break;
        case 96: st = wgrad_bn<96>(ctx, g, x, dz, part); break;
        case 128: st = wgrad_bn<128>(ctx, g, x, dz, part); break;
        case 192: st = wgrad_bn<192>(ctx, g, x, dz, part); break;
        case 256: st = wgrad_bn<256>(ctx, g, x, dz, part); break;
        default: return CF_ERR_UNSUPPORTED;
    }
    if (st != CF_OK) return st;
    return launch_splitk_reduce(ctx, part, dw, (int64_t)c_out * 27 * c_in, n_splits, accumulate);
}

}  // namespace cf
