// conv_wgrad_halo.cu -- backward-weight convolution that reads the layer input
// once per K block as a halo tile (c_in 32 or 64, c_out 32..256).
//
//   dW[co, t, ci] = sum_{n,v} dZ[n,v,co] * X[n, v + t - 1, ci]
// (CosmoFlow page, section III-C: the weight-gradient work is split over
// voxels).  GEMM: M = (tap, ci) rows, N = co, K = voxels.
//
// K block: 2 planes x 16 lines x 8 voxels (PLANES = 2) or 1 plane x 16 x 8.
// The producer loads the input halo of the block, (KC, 10, 18, PLANES + 2),
// and the block's dZ rows (BSUB channels per box).  Both operands are
// MN-major in shared memory:
//   A: M atoms are taps.  The A rows of tap t for voxel (i, j, l) are halo row
//      o(t) + (i*18 + j)*10 + l with o(t) = (kd*18 + kh)*10 + kw, so one UMMA
//      K step (16 voxels = 2 line segments of 8) has its two 8-row groups 10
//      rows apart (SBO), and the atoms of one M block start o(t2) - o(t1) rows
//      apart (LBO).  64-channel chunks (SW128): an M block is 2 taps
//      (t, t+1); 32-channel chunks (SW64): 4 atoms, the kw = 0, 1, 2 taps of
//      one (kd, kh) 1 row apart plus one unused atom.
//   B: dZ box rows are the block's voxels in (i, j, l) order, 8-row groups
//      1 line apart.
// A CTA owns a set of M blocks of one channel chunk (as many as fit in 512
// TMEM columns of fp32 accumulators) and a contiguous range of K blocks; its
// accumulators go to the split-K partial buffer [split][co][27*c_in], summed
// afterwards in a fixed order.  The halo makes each input row feed every tap
// group of the CTA instead of being re-fetched per tap.
//
// c_in 32 with c_out 32 or 64 and c_in 64 with c_out 64 or 128 run the
// depth-stacked variant further down (the depth tap moved onto the B operand:
// per K step 3 MMAs of N = 96 instead of 9 of N = 64 for c_in 32, 5 instead of
// 14 of N = 128 for c_in 64).
#include "conv_common.cuh"

namespace cf {

struct WhGeom {
    int N, D, H, W, Cin, Cout;
    int nb_w, nb_h, nb_d;     // K blocks per dimension
    int64_t total_kb;         // N * nb_d * nb_h * nb_w
    int blocks_per_chunk;     // M blocks per channel chunk
    int n_chunks;
    int sets_per_chunk;       // M-block sets per chunk (one set per CTA unit)
    int g_per_set;            // M blocks per set (last set may be short)
    int n_sets;               // sets_per_chunk * n_chunks
    int n_splits;
    int64_t kb_per_split;
    int num_units;            // n_sets * n_splits
};

__host__ __device__ constexpr int wh_tap_offset(int t) { return ((t / 9) * 18 + (t / 3) % 3) * 10 + t % 3; }

template <int KC, int BN, int PLANES>
struct WhCfg {
    static constexpr int ROW = KC * 2;
    static constexpr int HALO_ROWS = 10 * 18 * (PLANES + 2);
    static constexpr uint32_t HALO_BYTES = HALO_ROWS * ROW;
    static constexpr uint32_t HALO_STRIDE = (HALO_BYTES + 1024 + 1023) / 1024 * 1024;  // + slack for unused atoms
    static constexpr int KV = 128 * PLANES;  // voxels per K block
    static constexpr int BSUB = BN >= 64 ? 64 : BN;
    static constexpr uint32_t B_SUB_BYTES = KV * BSUB * 2;
    static constexpr uint32_t B_BYTES = KV * BN * 2;
    static constexpr uint32_t STAGE_BYTES = HALO_STRIDE + B_BYTES;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr int STAGES_RAW = (int)((227 * 1024 - 1024 - BAR_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_RAW > 4 ? 4 : STAGES_RAW;
    static constexpr uint32_t SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static constexpr uint32_t SWZ_A = KC == 64 ? SWZ_128B : SWZ_64B;
    static constexpr uint32_t SWZ_B = BSUB == 64 ? SWZ_128B : SWZ_64B;
    static constexpr uint32_t SBO_A = 10 * ROW;        // next line segment of the block
    static constexpr uint32_t SBO_B = 8 * BSUB * 2;    // next 8 voxels of the block
    static constexpr int GMAX = 512 / BN;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 1, 1);
    static_assert(STAGES >= 2, "shared memory");
};

struct WhParams {
    WhGeom g;
    float* part;
    int* status;
    uint64_t wait_ns;
};

// Taps of M block b of a chunk: first tap and the byte distance between atoms.
template <int KC>
__device__ __forceinline__ void wh_block_taps(int b, int& t_first, int& lbo_rows, int& natoms_real) {
    if (KC == 64) {  // pairs (2b, 2b+1); the last block has one tap
        t_first = 2 * b;
        const int t2 = 2 * b + 1;
        natoms_real = t2 < 27 ? 2 : 1;
        lbo_rows = t2 < 27 ? wh_tap_offset(t2) - wh_tap_offset(t_first) : 1;
    } else {  // (kd, kh) = b: taps kw = 0, 1, 2 one row apart, fourth atom unused
        t_first = 3 * b;
        lbo_rows = 1;
        natoms_real = 3;
    }
}

// Unit u of the CTA grid (size G) -> (M-block set, K split).  With two sets,
// the CTAs pair up on a split in every round (b and b^1 read the same K
// blocks, so the second read hits L2) and alternate sets between rounds, so
// that a CTA's units are not all of the larger set.
__device__ __forceinline__ void wh_unit(const WhGeom& g, int u, int G, int& set, int& split) {
    if (g.n_sets == 2 && (G & 1) == 0) {
        const int r = u / G, b = u - r * G;
        split = r * (G / 2) + (b >> 1);
        set = (b + r) & 1;
    } else {
        set = u % g.n_sets;
        split = u / g.n_sets;
    }
}

template <int KC, int BN, int PLANES>
__global__ void __launch_bounds__(224, 1)
    wgrad_halo_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                      const WhParams p) {
    using C = WhCfg<KC, BN, PLANES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;  // stage: [halo][dZ]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;  // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WhGeom& g = p.g;

    if (threadIdx.x == 0) {
        // stages are released and the accumulators completed by both MMA issuers
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);
        }
        mbar_init(tfull, 2);
        mbar_init(tempty, 128);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: halo + dZ of every K block of the unit
            int stage = 0;
            uint32_t phase = 0, issued = 0, par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x) {
                int set, split;
                wh_unit(g, u, (int)gridDim.x, set, split);
                const int chunk = set / g.sets_per_chunk;
                const int64_t k0 = (int64_t)split * g.kb_per_split;
                const int64_t k1 = k0 + g.kb_per_split < g.total_kb ? k0 + g.kb_per_split : g.total_kb;
                int64_t b = k0;
                int bw = (int)(b % g.nb_w);
                b /= g.nb_w;
                int bh = (int)(b % g.nb_h);
                b /= g.nb_h;
                int bd = (int)(b % g.nb_d);
                int n = (int)(b / g.nb_d);
                for (int64_t kb = k0; kb < k1; ++kb) {
                    const int w0 = bw * 8, h0 = bh * 16, d0 = bd * PLANES;
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = ring + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::HALO_BYTES + C::B_BYTES);
                    tma_load_5d(st, &tmX, &full[stage], chunk * KC, w0 - 1, h0 - 1, d0 - 1, n);
#pragma unroll
                    for (int a = 0; a < BN / C::BSUB; ++a)
                        tma_load_5d(st + C::HALO_STRIDE + a * C::B_SUB_BYTES, &tmG, &full[stage], a * C::BSUB, w0, h0,
                                    d0, n);
                    issued |= 1u << stage;
                    par = (par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
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
            }
            if (!ok) {
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&full[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 6) {
        if (lane == 0) {
            // ---------------- MMA issuers: warp 1 takes the even M blocks of the set,
            // warp 6 the odd ones (one thread's issue rate bounds narrow-N MMAs)
            const int mi = warp == 1 ? 0 : 1;
            int stage = 0;
            uint32_t phase = 0, local = 0;
            bool ok = true;
            const uint64_t adesc_base = sdesc(smem_u32(ring), 0, C::SBO_A, C::SWZ_A);
            const uint64_t bdesc_base = sdesc(smem_u32(ring) + C::HALO_STRIDE, C::B_SUB_BYTES, C::SBO_B, C::SWZ_B);
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x, ++local) {
                int set, split;
                wh_unit(g, u, (int)gridDim.x, set, split);
                const int sub = set % g.sets_per_chunk;
                const int mb0 = sub * g.g_per_set;
                const int nmb = min(g.g_per_set, g.blocks_per_chunk - mb0);
                const int64_t k0 = (int64_t)split * g.kb_per_split;
                const int64_t k1 = k0 + g.kb_per_split < g.total_kb ? k0 + g.kb_per_split : g.total_kb;
                if (!mbar_wait(tempty, (local & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int64_t kb = k0; kb < k1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_st = adesc_base + ((stage * C::STAGE_BYTES) >> 4);
                    const uint64_t b_st = bdesc_base + ((stage * C::STAGE_BYTES) >> 4);
                    for (int m = mi; m < nmb; m += 2) {
                        int t1, lbo_rows, nreal;
                        wh_block_taps<KC>(mb0 + m, t1, lbo_rows, nreal);
                        const uint64_t a_m = (a_st + ((uint32_t)(wh_tap_offset(t1) * C::ROW) >> 4)) |
                                             ((uint64_t)(((uint32_t)(lbo_rows * C::ROW) >> 4) & 0x3FFFu) << 16);
                        const uint32_t d_tmem = tmem_base + m * BN;
#pragma unroll
                        for (int s = 0; s < C::KV / 16; ++s) {
                            // K step s: voxels 16s..16s+15 = plane s/8, lines 2(s%8), 2(s%8)+1
                            const int i = s >> 3, j = 2 * (s & 7);
                            const uint64_t ad = a_m + ((uint32_t)((i * 18 + j) * 10 * C::ROW) >> 4);
                            const uint64_t bd = b_st + ((uint32_t)(s * 16 * C::BSUB * 2) >> 4);
                            umma_bf16(d_tmem, ad, bd, C::IDESC, (kb != k0 || s != 0) ? 1u : 0u);
                        }
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
                umma_commit(&drain[mi]);
                mbar_wait_timed(&drain[mi], 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5): accumulator rows (atom, ci) -> partial[split][co][t*Cin + ci]
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        const int r = q * 32 + lane;
        const int KK = 27 * g.Cin;
        uint32_t local = 0;
        for (int u = blockIdx.x; u < g.num_units; u += gridDim.x, ++local) {
            int set, split;
            wh_unit(g, u, (int)gridDim.x, set, split);
            const int chunk = set / g.sets_per_chunk, sub = set % g.sets_per_chunk;
            const int mb0 = sub * g.g_per_set;
            const int nmb = min(g.g_per_set, g.blocks_per_chunk - mb0);
            if (!epi_wait(tfull, local & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            const int atom = r / KC, ci = chunk * KC + r % KC;
            for (int m = 0; m < nmb; ++m) {
                int t1, lbo_rows, nreal;
                wh_block_taps<KC>(mb0 + m, t1, lbo_rows, nreal);
                const bool real = atom < nreal;
                const int t = t1 + atom;
                float* dst = p.part + (int64_t)split * g.Cout * KK + (int64_t)t * g.Cin + ci;
                const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + m * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t v[32];
                    tmem_ld16(lane_addr + c, v);
                    tmem_ld_wait();
                    if (real) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (c + k < g.Cout) dst[(int64_t)(c + k) * KK] = __uint_as_float(v[k]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------
// Depth-stacked variant for c_in = 32 or 64 (the layer-2 and layer-3 shapes):
//
//   dW[co, (kd,kh,kw), ci] = sum_u dZ[u - (kd-1) e_d, co] * X[u + (0, kh-1, kw-1), ci]
//
// (the sum over v with u = v + (kd-1) e_d).  The depth tap moves from the A
// operand to the B operand: A = the input halo of the K block without a depth
// halo (PLANES x 18 x 10 rows); B = dZ of the block's planes and one plane on
// either side, for one set of 32 output channels, and its N atoms are the
// kd = 2, 1, 0 shifts of it, one plane (8 KB) apart, so one MMA of width 96
// covers all three depth taps.  M blocks cover the nine (kh, kw) taps:
//   c_in 32 (64-byte rows): one block per kh, atoms kw = 0, 1, 2 one row
//     apart plus an unused fourth atom;
//   c_in 64 (128-byte rows): blocks of two taps in (kh, kw) order, the second
//     atom at its own row distance (LBO), the fifth block one tap.
// Per K step that is 3 (or 5) MMAs of N = 96 instead of 9 (or 14) MMAs of
// N = 64 (or 128) over a depth halo, and each K block is loaded once per
// 32-channel output set with a third of the input planes.  Accumulator of
// block m: TMEM columns m*96 + a*32 + co (a = 2 - kd), lanes atom*KC + ci.
// A CTA unit is one output set and a contiguous K range.
namespace {
constexpr int WK_PLANES = 2;
constexpr int WK_KV = 128 * WK_PLANES;  // voxels per K block
constexpr uint32_t WK_G_PLANE = 128 * 64;  // one dZ plane of the set
constexpr uint32_t WK_G_BYTES = (WK_PLANES + 2) * WK_G_PLANE;
constexpr uint32_t WK_IDESC = idesc_bf16(128, 96, 1, 1);

template <int KC>
struct WkCfg {
    static constexpr uint32_t ROW = KC * 2;
    static constexpr uint32_t X_BYTES = 10 * 18 * WK_PLANES * ROW;
    static constexpr uint32_t X_STRIDE = (X_BYTES + 1024 + 1023) / 1024 * 1024;  // + slack read by a spare atom
    static constexpr uint32_t STAGE = X_STRIDE + WK_G_BYTES;
    static constexpr int STAGES_RAW = (int)((227 * 1024 - 1024 - 256) / STAGE);
    static constexpr int STAGES = STAGES_RAW > 4 ? 4 : STAGES_RAW;
    static constexpr uint32_t SMEM = 1024 + STAGES * STAGE + 256;
    static constexpr int NBLK = KC == 32 ? 3 : 5;
    static constexpr uint32_t SWZ = KC == 32 ? SWZ_64B : SWZ_128B;
    static_assert(STAGES >= 2, "shared memory");
    static_assert(NBLK * 96 <= 512, "tensor memory");
};

// Row offset of (kh, kw) tap p in the halo, its block's first row and the row
// distance of the block's second atom.
__host__ __device__ constexpr int wk_tap_rows(int p) { return (p / 3) * 10 + p % 3; }
template <int KC>
__device__ __forceinline__ void wk_block(int m, int& first_rows, int& lbo_rows) {
    if (KC == 32) {
        first_rows = m * 10;
        lbo_rows = 1;
    } else {
        first_rows = wk_tap_rows(2 * m);
        lbo_rows = 2 * m + 1 < 9 ? wk_tap_rows(2 * m + 1) - first_rows : 1;
    }
}
}  // namespace

template <int KC>
__global__ void __launch_bounds__(224, 1)
    wgrad_halo_kd_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                         const WhParams p) {
    using C = WkCfg<KC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;  // stage: [input halo][dZ planes d0-1 .. d0+PLANES]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;  // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WhGeom& g = p.g;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);
        }
        mbar_init(tfull, 2);
        mbar_init(tempty, 128);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: input halo + the set's dZ planes per K block
            int stage = 0;
            uint32_t phase = 0, issued = 0, par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x) {
                int set, split;
                wh_unit(g, u, (int)gridDim.x, set, split);
                const int64_t k0 = (int64_t)split * g.kb_per_split;
                const int64_t k1 = k0 + g.kb_per_split < g.total_kb ? k0 + g.kb_per_split : g.total_kb;
                // K blocks depth fastest: consecutive blocks share two of their
                // four dZ planes, which the next load then finds in L2
                int64_t b = k0;
                int bd = (int)(b % g.nb_d);
                b /= g.nb_d;
                int bw = (int)(b % g.nb_w);
                b /= g.nb_w;
                int bh = (int)(b % g.nb_h);
                int n = (int)(b / g.nb_h);
                for (int64_t kb = k0; kb < k1; ++kb) {
                    const int w0 = bw * 8, h0 = bh * 16, d0 = bd * WK_PLANES;
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = ring + stage * C::STAGE;
                    mbar_arrive_expect_tx(&full[stage], C::X_BYTES + WK_G_BYTES);
                    tma_load_5d(st, &tmX, &full[stage], 0, w0 - 1, h0 - 1, d0, n);
                    tma_load_5d(st + C::X_STRIDE, &tmG, &full[stage], set * 32, w0, h0, d0 - 1, n);
                    issued |= 1u << stage;
                    par = (par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++bd == g.nb_d) {
                        bd = 0;
                        if (++bw == g.nb_w) {
                            bw = 0;
                            if (++bh == g.nb_h) {
                                bh = 0;
                                ++n;
                            }
                        }
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&full[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 6) {
        if (lane == 0) {
            // ---------------- MMA issuers: warp 1 takes the even M blocks, warp 6 the odd ones
            const int mi = warp == 1 ? 0 : 1;
            int stage = 0;
            uint32_t phase = 0, local = 0;
            bool ok = true;
            const uint64_t adesc_base = sdesc(smem_u32(ring), 0, 10 * C::ROW, C::SWZ);
            const uint64_t bdesc_base = sdesc(smem_u32(ring) + C::X_STRIDE, WK_G_PLANE, 8 * 64, SWZ_64B);
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x, ++local) {
                int set, split;
                wh_unit(g, u, (int)gridDim.x, set, split);
                const int64_t k0 = (int64_t)split * g.kb_per_split;
                const int64_t k1 = k0 + g.kb_per_split < g.total_kb ? k0 + g.kb_per_split : g.total_kb;
                if (!mbar_wait(tempty, (local & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int64_t kb = k0; kb < k1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_st = adesc_base + ((stage * C::STAGE) >> 4);
                    const uint64_t b_st = bdesc_base + ((stage * C::STAGE) >> 4);
                    for (int m = mi; m < C::NBLK; m += 2) {
                        int first_rows, lbo_rows;
                        wk_block<KC>(m, first_rows, lbo_rows);
                        const uint64_t a_m = (a_st + ((uint32_t)(first_rows * C::ROW) >> 4)) |
                                             ((uint64_t)(((uint32_t)(lbo_rows * C::ROW) >> 4) & 0x3FFFu) << 16);
                        const uint32_t d_tmem = tmem_base + m * 96;
#pragma unroll
                        for (int s = 0; s < WK_KV / 16; ++s) {
                            // K step s: voxels 16s..16s+15 = plane s/8, lines 2(s%8), 2(s%8)+1
                            const int i = s >> 3, j = 2 * (s & 7);
                            const uint64_t ad = a_m + ((uint32_t)((i * 18 + j) * 10 * C::ROW) >> 4);
                            const uint64_t bd = b_st + ((uint32_t)((i * 128 + j * 8) * 64) >> 4);
                            umma_bf16(d_tmem, ad, bd, WK_IDESC, (kb != k0 || s != 0) ? 1u : 0u);
                        }
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
                umma_commit(&drain[mi]);
                mbar_wait_timed(&drain[mi], 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5): lane r = atom*KC + ci; column a*32 + c
        // of block m -> co = set*32 + c, kd = 2 - a, (kh, kw) tap p of the atom
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        const int KK = 27 * g.Cin;
        uint32_t local = 0;
        for (int u = blockIdx.x; u < g.num_units; u += gridDim.x, ++local) {
            int set, split;
            wh_unit(g, u, (int)gridDim.x, set, split);
            if (!epi_wait(tfull, local & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            const int r = q * 32 + lane, atom = r / KC, ci = r % KC;
            for (int m = 0; m < C::NBLK; ++m) {
                const int p9 = KC == 32 ? m * 3 + atom : 2 * m + atom;  // (kh, kw) tap
                if ((KC == 32 && atom == 3) || p9 >= 9) continue;        // spare atom: whole warp skips
                {
                    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + m * 96;
#pragma unroll 1
                    for (int c = 0; c < 96; c += 16) {
                        uint32_t v[32];
                        tmem_ld16(lane_addr + c, v);
                        tmem_ld_wait();
                        const int a = c >> 5, kd = 2 - a;
                        const int t = kd * 9 + p9;
                        float* dst = p.part + (int64_t)split * g.Cout * KK + (int64_t)(set * 32 + (c & 31)) * KK +
                                     t * g.Cin + ci;
#pragma unroll
                        for (int k = 0; k < 16; ++k) dst[(int64_t)k * KK] = __uint_as_float(v[k]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------
// host side

template <int KC, int BN, int PLANES>
static WhGeom wh_geom(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    using C = WhCfg<KC, BN, PLANES>;
    WhGeom g;
    g.N = (int)n;
    g.D = (int)d;
    g.H = (int)h;
    g.W = (int)w;
    g.Cin = c_in;
    g.Cout = c_out;
    g.nb_w = (int)((w + 7) / 8);
    g.nb_h = (int)((h + 15) / 16);
    g.nb_d = (int)((d + PLANES - 1) / PLANES);
    g.total_kb = n * g.nb_d * g.nb_h * g.nb_w;
    g.blocks_per_chunk = KC == 64 ? 14 : 9;
    g.n_chunks = c_in / KC;
    g.sets_per_chunk = (g.blocks_per_chunk + C::GMAX - 1) / C::GMAX;
    g.g_per_set = (g.blocks_per_chunk + g.sets_per_chunk - 1) / g.sets_per_chunk;
    g.n_sets = g.sets_per_chunk * g.n_chunks;
    // at most one unit per SM (one round of CTAs): half the partial sums of two
    // units per SM (measured in the five-block step: 1.470 -> 1.416 ms together
    // with the per-tap kernel's)
    int64_t target = std::max<int64_t>(1, (int64_t)num_sms / g.n_sets);
    target = std::min<int64_t>(target, std::max<int64_t>(1, g.total_kb / 4));
    g.kb_per_split = (g.total_kb + target - 1) / target;
    g.n_splits = (int)((g.total_kb + g.kb_per_split - 1) / g.kb_per_split);
    g.num_units = g.n_sets * g.n_splits;
    return g;
}

// Geometry of the depth-stacked variant: one M-block set per 32 output
// channels, K blocks of 2 planes.
static WhGeom wk_geom(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    WhGeom g;
    g.N = (int)n;
    g.D = (int)d;
    g.H = (int)h;
    g.W = (int)w;
    g.Cin = c_in;
    g.Cout = c_out;
    g.nb_w = (int)((w + 7) / 8);
    g.nb_h = (int)((h + 15) / 16);
    g.nb_d = (int)((d + WK_PLANES - 1) / WK_PLANES);
    g.total_kb = n * g.nb_d * g.nb_h * g.nb_w;
    g.blocks_per_chunk = c_in == 32 ? WkCfg<32>::NBLK : WkCfg<64>::NBLK;
    g.n_chunks = 1;
    g.sets_per_chunk = c_out / 32;
    g.g_per_set = g.blocks_per_chunk;
    g.n_sets = g.sets_per_chunk;
    // at most one unit per SM (one round of CTAs): half the partial sums of two
    // units per SM (measured in the five-block step: 1.470 -> 1.416 ms together
    // with the per-tap kernel's)
    int64_t target = std::max<int64_t>(1, (int64_t)num_sms / g.n_sets);
    target = std::min<int64_t>(target, std::max<int64_t>(1, g.total_kb / 4));
    g.kb_per_split = (g.total_kb + target - 1) / target;
    g.n_splits = (int)((g.total_kb + g.kb_per_split - 1) / g.kb_per_split);
    g.num_units = g.n_sets * g.n_splits;
    return g;
}

// c_in 32 with one or two output-channel sets and c_in 64 with two or four
// take the depth-stacked variant (measured on the layer-2 shape, 8 x 64^3,
// 32 -> 64: 0.246 -> 0.184 ms; on the layer-3 shape, 8 x 32^3, 64 -> 128:
// 0.097 -> 0.088 ms alone, and the five-block step 1.338 -> 1.315 ms).
static bool wk_path(int c_in, int c_out) {
    return (c_in == 32 && (c_out == 32 || c_out == 64)) || (c_in == 64 && (c_out == 64 || c_out == 128));
}

bool wgrad_halo_supported(int c_in, int c_out) {
    return (c_in == 32 && (c_out == 32 || c_out == 64 || c_out == 128)) ||
           (c_in == 64 && (c_out == 64 || c_out == 128));
}

// Geometry of the configuration launch_wgrad_halo picks for (c_in, c_out).
static bool wh_dispatch_geom(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                             WhGeom* g) {
    if (wk_path(c_in, c_out)) *g = wk_geom(num_sms, n, d, h, w, c_in, c_out);
    else if (c_in == 32 && c_out == 128) *g = wh_geom<32, 128, 1>(num_sms, n, d, h, w, c_in, c_out);
    else if (c_in == 64 && c_out == 64) *g = wh_geom<64, 64, 1>(num_sms, n, d, h, w, c_in, c_out);
    else if (c_in == 64 && c_out == 128) *g = wh_geom<64, 128, 1>(num_sms, n, d, h, w, c_in, c_out);
    else return false;
    return true;
}

size_t wgrad_halo_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    WhGeom g;
    if (!wh_dispatch_geom(num_sms, n, d, h, w, c_in, c_out, &g)) return 0;
    return (size_t)g.n_splits * c_out * 27 * c_in * sizeof(float);
}

template <int KC, int BN, int PLANES>
static cf_status run_wgrad_halo(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                                int c_out, const uint16_t* x, const uint16_t* dz, float* part, int* n_splits) {
    using C = WhCfg<KC, BN, PLANES>;
    WhGeom g = wh_geom<KC, BN, PLANES>(ctx.num_sms, n, d, h, w, c_in, c_out);
    *n_splits = g.n_splits;
    CUtensorMap tx, tg;
    const uint64_t dx[5] = {(uint64_t)c_in, (uint64_t)w, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t sx[4] = {(uint64_t)c_in * 2, (uint64_t)w * c_in * 2, (uint64_t)h * w * c_in * 2,
                            (uint64_t)d * h * w * c_in * 2};
    const uint32_t bx[5] = {(uint32_t)KC, 10u, 18u, (uint32_t)(PLANES + 2), 1u};
    if (!encode_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dx, sx, bx,
                     KC == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return CF_ERR_CUDA;
    const uint64_t dg[5] = {(uint64_t)c_out, (uint64_t)w, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t sg[4] = {(uint64_t)c_out * 2, (uint64_t)w * c_out * 2, (uint64_t)h * w * c_out * 2,
                            (uint64_t)d * h * w * c_out * 2};
    const uint32_t bg[5] = {(uint32_t)C::BSUB, 8u, 16u, (uint32_t)PLANES, 1u};
    if (!encode_tmap(&tg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, dz, dg, sg, bg,
                     C::BSUB == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return CF_ERR_CUDA;
    WhParams p{g, part, ctx.status, ctx.wait_ns};
    auto kern = wgrad_halo_kernel<KC, BN, PLANES>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = std::max(1, std::min(g.num_units, ctx.num_sms));
    kern<<<grid, 224, C::SMEM, ctx.stream>>>(tx, tg, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int KC>
static cf_status run_wgrad_halo_kd(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in,
                                   int c_out, const uint16_t* x, const uint16_t* dz, float* part, int* n_splits) {
    WhGeom g = wk_geom(ctx.num_sms, n, d, h, w, c_in, c_out);
    *n_splits = g.n_splits;
    CUtensorMap tx, tg;
    const uint64_t dx[5] = {(uint64_t)c_in, (uint64_t)w, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t sx[4] = {(uint64_t)c_in * 2, (uint64_t)w * c_in * 2, (uint64_t)h * w * c_in * 2,
                            (uint64_t)d * h * w * c_in * 2};
    const uint32_t bx[5] = {(uint32_t)KC, 10u, 18u, (uint32_t)WK_PLANES, 1u};
    if (!encode_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dx, sx, bx,
                     KC == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return CF_ERR_CUDA;
    const uint64_t dg[5] = {(uint64_t)c_out, (uint64_t)w, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t sg[4] = {(uint64_t)c_out * 2, (uint64_t)w * c_out * 2, (uint64_t)h * w * c_out * 2,
                            (uint64_t)d * h * w * c_out * 2};
    const uint32_t bg[5] = {32u, 8u, 16u, (uint32_t)(WK_PLANES + 2), 1u};
    if (!encode_tmap(&tg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, dz, dg, sg, bg, CU_TENSOR_MAP_SWIZZLE_64B))
        return CF_ERR_CUDA;
    WhParams p{g, part, ctx.status, ctx.wait_ns};
    auto kern = wgrad_halo_kd_kernel<KC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WkCfg<KC>::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = std::max(1, std::min(g.num_units, ctx.num_sms));
    kern<<<grid, 224, WkCfg<KC>::SMEM, ctx.stream>>>(tx, tg, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_wgrad_halo(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                            const uint16_t* x, const uint16_t* dz, float* part, int* n_splits) {
    if (wk_path(c_in, c_out))
        return c_in == 32 ? run_wgrad_halo_kd<32>(ctx, n, d, h, w, c_in, c_out, x, dz, part, n_splits)
                          : run_wgrad_halo_kd<64>(ctx, n, d, h, w, c_in, c_out, x, dz, part, n_splits);
    if (c_in == 32) {
        if (c_out == 128) return run_wgrad_halo<32, 128, 1>(ctx, n, d, h, w, c_in, c_out, x, dz, part, n_splits);
    } else if (c_in == 64) {
        if (c_out == 64) return run_wgrad_halo<64, 64, 1>(ctx, n, d, h, w, c_in, c_out, x, dz, part, n_splits);
        if (c_out == 128) return run_wgrad_halo<64, 128, 1>(ctx, n, d, h, w, c_in, c_out, x, dz, part, n_splits);
    }
    return CF_ERR_UNSUPPORTED;
}

}  // namespace cf
