// conv_smallc.cu -- forward conv of the small-channel first layer (c_in = 1
// or 4; CosmoFlow input: four redshift channels) as an implicit GEMM whose A
// operand lives in tensor memory.
//
// GEMM view: D[m, co] = sum_k A[m, k] * W[co, k] with k = 4*t + ci
// (t = 9*kd + 3*kh + kw), K = 27*c_in padded to 112 (c_in 4) or 32 (c_in 1).
//
// Output tile: 2 planes x 16 lines x 16 voxels (512 voxels), computed as four
// M=128 row blocks, one per (plane, line parity); row r of a block is voxel
// r % 16 of line pair r / 16.  The four (plane, line) members of a 2x2x2
// pooling window are thus the same TMEM lane of the four blocks and its two
// voxels are adjacent lanes: the pooling is a per-thread reduction plus one
// exchange between lane pairs, which also splits the finalisation (bias,
// activation, stores) of the window's channels between the two lanes.
//
// With only 8 (or 2) bytes per voxel, an im2col tile in shared memory would
// be written and read once per tap and bound the kernel by shared-memory
// bandwidth.  Instead:
//   warp 0      : TMA of the tile's input halo (one box of the input viewed as
//                 (W*C, H, D, N): 4 planes x 18 lines x (16 + 2*margin) voxels,
//                 zero outside the volume) into a ring;
//   warps 2..9  : builders, two groups of four warps (one per TMEM lane
//                 quarter); group g fills row blocks g and g + 2 of every tile.
//                 Each thread gathers the im2col row of its voxel from the halo
//                 (27 independent 8-byte loads; a half-warp reads 16
//                 consecutive voxels of one halo line, 128 contiguous bytes, so
//                 the loads are free of bank conflicts) and writes it into the
//                 block's tensor-memory A buffer with tcgen05.st;
//   warps 1, 18 : tcgen05.mma with A from tensor memory and the filter
//                 (resident in shared memory, K-major SW128) as B; warp 1
//                 issues row blocks 0 and 1, warp 18 blocks 2 and 3 (one
//                 thread's issue rate would bound these N = 32 MMAs);
//   warps 10..17: epilogue (fused bias + leaky ReLU + 2x2x2 max-pool with
//                 argmax, or plain bf16), two warps per TMEM lane quarter
//                 splitting the channels.
#include "halo_common.cuh"
#include "smallc_common.cuh"

namespace cf {

constexpr int SC_W = 16, SC_H = 16, SC_D = 2;  // output tile (voxels, lines, planes)
constexpr int SC_BLOCKS = 4;                   // M=128 row blocks per tile: (plane, line parity)

template <int CIN, int BN, int EPI>
struct SmallTmCfg {
    static constexpr int KREAL = 27 * CIN;
    static constexpr int KP = (KREAL + 15) / 16 * 16;  // 112 or 32
    static constexpr int KSTEPS = KP / 16;
    static constexpr int PCOLS = CIN == 4 ? 64 : 16;   // TMEM columns per A block (56 / 16 used)
    static constexpr int ATOMS = (KP + 63) / 64;
    static constexpr uint32_t B_BYTES = BN * 128 * ATOMS;
    static constexpr int MARGIN = 16 / (2 * CIN);       // halo voxels left of the tile (16-byte start)
    static constexpr int PITCH = (SC_W + 2 * MARGIN) * CIN * 2;  // bytes per halo line: 160 or 64
    static constexpr int HALO_BYTES = (SC_D + 2) * (SC_H + 2) * PITCH;  // 11520 or 4608
    static constexpr uint32_t HALO_STRIDE = (HALO_BYTES + 1023) / 1024 * 1024;
    static constexpr int HS = CIN == 4 ? 8 : 12;        // halo stages in flight (TMA latency)
    static constexpr int ACC_COLS = SC_BLOCKS * BN;      // accumulator columns of one tile
    static constexpr int NACC = (2 * ACC_COLS + SC_BLOCKS * PCOLS <= 512) ? 2 : 1;
    static constexpr uint32_t ACOL0 = NACC * ACC_COLS;   // first A column
    static constexpr uint32_t BAR_BYTES = 8 * (2 * HS + 2 * SC_BLOCKS + 2 * 2 + 2) + 16;
    static constexpr uint32_t SMEM = 1024 + B_BYTES + HS * HALO_STRIDE + BAR_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 0, 0);
    static_assert(ACOL0 + SC_BLOCKS * PCOLS <= TMEM_COLS, "tensor memory budget");
};

struct SmallTmParams {
    HaloParams hp;
    const uint16_t* w;  // [Cout][27*CIN]
};

struct SmallTile {
    int n, d0, h0, w0;
};

// Tiles are numbered N tile fastest, then w, h, d, n.
__device__ __forceinline__ SmallTile small_decode(const HaloParams& p, int tile) {
    SmallTile t;
    const TileIdx r = tile_index(p, tile);
    t.n = r.n;
    t.w0 = r.tw * SC_W;
    t.h0 = r.th * SC_H;
    t.d0 = r.td * SC_D;
    return t;
}

// im2col row of the voxel (plane pl, line ln, voxel v) of the tile, from its
// halo.  c_in = 4: tap t = 9*kd + 3*kh + kw is halo voxel v + kw of halo line
// (pl + kd, ln + kh), K index 4*t + ci (54 words + 2 zero words).  c_in = 1:
// 27 taps padded to 32 (16 words).
template <int CIN>
__device__ __forceinline__ void gather_row(const uint8_t* halo, int pl, int ln, int v, uint32_t (&wd)[56]) {
    using C = SmallTmCfg<CIN, 16, EPI_PLAIN>;
    if (CIN == 4) {
        const uint8_t* base = halo + (pl * (SC_H + 2) + ln) * C::PITCH + (v + C::MARGIN - 1) * 8;
#pragma unroll
        for (int kd = 0; kd < 3; ++kd)
#pragma unroll
            for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                for (int kw = 0; kw < 3; ++kw) {
                    const uint2 x = *reinterpret_cast<const uint2*>(base + (kd * (SC_H + 2) + kh) * C::PITCH + kw * 8);
                    const int t = kd * 9 + kh * 3 + kw;
                    wd[2 * t] = x.x;
                    wd[2 * t + 1] = x.y;
                }
        wd[54] = wd[55] = 0u;
    } else {
        uint32_t e[32];
#pragma unroll
        for (int t = 27; t < 32; ++t) e[t] = 0u;
#pragma unroll
        for (int kd = 0; kd < 3; ++kd)
#pragma unroll
            for (int kh = 0; kh < 3; ++kh) {
                const uint16_t* line =
                    reinterpret_cast<const uint16_t*>(halo + ((pl + kd) * (SC_H + 2) + ln + kh) * C::PITCH);
#pragma unroll
                for (int kw = 0; kw < 3; ++kw) e[kd * 9 + kh * 3 + kw] = line[v + C::MARGIN - 1 + kw];
            }
#pragma unroll
        for (int q = 0; q < 16; ++q) wd[q] = e[2 * q] | (e[2 * q + 1] << 16);
    }
}

template <int CIN, int BN, int EPI>
__global__ void __launch_bounds__(608, 1)
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
    uint64_t* aempty = afull + SC_BLOCKS;
    uint64_t* tfull = aempty + SC_BLOCKS;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;  // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int co0 = (blockIdx.x % p.n_ntiles) * BN;  // the CTA's N tile (see the launch)

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::HS; ++s) {
            mbar_init(&hfull[s], 1);
            mbar_init(&hempty[s], 8);  // one arrival per builder warp
        }
        for (int b = 0; b < SC_BLOCKS; ++b) {
            mbar_init(&afull[b], 4);   // one arrival per builder warp of the group
            mbar_init(&aempty[b], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 2);  // both MMA issuers
            mbar_init(&tempty[a], 8);  // one arrival per epilogue warp
            mbar_init(&drain[a], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmH);
    }
    // resident filter of the CTA's N tile: rows co0 .. co0+BN-1 (zero at and
    // above Cout), K padded with zeros, SW128 K-major atoms of 64 K-elements.
    // Tiles are dealt with stride gridDim.x and the launch makes gridDim.x a
    // multiple of n_ntiles, so every tile of this CTA has the same N tile.
    {
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
                const SmallTile t = small_decode(p, tile);
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
    } else if (warp == 1 || warp == 18) {
        if (lane == 0) {
            // ---------------- MMA issuers: per tile, row blocks 0, 1 (warp 1) or 2, 3 (warp 18)
            const int bi = warp == 1 ? 0 : 1;
            uint32_t aph = 0, local = 0;
            bool ok = true;
            const uint32_t b_addr = smem_u32(bsm);
            uint64_t bdk[C::KSTEPS];  // the filter's K-step descriptors (fixed)
#pragma unroll
            for (int k = 0; k < C::KSTEPS; ++k)
                bdk[k] = sdesc(b_addr + (k >> 2) * (BN * 128) + (k & 3) * 32, 16, 1024, SWZ_128B);
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
                const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
#pragma unroll 1
                for (int blk = 2 * bi; blk < 2 * bi + 2; ++blk) {
                    if (!mbar_wait(&afull[blk], aph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS + blk * BN;
                    const uint32_t a_tmem = tmem_base + C::ACOL0 + blk * C::PCOLS;
#pragma unroll
                    for (int k = 0; k < C::KSTEPS; ++k)
                        umma_bf16_tmem_a(d_tmem, a_tmem + 8 * k, bdk[k], C::IDESC, k != 0);
                    umma_commit(&aempty[blk]);
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                aph ^= 1;
            }
            if (!ok) {
                umma_commit(&drain[bi]);
                mbar_wait_timed(&drain[bi], 0, p.wait_ns);
            }
        }
    } else if (warp < 10) {
        // ---------------- builders: group g (warps 2..5 / 6..9) fills blocks g and g + 2
        const int q = warp & 3;
        const int g = (warp - 2) >> 2;
        const int lp = 2 * q + (lane >> 4), v = lane & 15;  // row 32q + lane: line pair, voxel
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + C::ACOL0;
        int hs = 0;
        uint32_t hph = 0, aph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            // every lane waits, and the warp leaves together if any lane gave up, so
            // the .sync.aligned tensor-memory stores below always see the full warp
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&hfull[hs], hph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)))
                break;
            const uint8_t* halo = hring + hs * C::HALO_STRIDE;
#pragma unroll 1
            for (int b2 = 0; b2 < 2; ++b2) {
                const int blk = g + 2 * b2;
                uint32_t wd[56];
                gather_row<CIN>(halo, blk >> 1, 2 * lp + (blk & 1), v, wd);
                if (b2 == 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&hempty[hs]);
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&aempty[blk], aph ^ 1, abort_flag, p.wait_ns, p.status,
                                                       WAIT_PRODUCER_EMPTY))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = lane_addr + blk * C::PCOLS;
                if (CIN == 4) {
                    tmem_st32(ta, wd);
                    tmem_st16(ta + 32, wd + 32);
                    tmem_st8(ta + 48, wd + 48);
                } else {
                    tmem_st16(ta, wd);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[blk]);
            }
            if (++hs == C::HS) {
                hs = 0;
                hph ^= 1;
            }
            aph ^= 1;
        }
    } else if (warp < 18) {
        // ---------------- epilogue warps 10..17: two per lane quarter, each taking
        // 16 of every 32 channels (when BN is 16, the second warp of a quarter idles)
        const int q = warp & 3;
        const int half = (warp - 10) >> 2;
        const int lp = 2 * q + (lane >> 4), v = lane & 15, dw = v & 1;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
        constexpr int NPASS = (BN + 31) / 32;
        // bias of the 8 channels this lane finalises in each pass
        float bias[NPASS][8];
#pragma unroll
        for (int ps = 0; ps < NPASS; ++ps)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int co = co0 + 32 * ps + 16 * half + 8 * dw + i;
                bias[ps][i] = (EPI == EPI_POOL && p.ea.bias != nullptr && co < p.Cout) ? __ldg(p.ea.bias + co) : 0.f;
            }
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
            const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
            // each warp waits on its own (no barrier across the eight warps: the
            // slowest warp of a tile would hold the others and the accumulator's
            // release); a warp that gives up raises the abort flag for all
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&tfull[acc], use & 1, abort_flag, p.wait_ns, p.status, WAIT_EPI_TMEM_FULL)))
                break;
            tc_fence_after();
            const SmallTile t = small_decode(p, tile);
            const uint32_t acol = lane_addr + acc * C::ACC_COLS;
            bool released = false;
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
                const int c = 32 * ps + 16 * half;  // first of the warp's 16 accumulator columns
                if (c >= BN) break;
                if (EPI == EPI_POOL || EPI == EPI_AVG) {
                    // per channel: first maximum over the lane's four (plane, line) values,
                    // in the window's scan order (code dd*4 + dh*2 + dw)
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    float m[16];
                    int k[16];
                    tmem_ld16(acol + 0 * BN + c, r0);
                    tmem_ld16(acol + 1 * BN + c, r1);
                    tmem_ld16(acol + 2 * BN + c, r2);
                    tmem_ld16(acol + 3 * BN + c, r3);
                    tmem_ld_wait();
                    if (ps == NPASS - 1 || c + 32 >= BN) {
                        // the tile's accumulator is in registers: hand it back to the MMA
                        // before the pooling arithmetic and the stores
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[acc]);
                        released = true;
                    }
                    float y[8];
                    uint32_t codes[2] = {0u, 0u};
                    if (EPI == EPI_AVG) {
                        // average of the activated window: the lane's four (plane, line)
                        // values, then the partner lane's (the w neighbour); code = the
                        // window's sign mask, bit dd*4 + dh*2 + dw
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) {
                            const int co = co0 + c + cc;
                            const float b = (p.ea.bias != nullptr && co < p.Cout) ? __ldg(p.ea.bias + co) : 0.f;
                            const float s0 = __uint_as_float(r0[cc]) + b, s1 = __uint_as_float(r1[cc]) + b;
                            const float s2 = __uint_as_float(r2[cc]) + b, s3 = __uint_as_float(r3[cc]) + b;
                            m[cc] = (lrelu(s0, p.ea.slope) + lrelu(s1, p.ea.slope)) +
                                    (lrelu(s2, p.ea.slope) + lrelu(s3, p.ea.slope));
                            k[cc] = ((s0 > 0.f ? 1 : 0) << dw) | ((s1 > 0.f ? 1 : 0) << (2 + dw)) |
                                    ((s2 > 0.f ? 1 : 0) << (4 + dw)) | ((s3 > 0.f ? 1 : 0) << (6 + dw));
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float kv = dw ? m[8 + i] : m[i];
                            const int kk = dw ? k[8 + i] : k[i];
                            const float ov = __shfl_xor_sync(0xffffffffu, dw ? m[i] : m[8 + i], 1);
                            const int ok2 = __shfl_xor_sync(0xffffffffu, dw ? k[i] : k[8 + i], 1);
                            y[i] = (kv + ov) * 0.125f;
                            codes[i >> 2] |= (uint32_t)(kk | ok2) << (8 * (i & 3));
                        }
                    } else {
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        const float v0 = __uint_as_float(r0[cc]), v1 = __uint_as_float(r1[cc]);
                        const float v2 = __uint_as_float(r2[cc]), v3 = __uint_as_float(r3[cc]);
                        m[cc] = v0;
                        k[cc] = dw;
                        if (v1 > m[cc]) {
                            m[cc] = v1;
                            k[cc] = 2 + dw;
                        }
                        if (v2 > m[cc]) {
                            m[cc] = v2;
                            k[cc] = 4 + dw;
                        }
                        if (v3 > m[cc]) {
                            m[cc] = v3;
                            k[cc] = 6 + dw;
                        }
                    }
                    // lane pair (dw = 0, 1): each keeps 8 channels and takes the
                    // partner's values for them; larger value wins, ties keep the
                    // smaller code
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float kv = dw ? m[8 + i] : m[i];
                        int kk = dw ? k[8 + i] : k[i];
                        const float sv = dw ? m[i] : m[8 + i];
                        const int sk = dw ? k[i] : k[8 + i];
                        const float ov = __shfl_xor_sync(0xffffffffu, sv, 1);
                        const int ok2 = __shfl_xor_sync(0xffffffffu, sk, 1);
                        if (ov > kv || (ov == kv && ok2 < kk)) {
                            kv = ov;
                            kk = ok2;
                        }
                        const float s = kv + bias[ps][i];
                        y[i] = s > 0.f ? s : p.ea.slope * s;
                        codes[i >> 2] |= (uint32_t)kk << (8 * (i & 3));
                    }
                    }
                    const int D2 = p.D >> 1, H2 = p.H >> 1, W2 = p.W >> 1;
                    const int pd = t.d0 >> 1, ph = (t.h0 >> 1) + lp, pw = (t.w0 + v) >> 1;
                    if (pd < D2 && ph < H2 && pw < W2 && co0 + c + 8 * dw < p.Cout) {
                        const int64_t po =
                            ((((int64_t)t.n * D2 + pd) * H2 + ph) * W2 + pw) * p.Cout + co0 + c + 8 * dw;
                        *reinterpret_cast<uint4*>(p.ea.y + po) =
                            make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                       pack_bf16x2(y[6], y[7]));
                        if (p.ea.idx) *reinterpret_cast<uint2*>(p.ea.idx + po) = make_uint2(codes[0], codes[1]);
                    }
                } else {
#pragma unroll 1
                    for (int blk = 0; blk < SC_BLOCKS; ++blk) {
                        uint32_t r[32];
                        tmem_ld16(acol + blk * BN + c, r);
                        tmem_ld_wait();
                        const int d = t.d0 + (blk >> 1), h = t.h0 + 2 * lp + (blk & 1), w = t.w0 + v;
                        if (d >= p.D || h >= p.H || w >= p.W) continue;
                        const int64_t o = ((((int64_t)t.n * p.D + d) * p.H + h) * p.W + w) * p.Cout + co0 + c;
                        if (EPI == EPI_ACT) {  // unpooled block: bias + leaky ReLU
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const int co = co0 + c + q;
                                const float b = (p.ea.bias != nullptr && co < p.Cout) ? __ldg(p.ea.bias + co) : 0.f;
                                r[q] = __float_as_uint(lrelu(__uint_as_float(r[q]) + b, p.ea.slope));
                            }
                        }
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8) {
                            if (co0 + c + 8 * q8 >= p.Cout) break;
                            *reinterpret_cast<uint4*>(p.ea.y + o + 8 * q8) = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * q8 + 0]), __uint_as_float(r[8 * q8 + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * q8 + 2]), __uint_as_float(r[8 * q8 + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * q8 + 4]), __uint_as_float(r[8 * q8 + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * q8 + 6]), __uint_as_float(r[8 * q8 + 7])));
                        }
                    }
                }
            }
            if (!released) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
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

bool make_halo_map(CUtensorMap* m, const uint16_t* x, int n, int d, int h, int w, int cin, int tw, int th, int td) {
    const uint64_t dims[4] = {(uint64_t)w * cin, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t str[3] = {(uint64_t)w * cin * 2, (uint64_t)h * w * cin * 2, (uint64_t)d * h * w * cin * 2};
    const uint32_t box[4] = {(uint32_t)(halo_line_voxels(tw, cin) * cin), (uint32_t)(th + 2), (uint32_t)(td + 2), 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int CIN, int BN, int EPI>
static cf_status run_smallc(const LaunchCtx& ctx, const HaloParams& hp, const uint16_t* x, const uint16_t* wk) {
    using C = SmallTmCfg<CIN, BN, EPI>;
    static_assert(halo_bytes(SC_W, SC_H, SC_D, CIN) == C::HALO_BYTES, "halo box and ring stage disagree");
    CUtensorMap th;
    if (!make_halo_map(&th, x, hp.N, hp.D, hp.H, hp.W, CIN, SC_W, SC_H, SC_D)) return CF_ERR_CUDA;
    SmallTmParams sp{hp, wk};
    auto kern = conv_smallc_kernel<CIN, BN, EPI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    int grid = grid_for(kern, C::SMEM, 608, ctx.num_sms, hp.num_tiles, C::TMEM_COLS);
    grid = std::max(hp.n_ntiles, grid / hp.n_ntiles * hp.n_ntiles);  // each CTA keeps one N tile
    kern<<<grid, 608, C::SMEM, ctx.stream>>>(th, sp);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int CIN, int BN>
static cf_status smallc_epi(const LaunchCtx& ctx, const HaloParams& hp, const uint16_t* x, const uint16_t* wk,
                            int epi) {
    if (epi == EPI_POOL) return run_smallc<CIN, BN, EPI_POOL>(ctx, hp, x, wk);
    if (epi == EPI_AVG) return run_smallc<CIN, BN, EPI_AVG>(ctx, hp, x, wk);
    if (epi == EPI_ACT) return run_smallc<CIN, BN, EPI_ACT>(ctx, hp, x, wk);
    if (epi == EPI_PLAIN) return run_smallc<CIN, BN, EPI_PLAIN>(ctx, hp, x, wk);
    return CF_ERR_UNSUPPORTED;
}

cf_status launch_conv_smallc(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_in, int c_out,
                             const uint16_t* x, const uint16_t* wk, int epi, uint16_t* y, uint8_t* idx,
                             const float* bias, float slope, int pool_kind, int act) {
    if (c_out % 8 != 0 || c_out > 256) return CF_ERR_UNSUPPORTED;
    if (c_in != 1 && c_in != 4) return CF_ERR_UNSUPPORTED;
    if ((w * c_in) % 8 != 0) return CF_ERR_UNSUPPORTED;  // halo rows must be 16-byte multiples
    // N tile: c_out rounded up to 16, at most 64 (four accumulators of a tile
    // and the four A blocks share the 512 tensor-memory columns)
    const int bn = c_out <= 64 ? (c_out + 15) / 16 * 16 : 64;
    HaloParams hp;
    hp.N = (int)n;
    hp.D = (int)d;
    hp.H = (int)h;
    hp.W = (int)w;
    hp.Cin = c_in;
    hp.Cout = c_out;
    hp.tiles_w = (int)((w + SC_W - 1) / SC_W);
    hp.tiles_h = (int)((h + SC_H - 1) / SC_H);
    hp.tiles_d = (int)((d + SC_D - 1) / SC_D);
    hp.n_ntiles = (c_out + bn - 1) / bn;
    hp.num_tiles = (int)(n * hp.tiles_d * hp.tiles_h * hp.tiles_w * hp.n_ntiles);
    set_tile_dividers(hp);
    hp.n_chunks = 1;
    hp.ea = EpiArgs{y, idx, bias, nullptr, slope};
    if (epi == EPI_POOL && pool_kind == 1) epi = EPI_AVG;
    if (epi == EPI_PLAIN && act) epi = EPI_ACT;
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
        default: return CF_ERR_UNSUPPORTED;
    }
#undef CF_SC_CASE
}

}  // namespace cf
