// conv_wgrad_smallc.cu -- backward-weight conv of the small-channel first
// layer (c_in = 1 or 4), optionally with the max-pool backward fused in.
//
// (CosmoFlow page, section III-C "backward weights".)
//   dW[co, t, ci] = sum_{n,v} dZ[n,v,co] * X[n, v + t - 1, ci]
// GEMM view: M = (t, ci) = 27*c_in rows padded to 128, N = co (the whole
// c_out), K = voxels, in boxes of 2 planes x 4 lines x 16 voxels (128).  Both
// operands are MN-major in shared memory:
//   A[(t,ci), v]: the im2col rows of the box (row = voxel, 128 (t,ci) columns
//                 in two SW128 atoms), gathered from the box's input halo;
//   B[co, v]    : dZ rows of the box.
// Routed form: the layer's max-pool keeps one voxel per window and channel,
// so dZ[v, co] = dYpre[p(v), co] where idx[p(v), co] is v's position in its
// window p(v), else 0.  Given the pooled gradient and the argmax codes, the
// kernel expands the box's dZ rows in shared memory instead of reading a dense
// dZ (eight times larger) from memory.
//
// Roles (480 threads):
//   warp 0      : TMA per box into a deep load ring: the input halo (4 planes x
//                 6 lines x (16 + 2*margin) voxels, zero outside the volume),
//                 and the dZ rows (dense) or the pooled gradient + codes (routed);
//   warps 2..9  : builders, two groups of four warps taking alternate boxes;
//                 thread r builds row r (voxel (r/64, r/16 % 4, r % 16)) of the
//                 box's A tile in a short build ring: 27 8-byte loads from the
//                 halo (a half-warp reads 16 consecutive voxels of one line: no
//                 bank conflicts) stored as 14 swizzled 16-byte chunks, and in
//                 the routed form its dZ row;
//   warps 1, 14 : MMA issuers, one per builder group (alternate boxes), 8
//                 tcgen05.mma (K = 16 voxels) per box into the issuer's own
//                 accumulator (two per issuer when tensor memory allows);
//   warps 10..13: at the end of a unit of boxes, the sum of the two issuers'
//                 accumulators to the split-K partials.
// The load ring (as many boxes as shared memory leaves, up to 12) hides the
// TMA latency, the build ring the MMA-completion latency; each box's load
// stage is released by the MMA commit.
#include <algorithm>

#include "smallc_common.cuh"
#include "wgrad_common.cuh"

namespace cf {

constexpr int WS_VW = 16, WS_VH = 4, WS_VD = 2;  // voxel box (K block); wgrad_geom uses the same

template <int CIN, int BN, int SUBB, bool ROUTED>
struct WsCfg {
    static constexpr uint32_t A_BYTES = 128 * 128 * 2;  // [2 atoms][128 voxels][64 (t,ci)], SW128
    static constexpr uint32_t B_BYTES = BN * 128 * 2;   // BN/SUBB sub-blocks [128 voxels][SUBB co]
    static constexpr uint32_t B_SUB_BYTES = 128 * SUBB * 2;
    static constexpr int MARGIN = 16 / (2 * CIN);       // halo voxels left of the box (16-byte start)
    static constexpr int PITCH = (WS_VW + 2 * MARGIN) * CIN * 2;          // bytes per halo line
    static constexpr int HALO_BYTES = (WS_VD + 2) * (WS_VH + 2) * PITCH;  // 3840 or 1536
    static constexpr int PBOX = (WS_VW / 2) * (WS_VH / 2);                // pooled voxels per box
    static constexpr uint32_t DY_BYTES = ROUTED ? PBOX * BN * 2 : 0;
    static constexpr uint32_t IX_BYTES = ROUTED ? PBOX * BN : 0;
    // load stage: [halo][dense dZ B | pooled gradient][codes]; build stage: [A][routed dZ B]
    static constexpr uint32_t L_B = (HALO_BYTES + 1023) / 1024 * 1024;   // dense B or pooled gradient
    static constexpr uint32_t L_IX = L_B + (ROUTED ? (DY_BYTES + 1023) / 1024 * 1024 : B_BYTES);
    static constexpr uint32_t LOAD_BYTES = L_IX + (IX_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t BUILD_BYTES = A_BYTES + (ROUTED ? B_BYTES : 0);
    static constexpr uint32_t TX_BYTES = HALO_BYTES + (ROUTED ? DY_BYTES + IX_BYTES : B_BYTES);
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t BUDGET = 227 * 1024 - 1024 - BAR_BYTES;
    // Both rings have an even number of stages: box lb uses stage lb % S, so
    // every stage belongs to one builder group and one issuer (lb % 2), which
    // wait on each of its phases in turn.  (With an odd count a party that
    // skips the other parity's boxes could wait two phases ahead and take the
    // stale completed phase of the same parity for its own.)
    static constexpr int BS = (4 * BUILD_BYTES + 2 * LOAD_BYTES <= BUDGET) ? 4 : 2;  // build stages
    static constexpr int LS_RAW = (int)((BUDGET - BS * BUILD_BYTES) / LOAD_BYTES);
    static constexpr int LS = (LS_RAW > 12 ? 12 : LS_RAW) & ~1;                   // load stages
    static constexpr uint32_t SMEM = 1024 + BS * BUILD_BYTES + LS * LOAD_BYTES + BAR_BYTES;
    static constexpr uint32_t SWZ_B = SUBB == 64 ? SWZ_128B : (SUBB == 32 ? SWZ_64B : SWZ_32B);
    static constexpr uint32_t SBO_B = 8 * SUBB * 2;
    static constexpr uint32_t ACC_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr int NACC = 4 * ACC_COLS <= 512 ? 2 : 1;  // accumulators per issuer
    static constexpr uint32_t TMEM_COLS = 2 * NACC * ACC_COLS;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN, 1, 1);
    static_assert(LS >= 2, "not enough shared memory");
    static_assert(BS % 2 == 0 && LS % 2 == 0, "stages must alternate between the two box parities");
    static_assert(8 * (2 * LS + 2 * BS + 2 * NACC + 2) + 16 <= (int)BAR_BYTES, "barrier area");
};

struct WsParams {
    WgradGeom g;
    float* part;
    int* status;
    uint64_t wait_ns;
};

// 16-byte chunk index XOR of the MN-major dZ sub-block (SUBB channels per
// row) for row r: the TMA swizzle of that row width.
template <int SUBB>
__device__ __forceinline__ int dz_chunk_xor(int r) {
    return SUBB == 64 ? (r & 7) : (SUBB == 32 ? ((r >> 1) & 3) : ((r >> 2) & 1));
}

// Box bookkeeping shared by the roles: each walks its CTA's units in order
// and the boxes of each unit in order; lb counts the CTA's boxes.
template <int CIN, int BN, int SUBB, bool ROUTED>
__global__ void __launch_bounds__(480, 1)
    wgrad_smallc_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmG,
                        const __grid_constant__ CUtensorMap tmI, const WsParams p) {
    using C = WsCfg<CIN, BN, SUBB, ROUTED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* bring = smem;                           // build ring
    uint8_t* lring = smem + C::BS * C::BUILD_BYTES;  // load ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(lring + C::LS * C::LOAD_BYTES);
    uint64_t* lfull = bars;               // TMA of a load stage landed (tx)
    uint64_t* lempty = lfull + C::LS;     // MMAs reading (from) the load stage done
    uint64_t* bfull = lempty + C::LS;     // build stage written (4 builder warps)
    uint64_t* bempty = bfull + C::BS;     // MMAs of the build stage done
    uint64_t* tfull = bempty + C::BS;     // [NACC] both issuers' unit accumulators complete
    uint64_t* tempty = tfull + C::NACC;   // [NACC] accumulators read by the epilogue
    uint64_t* drain = tempty + C::NACC;   // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WgradGeom& g = p.g;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::LS; ++s) {
            mbar_init(&lfull[s], 1);
            mbar_init(&lempty[s], 1);
        }
        for (int s = 0; s < C::BS; ++s) {
            mbar_init(&bfull[s], 4);
            mbar_init(&bempty[s], 1);
        }
        for (int a = 0; a < C::NACC; ++a) {
            mbar_init(&tfull[a], 2);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmG);
        if (ROUTED) tma_prefetch_desc(&tmI);
    }
    // the A columns the builders never write ((t,ci) >= 8 * chunks written) stay zero
    for (int e = threadIdx.x; e < C::BS * (int)(C::A_BYTES / 16); e += blockDim.x) {
        const int s = e / (C::A_BYTES / 16), o = e % (C::A_BYTES / 16);
        *reinterpret_cast<uint4*>(bring + s * C::BUILD_BYTES + o * 16) = make_uint4(0u, 0u, 0u, 0u);
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
            // ---------------- TMA producer
            int ls = 0;
            uint32_t lph = 0, issued = 0, par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x) {
                const int64_t b0 = (int64_t)u * g.boxes_per_split;
                const int64_t b1 = std::min<int64_t>(b0 + g.boxes_per_split, g.total_boxes);
                BoxCursor cur;
                cur.init(g, b0);
                for (int64_t b = b0; b < b1; ++b, cur.next(g)) {
                    const int n = cur.n, d0 = cur.bd * WS_VD, h0 = cur.bh * WS_VH, w0 = cur.bw * WS_VW;
                    if (!mbar_wait(&lempty[ls], lph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = lring + ls * C::LOAD_BYTES;
                    mbar_arrive_expect_tx(&lfull[ls], C::TX_BYTES);
                    load_halo<CIN>(st, &tmH, &lfull[ls], n, d0, h0, w0);
                    if (ROUTED) {
                        tma_load_5d(st + C::L_B, &tmG, &lfull[ls], 0, w0 >> 1, h0 >> 1, d0 >> 1, n);
                        tma_load_5d(st + C::L_IX, &tmI, &lfull[ls], 0, w0 >> 1, h0 >> 1, d0 >> 1, n);
                    } else {
#pragma unroll
                        for (int s = 0; s < BN / SUBB; ++s)
                            tma_load_5d(st + C::L_B + s * C::B_SUB_BYTES, &tmG, &lfull[ls], s * SUBB, w0, h0, d0,
                                        n);
                    }
                    issued |= 1u << ls;
                    par = (par & ~(1u << ls)) | (lph << ls);
                    if (++ls == C::LS) {
                        ls = 0;
                        lph ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < C::LS; ++s)
                    if (issued & (1u << s)) mbar_wait_timed(&lfull[s], (par >> s) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 14) {
        if (lane == 0) {
            // ---------------- MMA issuer mi: the boxes with lb = mi (mod 2)
            const int mi = warp == 1 ? 0 : 1;
            int ls = 0, bs = 0;
            uint32_t lph = 0, bph = 0, lb = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x, ++local) {
                const int64_t b0 = (int64_t)u * g.boxes_per_split;
                const int64_t b1 = std::min<int64_t>(b0 + g.boxes_per_split, g.total_boxes);
                const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
                const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
                if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (mi * C::NACC + acc) * C::ACC_COLS;
                bool first = true;
                for (int64_t b = b0; b < b1; ++b, ++lb) {
                    if ((int)(lb & 1) == mi) {
                        if (!mbar_wait(&bfull[bs], bph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        if (!ROUTED &&
                            !mbar_wait(&lfull[ls], lph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(bring + bs * C::BUILD_BYTES);
                        const uint32_t b_addr =
                            ROUTED ? a_addr + C::A_BYTES : smem_u32(lring + ls * C::LOAD_BYTES + C::L_B);
#pragma unroll
                        for (int k = 0; k < 128 / 16; ++k) {
                            const uint64_t ad = sdesc(a_addr + k * 16 * 128, 128 * 128, 1024, SWZ_128B);
                            const uint64_t bd =
                                sdesc(b_addr + k * 16 * SUBB * 2, C::B_SUB_BYTES, C::SBO_B, C::SWZ_B);
                            umma_bf16(d_tmem, ad, bd, C::IDESC, first ? 0u : 1u);
                            first = false;
                        }
                        umma_commit(&bempty[bs]);
                        umma_commit(&lempty[ls]);
                    }
                    if (++ls == C::LS) {
                        ls = 0;
                        lph ^= 1;
                    }
                    if (++bs == C::BS) {
                        bs = 0;
                        bph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
            }
            if (!ok) {
                umma_commit(&drain[mi]);
                mbar_wait_timed(&drain[mi], 0, p.wait_ns);
            }
        }
    } else if (warp < 10) {
        // ---------------- builders: group grp takes the boxes with lb = grp (mod 2)
        const int grp = (warp - 2) >> 2;
        const int r = (warp - 2 - 4 * grp) * 32 + lane;
        const int i = r >> 6, j = (r >> 4) & 3, l = r & 15;
        int ls = 0, bs = 0;
        uint32_t lph = 0, bph = 0, lb = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < g.num_units && ok; u += gridDim.x) {
            const int64_t b0 = (int64_t)u * g.boxes_per_split;
            const int64_t b1 = std::min<int64_t>(b0 + g.boxes_per_split, g.total_boxes);
            for (int64_t b = b0; b < b1; ++b, ++lb) {
                if ((int)(lb & 1) == grp) {
                    // all lanes wait; the warp leaves together
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&lfull[ls], lph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL) &&
                                        mbar_wait(&bempty[bs], bph ^ 1, abort_flag, p.wait_ns, p.status,
                                                  WAIT_PRODUCER_EMPTY))) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = bring + bs * C::BUILD_BYTES;
                    const uint8_t* ld = lring + ls * C::LOAD_BYTES;
                    if (CIN == 4) {
                        // 27 independent 8-byte loads (warp shuffles for the w neighbours
                        // measured slower: shuffle throughput, not bank bandwidth, binds)
                        const uint8_t* base = ld + (i * (WS_VH + 2) + j) * C::PITCH + (l + C::MARGIN - 1) * 8;
                        uint32_t wd[56];
#pragma unroll
                        for (int kd = 0; kd < 3; ++kd)
#pragma unroll
                            for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                                for (int kw = 0; kw < 3; ++kw) {
                                    const uint2 x = *reinterpret_cast<const uint2*>(
                                        base + (kd * (WS_VH + 2) + kh) * C::PITCH + kw * 8);
                                    const int t = kd * 9 + kh * 3 + kw;
                                    wd[2 * t] = x.x;
                                    wd[2 * t + 1] = x.y;
                                }
                        wd[54] = wd[55] = 0u;
#pragma unroll
                        for (int c = 0; c < 14; ++c)
                            *reinterpret_cast<uint4*>(st + (c >> 3) * (128 * 128) + r * 128 +
                                                      (((c & 7) ^ (r & 7)) << 4)) =
                                make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]);
                    } else {
                        uint32_t e[32];
#pragma unroll
                        for (int t = 27; t < 32; ++t) e[t] = 0u;
#pragma unroll
                        for (int kd = 0; kd < 3; ++kd)
#pragma unroll
                            for (int kh = 0; kh < 3; ++kh) {
                                const uint16_t* line = reinterpret_cast<const uint16_t*>(
                                    ld + ((i + kd) * (WS_VH + 2) + j + kh) * C::PITCH);
#pragma unroll
                                for (int kw = 0; kw < 3; ++kw)
                                    e[kd * 9 + kh * 3 + kw] = line[l + C::MARGIN - 1 + kw];
                            }
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(st + r * 128 + ((c ^ (r & 7)) << 4)) =
                                make_uint4(e[8 * c] | (e[8 * c + 1] << 16), e[8 * c + 2] | (e[8 * c + 3] << 16),
                                           e[8 * c + 4] | (e[8 * c + 5] << 16), e[8 * c + 6] | (e[8 * c + 7] << 16));
                    }
                    if (ROUTED) {
                        // dZ rows of the box: thread (pooled voxel pp, w parity hw, 8-channel
                        // chunks c8, c8 + 4, ...) reads its pooled gradient and codes once and
                        // writes the chunk of the four window voxels with that w parity: the
                        // gradient where the window's argmax code is the voxel's, else zero
                        const int pp = r >> 3, hw = (r >> 2) & 1;
                        const uint8_t* dyrow = ld + C::L_B + pp * (BN * 2);
                        const uint8_t* ixrow = ld + C::L_IX + pp * BN;
                        const int vrow = (pp >> 3) * 2 * WS_VW + 2 * (pp & 7) + hw;  // window voxel (0, 0, hw)
#pragma unroll
                        for (int c8 = r & 3; c8 < BN / 8; c8 += 4) {
                            const uint4 dv = *reinterpret_cast<const uint4*>(dyrow + c8 * 16);
                            const uint2 iv = *reinterpret_cast<const uint2*>(ixrow + c8 * 8);
                            const int sb = (c8 * 8) / SUBB, cc = c8 % (SUBB / 8);
#pragma unroll
                            for (int dd = 0; dd < 2; ++dd)
#pragma unroll
                                for (int dh = 0; dh < 2; ++dh) {
                                    const int rr = vrow + dd * (WS_VH * WS_VW) + dh * WS_VW;
                                    const uint32_t code4 = (uint32_t)(dd * 4 + dh * 2 + hw) * 0x01010101u;
                                    uint32_t m0, m1, m2, m3;
                                    code_mismatch(iv.x, code4, m0, m1);
                                    code_mismatch(iv.y, code4, m2, m3);
                                    *reinterpret_cast<uint4*>(st + C::A_BYTES + sb * C::B_SUB_BYTES + rr * (SUBB * 2) +
                                                              ((cc ^ dz_chunk_xor<SUBB>(rr)) << 4)) =
                                        make_uint4(dv.x & ~m0, dv.y & ~m1, dv.z & ~m2, dv.w & ~m3);
                                }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bfull[bs]);
                }
                if (++ls == C::LS) {
                    ls = 0;
                    lph ^= 1;
                }
                if (++bs == C::BS) {
                    bs = 0;
                    bph ^= 1;
                }
            }
        }
    } else {
        // ---------------- epilogue warps 10..13: dW rows (t,ci) = sum of the issuers'
        // accumulators (an issuer without a box in the unit contributes nothing)
        const int q = warp & 3;
        const int et = threadIdx.x - 320;
        const int row = q * 32 + lane;
        const int KK = 27 * g.Cin;
        uint32_t local = 0, lb = 0;
        for (int u = blockIdx.x; u < g.num_units; u += gridDim.x, ++local) {
            const int64_t b0 = (int64_t)u * g.boxes_per_split;
            const int64_t nb = std::min<int64_t>(b0 + g.boxes_per_split, g.total_boxes) - b0;
            const bool has0 = nb >= 2 || (lb & 1) == 0, has1 = nb >= 2 || (lb & 1) == 1;
            lb += (uint32_t)nb;
            const uint32_t acc = C::NACC == 2 ? (local & 1) : 0u;
            const uint32_t use = C::NACC == 2 ? (local >> 1) : local;
            if (!epi_wait(&tfull[acc], use & 1, et, epi_flag, abort_flag, p.wait_ns, p.status)) break;
            tc_fence_after();
            const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
            const uint32_t a0 = lane_addr + acc * C::ACC_COLS, a1 = lane_addr + (C::NACC + acc) * C::ACC_COLS;
            float* base = p.part + (int64_t)u * g.Cout * KK + row;
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t v0[32], v1[32];
                tmem_ld16(a0 + c, v0);
                tmem_ld16(a1 + c, v1);
                tmem_ld_wait();
                if (row < KK) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float s = (has0 ? __uint_as_float(v0[k]) : 0.f) + (has1 ? __uint_as_float(v1[k]) : 0.f);
                        if (c + k < g.Cout) base[(int64_t)(c + k) * KK] = s;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
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

// 5-D map over an NDHWC tensor [n][d][h][w][c] of `esize`-byte elements with
// box (box_c, bw, bh, bd, 1) and the swizzle of box_c channels (none if 0).
static bool make_box_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int64_t n, int64_t d,
                         int64_t h, int64_t w, int c, int box_c, int bw, int bh, int bd, bool swizzle) {
    const uint64_t dims[5] = {(uint64_t)c, (uint64_t)w, (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t str[4] = {(uint64_t)c * esize, (uint64_t)w * c * esize, (uint64_t)h * w * c * esize,
                             (uint64_t)d * h * w * c * esize};
    const uint32_t box[5] = {(uint32_t)box_c, (uint32_t)bw, (uint32_t)bh, (uint32_t)bd, 1u};
    CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle)
        swz = box_c * esize == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
              : box_c * esize == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                    : CU_TENSOR_MAP_SWIZZLE_32B;
    return encode_tmap(m, dt, 5, base, dims, str, box, swz);
}

template <int CIN, int BN, bool ROUTED>
static cf_status run_wgrad_smallc(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                                  const uint8_t* idx, float* part) {
    constexpr int SUBB = BN >= 64 ? 64 : BN;
    using C = WsCfg<CIN, BN, SUBB, ROUTED>;
    static_assert(halo_bytes(WS_VW, WS_VH, WS_VD, CIN) == C::HALO_BYTES, "halo box and stage disagree");
    CUtensorMap th, tg, ti;
    if (!make_halo_map(&th, x, g.N, g.D, g.H, g.W, CIN, WS_VW, WS_VH, WS_VD)) return CF_ERR_CUDA;
    if (ROUTED) {
        if (!make_box_map(&tg, dz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.N, g.D / 2, g.H / 2, g.W / 2, g.Cout, BN,
                          WS_VW / 2, WS_VH / 2, WS_VD / 2, false))
            return CF_ERR_CUDA;
        if (!make_box_map(&ti, idx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.N, g.D / 2, g.H / 2, g.W / 2, g.Cout, BN,
                          WS_VW / 2, WS_VH / 2, WS_VD / 2, false))
            return CF_ERR_CUDA;
    } else {
        if (!make_box_map(&tg, dz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.N, g.D, g.H, g.W, g.Cout, SUBB, WS_VW,
                          WS_VH, WS_VD, true))
            return CF_ERR_CUDA;
        ti = tg;  // unused
    }
    WsParams p{g, part, ctx.status, ctx.wait_ns};
    auto kern = wgrad_smallc_kernel<CIN, BN, SUBB, ROUTED>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = std::max(1, std::min(g.num_units, ctx.num_sms));
    kern<<<grid, 480, C::SMEM, ctx.stream>>>(th, tg, ti, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

template <int CIN, int BN>
static cf_status wgrad_smallc_route(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                                    const uint8_t* idx, float* part) {
    if (idx) return run_wgrad_smallc<CIN, BN, true>(ctx, g, x, dz, idx, part);
    return run_wgrad_smallc<CIN, BN, false>(ctx, g, x, dz, nullptr, part);
}

template <int CIN>
static cf_status wgrad_smallc_cin(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                                  const uint8_t* idx, float* part) {
    switch (g.bn) {  // c_out rounded up to a compiled width (extra channels read as zero)
        case 16: return wgrad_smallc_route<CIN, 16>(ctx, g, x, dz, idx, part);
        case 32: return wgrad_smallc_route<CIN, 32>(ctx, g, x, dz, idx, part);
        case 64: return wgrad_smallc_route<CIN, 64>(ctx, g, x, dz, idx, part);
        case 128: return wgrad_smallc_route<CIN, 128>(ctx, g, x, dz, idx, part);
        case 192: return wgrad_smallc_route<CIN, 192>(ctx, g, x, dz, idx, part);
        case 256: return wgrad_smallc_route<CIN, 256>(ctx, g, x, dz, idx, part);
        default: return CF_ERR_UNSUPPORTED;
    }
}

cf_status launch_wgrad_smallc(const LaunchCtx& ctx, const WgradGeom& g, const uint16_t* x, const uint16_t* dz,
                              const uint8_t* idx, float* part) {
    if (g.vw != WS_VW || g.vh != WS_VH || g.vd != WS_VD || g.n_mblocks != 1 || g.n_ntiles != 1)
        return CF_ERR_UNSUPPORTED;
    if (idx && ((g.D | g.H | g.W) & 1)) return CF_ERR_UNSUPPORTED;
    if (g.Cin == 4) return wgrad_smallc_cin<4>(ctx, g, x, dz, idx, part);
    if (g.Cin == 1) return wgrad_smallc_cin<1>(ctx, g, x, dz, idx, part);
    return CF_ERR_UNSUPPORTED;
}

}  // namespace cf
