// conv_wgrad_quad.cu -- backward-weight conv of the CosmoFlow first layer
// (c_in = 4, c_out = 32) with the max-pool backward fused in, as the weight
// gradient of the quad-row forward (conv_quad.cu).
//
// (CosmoFlow page, section III-C "backward weights".)
//   dW[co, t, ci] = sum_{n,v} dZ[n,v,co] * X[n, v + t - 1, ci]
//
// The quad-row forward computes, per tap pair (kd, kh) and half hf,
//   Z[r, (f, co)] += sum_k A_{kd,kh,hf}[r, k] * B_{kd,kh,hf}[(f, co), k]
// with row r a quad of voxels 4r .. 4r+3, phase f the voxel 4r + f, and K slot
// k = (voxel slot s, ci) of the input rows E / O (even / odd voxel pairs).
// Its weight gradient is the transposed product
//   G_{kd,hf}[(f, co), (kh, k)] = sum_r dZ[4r + f, co] * A_{kd,kh,hf}[r, k]
// and dW[co, kd, kh, kw, ci] = sum_f G[(f, co), (kh, (s, ci))] with
// s = f + kw - 1 (one K slot per phase and tap).  Here:
//   A operand (tensor memory): dZ arranged as M = (phase f, co) = 128 lanes by
//     K = rows of the tile; built per tile by four builder warps (warp f, lane
//     co) from the pooled gradient and the argmax codes: dZ at voxel v is the
//     gradient of v's window where the window's code is v's position, else 0.
//   B operand (shared memory, MN-major, no swizzle): the E / O input rows,
//     N = (kh, E/O, two voxels x 4 channels), K = 16 rows (2 lines x 8 quads)
//     per MMA.  The input lines arrive as one TMA box of plain lines (288-byte
//     rows: a box of 16-byte E / O rows measured TMA-bound) and the builder
//     warps copy their pairs into the E and O rows, in an order that hits
//     every shared-memory bank once per eight pairs.
// The builders store each input line as [E row | O row], so that one MMA
// takes the pairs E[r] and O[r] (voxel slots 0-1 and -2..-1, the low half) or
// E[r+1] and O[r+1] (slots 4-5 and 2-3, the high half) of the three lines kh:
// N = 3 kh x 2 x 8 = 48, the N groups one row (144 bytes) apart.  Per K step 6
// MMAs of 128 x 48 x 16 (3 kd x 2 halves), one accumulator of 48 columns
// each (288 of the 512 tensor-memory columns; columns 288.. hold one dZ tile
// per builder group).  Three issuer threads take one kd each (measured: N = 32
// MMAs with A in tensor memory run at ~27 cycles, so fewer wider MMAs pay).
//
// Tile: 1 plane x 16 lines x 32 voxels (128 rows).  Each CTA sums a
// contiguous range of tiles and writes, per phase, its 32 x 108 partial dW
// (phase-major split-K partials, summed afterwards in a fixed order).
//
// Roles (512 threads): warp 0 TMA producer; warps 1, 2, 3 MMA issuers
// (kd = 0, 1, 2); warps 4..15 three builder groups of four warps.  Group g
// takes every third tile (g, g + 3, ...), with its own dZ slot and E / O
// buffer, so three tiles are built at once: one group building a tile (a
// chain of waits, shared-memory loads and tensor-memory stores) was the
// bound with all eight builder warps on the same tile.  Warp f of a group
// builds phase f (lane = channel co) over all 16 lines; after the last tile
// group 0 runs the epilogue.
#include <algorithm>

#include "conv_common.cuh"

namespace cf {

constexpr int WQ_W = 32, WQ_H = 16;                 // tile (one plane)
constexpr int WQ_QUADS = WQ_W / 4 + 1;              // E / O entries per line (9)
constexpr int WQ_LINES = WQ_H + 2, WQ_PLANES = 3;
constexpr uint32_t WQ_RP = WQ_QUADS * 16;           // 144: one E or O row
constexpr uint32_t WQ_LP = 2 * WQ_RP;               // 288: line pitch of the rows ([E | O] per line)
constexpr int WQ_PAIRS = 2 * WQ_QUADS;              // 18 voxel pairs per input line (w0-2 .. w0+33)
constexpr uint32_t WQ_PBOX = WQ_PLANES * WQ_LINES * WQ_PAIRS * 16;  // 15552: the TMA box (plain lines)
constexpr uint32_t WQ_G = 15616;                    // pooled gradient [8][16][32] bf16
constexpr uint32_t WQ_I = WQ_G + 8192;              // codes [8][16][32]
constexpr uint32_t WQ_STAGE = WQ_I + 4096;          // one TMA stage: box, pooled gradient, codes
constexpr uint32_t WQ_TX = WQ_PBOX + 8192 + 4096;
constexpr int WQ_GROUPS = 3;                        // builder groups, taking every third tile
constexpr int WQ_STAGES = 2 * WQ_GROUPS;            // stage s is only ever read by group s % 3
// E / O rows of one tile (the B operand), one buffer per builder group,
// including the last MMA's descriptor extent past the rows
constexpr uint32_t WQ_EOB = (2 * WQ_LINES + 14) * WQ_LP + 16 + 5 * WQ_LP + WQ_RP + 128;
constexpr uint32_t WQ_EO0 = WQ_STAGES * WQ_STAGE;   // first E / O buffer
constexpr uint32_t WQ_BAR = 256;
constexpr uint32_t WQ_SMEM = 1024 + WQ_EO0 + WQ_GROUPS * WQ_EOB + WQ_BAR;
constexpr int WQ_NSLOT = WQ_GROUPS;                 // dZ tiles in tensor memory, one per builder group
constexpr int WQ_THREADS = 128 + 128 * WQ_GROUPS;
constexpr uint32_t WQ_ACOL = 288;                   // first column of the dZ tiles (after 6 x 48 accumulator columns)
constexpr int WQ_N = 48;                            // 3 kh x (E, O) x 8
constexpr uint32_t WQ_IDESC = idesc_bf16(128, WQ_N, 0, 1);
static_assert(WQ_G >= WQ_PBOX && WQ_STAGE % 128 == 0 && WQ_EOB % 128 == 0, "stage layout");
static_assert(WQ_EOB >= WQ_PLANES * WQ_LINES * WQ_LP, "E / O rows");
static_assert(WQ_SMEM <= 227 * 1024, "shared memory");
static_assert(6 * WQ_N <= (int)WQ_ACOL && WQ_ACOL + WQ_NSLOT * 64 <= 512, "tensor memory");
static_assert(WQ_STAGES % WQ_GROUPS == 0, "stage ownership");
static_assert(8 * (2 * WQ_STAGES + 2 * WQ_NSLOT + 1 + 4) + 8 <= (int)WQ_BAR, "barrier area");

struct WqParams {
    int N, D, H, W;
    int tiles_w, tiles_h, num_tiles;
    FastDiv fd_w, fd_h, fd_d;
    float* part;  // [units][4 phases][32][108]
    int* status;
    uint64_t wait_ns;
};

struct WqTile {
    int n, d0, h0, w0;
};

// Tiles are numbered d fastest (one plane each), then w, h, n: the next tile of
// a CTA reads two of the same three input planes and, every other plane, the
// same pooled tile, which are still in L2.
__device__ __forceinline__ WqTile wq_decode(const WqParams& p, int tile) {
    WqTile t;
    uint32_t m = (uint32_t)tile, q = p.fd_d.div(m);
    t.d0 = (int)(m - q * p.fd_d.d);
    m = q;
    q = p.fd_w.div(m);
    t.w0 = (int)(m - q * p.fd_w.d) * WQ_W;
    m = q;
    q = p.fd_h.div(m);
    t.h0 = (int)(m - q * p.fd_h.d) * WQ_H;
    t.n = (int)q;
    return t;
}

// The CTA's tile range: num_tiles split into gridDim.x near-equal contiguous parts.
__device__ __forceinline__ void wq_range(const WqParams& p, int& t0, int& t1) {
    const int G = (int)gridDim.x, u = (int)blockIdx.x;
    const int base = p.num_tiles / G, rem = p.num_tiles - base * G;
    t0 = u * base + min(u, rem);
    t1 = t0 + base + (u < rem ? 1 : 0);
}

// De-interleave of one stage: item k < 972 copies one 16-byte voxel pair of the
// TMA box (54 lines x 18 pairs; pair 2q + 1 is E[q], pair 2q is O[q]) to its E
// or O row.  Items run in groups of eight that each hit all 32 banks once, on
// both the load and the store side (a line starts 288 = 32 mod 128 bytes after
// the previous one, in the box and in the rows; the O row 144 = 16 mod 128
// bytes after the E row): per line E[0..3] with O[3..6], then E[4..7] with
// O[7], O[0..2] (864 items), then E[8] and O[8] of four consecutive lines per
// group.  Returns source | destination << 16 (stage offsets), or all ones past
// the last item.
constexpr int WQ_DEINT = WQ_PLANES * WQ_LINES * WQ_PAIRS;  // 972
constexpr int WQ_DEINT_PER = (WQ_DEINT + 127) / 128;       // items per builder thread
__host__ __device__ constexpr uint32_t wq_deint_offsets(int k) {
    if (k >= WQ_DEINT) return 0xffffffffu;
    int line = 0, q = 0;
    bool odd = false;  // E (odd pair) or O
    if (k < 16 * WQ_PLANES * WQ_LINES) {
        const int e = k & 7, half = (k >> 3) & 1;
        line = k >> 4;
        odd = e < 4;
        q = half == 0 ? (odd ? e : e - 1) : (odd ? 4 + e : (e + 3) & 7);
    } else {
        const int j = k - 16 * WQ_PLANES * WQ_LINES;
        line = j >> 1;
        odd = (j & 1) == 0;
        q = 8;
    }
    const uint32_t src = (uint32_t)(line * WQ_PAIRS + 2 * q + (odd ? 1 : 0)) * 16u;
    const uint32_t dst = (uint32_t)line * WQ_LP + (odd ? 0u : WQ_RP) + (uint32_t)q * 16u;
    return src | (dst << 16);
}
static_assert((WQ_PLANES * WQ_LINES - 1) * WQ_LP + WQ_RP + 8 * 16 + 16 <= 65535, "packed offsets");
// only the last item of a thread can lie past the end (the guard in the builders)
static_assert(127 + 128 * (WQ_DEINT_PER - 2) < WQ_DEINT, "de-interleave items");

__global__ void __launch_bounds__(WQ_THREADS, 1)
    wgrad_quad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmI,
                      const WqParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + WQ_EO0 + WQ_GROUPS * WQ_EOB);
    uint64_t* full = bars;
    uint64_t* empty = full + WQ_STAGES;
    uint64_t* afull = empty + WQ_STAGES;
    uint64_t* aempty = afull + WQ_NSLOT;
    uint64_t* tfull = aempty + WQ_NSLOT;
    uint64_t* drain = tfull + 1;  // [4]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t0, t1;
    wq_range(p, t0, t1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < WQ_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);  // the four warps of one builder group
        }
        for (int b = 0; b < WQ_NSLOT; ++b) {
            mbar_init(&afull[b], 4);   // the four warps of builder group b
            mbar_init(&aempty[b], 3);  // three issuers' MMAs (dZ slot and E / O rows b)
        }
        mbar_init(tfull, 3);
        for (int k = 0; k < 3; ++k) mbar_init(&drain[k], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmG);
        tma_prefetch_desc(&tmI);
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
            // ---------------- TMA producer: E / O input rows, pooled gradient, codes
            int s = 0;
            uint32_t ph = 0, issued = 0, par = 0;
            bool ok = true;
            for (int tile = t0; tile < t1; ++tile) {
                const WqTile t = wq_decode(p, tile);
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                uint8_t* st = ring + s * WQ_STAGE;
                mbar_arrive_expect_tx(&full[s], WQ_TX);
                tma_load_5d(st, &tmX, &full[s], 4 * t.w0 - 8, t.h0 - 1, t.d0 - 1, t.n, 0);
                tma_load_5d(st + WQ_G, &tmG, &full[s], 0, t.w0 >> 1, t.h0 >> 1, t.d0 >> 1, t.n);
                tma_load_5d(st + WQ_I, &tmI, &full[s], 0, t.w0 >> 1, t.h0 >> 1, t.d0 >> 1, t.n);
                issued |= 1u << s;
                par = (par & ~(1u << s)) | (ph << s);
                if (++s == WQ_STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!ok) {
                for (int k = 0; k < WQ_STAGES; ++k)
                    if (issued & (1u << k)) mbar_wait_timed(&full[k], (par >> k) & 1, p.wait_ns);
            }
        }
    } else if (warp <= 3) {
        if (lane == 0) {
            // ---------------- MMA issuer of input plane kd: per K step the low half
            // (E[r] | O[r]: voxel slots 0-1 | -2..-1) and the high half (E[r+1] | O[r+1]:
            // slots 4-5 | 2-3), N = (kh, E/O, 8)
            const int kd = warp - 1;
            bool ok = true;
            uint32_t b = 0, bph = 0;  // dZ slot / E-O buffer and its phase
            for (int tile = t0, lt = 0; tile < t1; ++tile, ++lt) {
                if (!mbar_wait(&afull[b], bph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t rows = smem_u32(ring + WQ_EO0 + b * WQ_EOB) + kd * WQ_LINES * WQ_LP;
                const uint32_t a_tmem = tmem_base + WQ_ACOL + b * 64;
                // MN-major without swizzle: K groups (the next output line) WQ_LP apart
                // (leading byte offset), N groups (kh, E/O) WQ_RP apart (stride byte offset)
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
                        umma_bf16_tmem_a(tmem_base + (kd * 2 + hl) * WQ_N, a_tmem + 8 * j,
                                         sdesc(rows + 2 * j * WQ_LP + 16 * hl, WQ_LP, WQ_RP, SWZ_NONE), WQ_IDESC,
                                         (lt | j) ? 1u : 0u);
                umma_commit(&aempty[b]);
                if (++b == WQ_NSLOT) {
                    b = 0;
                    bph ^= 1;
                }
            }
            if (ok) {
                umma_commit(tfull);
            } else {
                umma_commit(&drain[kd]);
                mbar_wait_timed(&drain[kd], 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- builders: group g = warps 4 + 4g .. 7 + 4g takes the CTA's
        // tiles g, g + 3, ... (three tiles in flight) into dZ slot g and E / O buffer g;
        // warp f of a group builds phase f (lane = channel co) over all 16 lines,
        // then group 0 runs the epilogue
        const int f = warp & 3, grp = (warp - 4) >> 2, co = lane, gt = threadIdx.x - 128 - 128 * grp;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(f * 32) << 16);
        const uint32_t a_col = WQ_ACOL + (uint32_t)grp * 64;
        uint8_t* eo = ring + WQ_EO0 + grp * WQ_EOB;
        uint32_t doff[WQ_DEINT_PER];  // (source | destination << 16) of this thread's voxel pairs
#pragma unroll
        for (int i = 0; i < WQ_DEINT_PER; ++i) doff[i] = wq_deint_offsets(gt + 128 * i);
        int s = grp;
        uint32_t ph = 0, bph = 0;  // stage phase, slot phase
        bool ok = true;
        for (int tile = t0 + grp; tile < t1; tile += WQ_GROUPS) {
            // the stage's data, and the slot (dZ tile and E / O rows) free of the
            // MMAs of this group's previous tile
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&full[s], ph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL) &&
                                mbar_wait(&aempty[grp], bph ^ 1, abort_flag, p.wait_ns, p.status,
                                          WAIT_PRODUCER_EMPTY))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int dd = wq_decode(p, tile).d0 & 1;
            const uint8_t* st = ring + s * WQ_STAGE;
            // the input lines' voxel pairs (w0-2 .. w0+33: O[0], E[0], O[1], ...) into
            // the E and O rows of the MMA's B operand: all loads of a thread, then its
            // stores, in the bank-conflict-free order of wq_deint_offsets
            {
                uint4 dv[WQ_DEINT_PER];
#pragma unroll
                for (int i = 0; i < WQ_DEINT_PER; ++i)
                    if (i < WQ_DEINT_PER - 1 || doff[i] != 0xffffffffu)
                        dv[i] = *reinterpret_cast<const uint4*>(st + (doff[i] & 0xffffu));
#pragma unroll
                for (int i = 0; i < WQ_DEINT_PER; ++i)
                    if (i < WQ_DEINT_PER - 1 || doff[i] != 0xffffffffu)
                        *reinterpret_cast<uint4*>(eo + (doff[i] >> 16)) = dv[i];
            }
            fence_proxy_async_smem();
            const uint16_t* gp = reinterpret_cast<const uint16_t*>(st + WQ_G) + co;
            const uint8_t* ip = st + WQ_I + co;
            // column c holds rows 2c, 2c+1 = quads i, i+1 of line c/4 (i = 2 (c % 4)):
            // voxels w = 4i + f and 4i + 4 + f, pooled w 2i + f/2 and 2i + 2 + f/2.
            // Lines 2l and 2l + 1 (columns c and c + 4) share their pooled values.
            // Two halves of 32 columns (pooled lines 0-3, 4-7).
            const uint32_t code0 = (uint32_t)(dd * 4 + (f & 1)), code1 = code0 + 2;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t col[32];
#pragma unroll
                for (int l = 0; l < 4; ++l)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int o = (4 * hf + l) * 16 + 4 * q4 + (f >> 1);
                        const uint32_t k0 = ip[o * 32], k1 = ip[(o + 2) * 32];
                        const uint32_t g0 = gp[o * 32], g1 = gp[(o + 2) * 32];
                        col[8 * l + q4] = (k0 == code0 ? g0 : 0u) | ((k1 == code0 ? g1 : 0u) << 16);
                        col[8 * l + 4 + q4] = (k0 == code1 ? g0 : 0u) | ((k1 == code1 ? g1 : 0u) << 16);
                    }
                tmem_st32(lane_addr + a_col + 32 * hf, col);
            }
            // the stage is no longer read by this warp
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[grp]);
            s += WQ_GROUPS;
            if (s >= WQ_STAGES) {
                s -= WQ_STAGES;
                ph ^= 1;
            }
            bph ^= 1;
        }
        // ---------------- epilogue: this lane's (f, co) partial of every dW entry
        if (ok && grp == 0 &&
            __all_sync(0xffffffffu, mbar_wait(tfull, 0, abort_flag, p.wait_ns, p.status, WAIT_EPI_TMEM_FULL))) {
            tc_fence_after();
            float* out = p.part + (((int64_t)blockIdx.x * 4 + f) * 32 + co) * 108;
#pragma unroll 1
            for (int kd = 0; kd < 3; ++kd)
#pragma unroll 1
                for (int hl = 0; hl < 2; ++hl) {
                    uint32_t ra[32], rb[32];  // columns 0-31, 32-47
                    tmem_ld32(lane_addr + (kd * 2 + hl) * WQ_N, ra);
                    tmem_ld16(lane_addr + (kd * 2 + hl) * WQ_N + 32, rb);
                    tmem_ld_wait();
#pragma unroll
                    for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                        for (int eo = 0; eo < 2; ++eo)
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                // voxel slot of the E / O pair: low half 0-1 / -2..-1, high half 4-5 / 2-3
                                const int s0 = hl == 0 ? (eo == 0 ? 0 : -2) : (eo == 0 ? 4 : 2);
                                const int kw = s0 + (e >> 2) - f + 1;
                                if (kw >= 0 && kw <= 2)
                                {
                                    const int n = kh * 16 + eo * 8 + e;
                                    out[(kd * 9 + kh * 3 + kw) * 4 + (e & 3)] =
                                        __uint_as_float(n < 32 ? ra[n] : rb[n - 32]);
                                }
                            }
                }
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

bool wgrad_quad_supported(int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    return c_in == 4 && c_out == 32 && d % 2 == 0 && h % WQ_H == 0 && w % WQ_W == 0;
}

static int64_t wq_tiles(int64_t n, int64_t d, int64_t h, int64_t w) { return n * d * (h / WQ_H) * (w / WQ_W); }

static int wq_units(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(num_sms, wq_tiles(n, d, h, w)));
}

size_t wgrad_quad_workspace_bytes(int num_sms, int64_t n, int64_t d, int64_t h, int64_t w) {
    return (size_t)wq_units(num_sms, n, d, h, w) * 4 * 32 * 108 * sizeof(float);
}

// The input as (4*W elements per line, H, D, N, 1); box: 36 voxels x 18 lines x 3 planes.
static bool wq_lines_map(CUtensorMap* m, const void* x, int64_t n, int64_t d, int64_t h, int64_t w) {
    const uint64_t dims[5] = {(uint64_t)w * 4, (uint64_t)h, (uint64_t)d, (uint64_t)n, 1u};
    const uint64_t str[4] = {(uint64_t)w * 8, (uint64_t)(h * w * 8), (uint64_t)(d * h * w * 8),
                             (uint64_t)(n * d * h * w * 8)};
    const uint32_t box[5] = {(uint32_t)(WQ_PAIRS * 8), (uint32_t)WQ_LINES, (uint32_t)WQ_PLANES, 1u, 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bool wq_pooled_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int64_t n, int64_t d,
                          int64_t h, int64_t w) {
    const uint64_t d2 = d / 2, h2 = h / 2, w2 = w / 2;
    const uint64_t dims[5] = {32u, w2, h2, d2, (uint64_t)n};
    const uint64_t str[4] = {(uint64_t)32 * esz, w2 * 32 * esz, h2 * w2 * 32 * esz, d2 * h2 * w2 * 32 * esz};
    const uint32_t box[5] = {32u, (uint32_t)(WQ_W / 2), (uint32_t)(WQ_H / 2), 1u, 1u};
    return encode_tmap(m, dt, 5, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

cf_status launch_wgrad_quad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, const uint16_t* x,
                            const uint16_t* g, const uint8_t* idx, float* part, int* n_splits) {
    if (!wgrad_quad_supported(d, h, w, 4, 32)) return CF_ERR_UNSUPPORTED;
    const int64_t tiles = wq_tiles(n, d, h, w);
    if (tiles > INT32_MAX) return CF_ERR_UNSUPPORTED;
    CUtensorMap tx, tg, ti;
    if (!wq_lines_map(&tx, x, n, d, h, w) ||
        !wq_pooled_map(&tg, g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, n, d, h, w) ||
        !wq_pooled_map(&ti, idx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, n, d, h, w))
        return CF_ERR_CUDA;
    WqParams p;
    p.N = (int)n;
    p.D = (int)d;
    p.H = (int)h;
    p.W = (int)w;
    p.tiles_w = (int)(w / WQ_W);
    p.tiles_h = (int)(h / WQ_H);
    p.num_tiles = (int)tiles;
    p.fd_w = FastDiv::make((uint32_t)p.tiles_w);
    p.fd_h = FastDiv::make((uint32_t)p.tiles_h);
    p.fd_d = FastDiv::make((uint32_t)d);
    p.part = part;
    p.status = ctx.status;
    p.wait_ns = ctx.wait_ns;
    if (cudaFuncSetAttribute(wgrad_quad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WQ_SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = wq_units(ctx.num_sms, n, d, h, w);
    wgrad_quad_kernel<<<grid, WQ_THREADS, WQ_SMEM, ctx.stream>>>(tx, tg, ti, p);
    if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
    *n_splits = grid * 4;
    return CF_OK;
}

}  // namespace cf
