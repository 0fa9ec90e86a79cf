// conv_quad.cu -- forward conv of the CosmoFlow first layer (c_in = 4, c_out
// 16 or 32) with the bias + leaky ReLU + 2x2x2 max-pool epilogue, its A
// operand read by the tensor core straight from the input tile in shared
// memory (no im2col, no builder warps).
//
// (CosmoFlow page, section III-A: 3D conv layers on the 4-channel input, each
// followed by leaky ReLU and pooling.)
//
//   Z[n,d,h,w,co] = sum_{kd,kh,kw,ci} W[co,kd,kh,kw,ci] * X[n,d+kd-1,h+kh-1,w+kw-1,ci]
//
// One voxel of the input is 8 bytes, a pair of voxels one 16-byte row of a
// UMMA core matrix.  The input lines of a tile are loaded by two TMA boxes of
// the input viewed as (8 elements, 32-byte quads, lines, planes, n): E holds
// the even pairs of each line (E[j] = pair 2j of the tile), O, from the same
// view shifted by 16 bytes, the odd pairs (O[j] = pair 2j - 1).  Row r of an
// output line stands for the quad of voxels w = 4r .. 4r+3, whose 3-wide
// windows need voxels 4r-1 .. 4r+4, covered by two MMAs per tap pair (kd, kh):
//   half "a": K = [E[r] | O[r+1]] = voxels 4r, 4r+1 | 4r+2, 4r+3
//   half "b": K = [E[r+1] | O[r]] = voxels 4r+4, 4r+5 | 4r-2, 4r-1
// Both are plain K-major descriptors without swizzle: 8-row groups are the
// lines (SBO = the box's line pitch), the two K halves come from the E and O
// boxes (LBO = their distance, +-16 bytes).  N = 4 output phases x c_out: the
// filter is stored as 18 slabs (kd, kh, half) whose row (phase f, co) holds,
// for the K slot of voxel 4r + s, the tap kw = s - f + 1 (zero outside 0..2).
//
// Output tile: 2 planes x 16 lines x 32 voxels.  M = 128 rows = 16 lines x 8
// quads, one accumulator per output plane, each issued by its own MMA thread.
// A pooling window is then (the two plane accumulators) x (the lines of a
// lane pair 8 lanes apart) x (two phases of one row): the epilogue takes the
// first maximum of its four values per window and channel, trades one of its
// two windows with the lane 8 away, and finalises the other.
//
// Roles (384 threads): warp 0 TMA producer, warps 1 and 2 MMA issuers (plane
// 0 / 1), warp 3 tensor-memory allocation, warps 4..11 epilogue (two per TMEM
// lane quarter, each 16 of the 32 channels).
#include "halo_common.cuh"

namespace cf {

constexpr int QT_W = 32, QT_H = 16, QT_D = 2;  // output tile
constexpr int Q_QUADS = QT_W / 4 + 1;          // E / O entries per line (9)
constexpr int Q_LINES = QT_H + 2, Q_PLANES = QT_D + 2;
constexpr uint32_t Q_LINE_PITCH = Q_QUADS * 16;                        // 144
constexpr uint32_t Q_BOX = Q_PLANES * Q_LINES * Q_LINE_PITCH;          // 10368 bytes
constexpr uint32_t Q_STAGE = 2 * Q_BOX;                                // E then O

template <int CO>
struct QuadCfg {
    static constexpr int N = 4 * CO;                         // MMA width: 4 phases x c_out
    static constexpr uint32_t SLAB = N * 32;                 // one filter slab: N rows x 16 K (two halves)
    static constexpr uint32_t B_BYTES = 18 * SLAB;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr int STAGES_RAW = (int)((227 * 1024 - 1024 - B_BYTES - BAR_BYTES) / Q_STAGE);
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr uint32_t SMEM = 1024 + STAGES * Q_STAGE + B_BYTES + BAR_BYTES;
    static constexpr uint32_t ACC = 2 * N;                   // both planes of a tile
    static constexpr uint32_t TMEM_COLS = 2 * ACC;           // double-buffered
    static constexpr uint32_t IDESC = idesc_bf16(128, N, 0, 0);
    static_assert(STAGES >= 2, "shared memory");
    static_assert(TMEM_COLS <= 512, "tensor memory");
    static_assert(8 * (2 * STAGES + 2 + 2 + 2) + 8 <= (int)BAR_BYTES, "barrier area");
};

struct QuadParams {
    int N, D, H, W;
    int tiles_w, tiles_h, tiles_d, num_tiles;
    FastDiv fd_w, fd_h, fd_d;
    const uint16_t* w;   // [CO][27][4]
    const float* bias;   // [CO] or NULL
    float slope;
    uint16_t* y;         // pooled [N][D/2][H/2][W/2][CO]
    uint8_t* idx;        // same shape, or NULL
    int* status;
    uint64_t wait_ns;
};

struct QTile {
    int n, d0, h0, w0;
};

// Tiles are numbered w fastest, then h, d, n.
__device__ __forceinline__ QTile quad_decode(const QuadParams& p, int tile) {
    QTile t;
    uint32_t m = (uint32_t)tile, q = p.fd_w.div(m);
    t.w0 = (int)(m - q * p.fd_w.d) * QT_W;
    m = q;
    q = p.fd_h.div(m);
    t.h0 = (int)(m - q * p.fd_h.d) * QT_H;
    m = q;
    q = p.fd_d.div(m);
    t.d0 = (int)(m - q * p.fd_d.d) * QT_D;
    t.n = (int)q;
    return t;
}

template <int CO>
__global__ void __launch_bounds__(384, 1)
    conv_quad_kernel(const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmO,
                     const QuadParams p) {
    using C = QuadCfg<CO>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;                                  // stages: [E box][O box]
    uint8_t* bsm = smem + C::STAGES * Q_STAGE;             // filter slabs
    uint64_t* bars = reinterpret_cast<uint64_t*>(bsm + C::B_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;  // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // both issuers' MMAs on the stage done
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 2);   // both planes issued and complete
            mbar_init(&tempty[a], 8);  // one arrival per epilogue warp
            mbar_init(&drain[a], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmE);
        tma_prefetch_desc(&tmO);
    }
    // filter slabs: slab m = (kd*3 + kh)*2 + half, row (f, co) = f*CO + co, K
    // half hh (16 bytes: two voxels x 4 channels) at hh * N * 16.  The K slot
    // k8 of half hh of slab half "a" is voxel 4r + 2*hh + k8/4, of "b" voxel
    // 4r + 4 - 6*hh + k8/4; phase f reads tap kw = slot - f + 1.
    for (int e = threadIdx.x; e < 18 * 2 * C::N; e += blockDim.x) {
        const int m = e / (2 * C::N), rem = e - m * (2 * C::N);
        const int hh = rem / C::N, row = rem - hh * C::N;
        const int f = row / CO, co = row - f * CO;
        const int kdkh = m >> 1, half = m & 1;
        const int s0 = half == 0 ? 2 * hh : 4 - 6 * hh;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int kw = s0 + (k8 >> 2) - f + 1, ci = k8 & 3;
            uint32_t bits = 0;
            if (kw >= 0 && kw <= 2) bits = p.w[((int64_t)co * 27 + kdkh * 3 + kw) * 4 + ci];
            v[k8 >> 1] |= bits << (16 * (k8 & 1));
        }
        *reinterpret_cast<uint4*>(bsm + m * C::SLAB + hh * (C::N * 16) + row * 16) = make_uint4(v[0], v[1], v[2], v[3]);
    }
    fence_proxy_async_smem();
    if (warp == 3) {
        tmem_alloc(tmem_holder, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: the E and O boxes of each tile
            int s = 0;
            uint32_t ph = 0, issued = 0, par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const QTile t = quad_decode(p, tile);
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.wait_ns, p.status, WAIT_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                uint8_t* st = ring + s * Q_STAGE;
                mbar_arrive_expect_tx(&full[s], Q_STAGE);
                const int q0 = t.w0 >> 2;
                tma_load_5d(st, &tmE, &full[s], 0, q0, t.h0 - 1, t.d0 - 1, t.n);
                tma_load_5d(st + Q_BOX, &tmO, &full[s], 0, q0 - 1, t.h0 - 1, t.d0 - 1, t.n);
                issued |= 1u << s;
                par = (par & ~(1u << s)) | (ph << s);
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!ok) {
                for (int k = 0; k < C::STAGES; ++k)
                    if (issued & (1u << k)) mbar_wait_timed(&full[k], (par >> k) & 1, p.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 2) {
        if (lane == 0) {
            // ---------------- MMA issuer of output plane pl: 9 tap pairs x 2 halves
            const int pl = warp - 1;
            int s = 0;
            uint32_t ph = 0, local = 0;
            bool ok = true;
            const uint32_t b_addr = smem_u32(bsm);
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
                const uint32_t a = local & 1, use = local >> 1;
                if (!mbar_wait(&tempty[a], (use & 1) ^ 1, abort_flag, p.wait_ns, p.status, WAIT_MMA_TMEM_EMPTY) ||
                    !mbar_wait(&full[s], ph, abort_flag, p.wait_ns, p.status, WAIT_MMA_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + a * C::ACC + pl * C::N;
                const uint32_t e_addr = smem_u32(ring + s * Q_STAGE);
#pragma unroll
                for (int kd = 0; kd < 3; ++kd)
#pragma unroll
                    for (int kh = 0; kh < 3; ++kh) {
                        const uint32_t line = e_addr + ((pl + kd) * Q_LINES + kh) * Q_LINE_PITCH;
                        const int m = (kd * 3 + kh) * 2;
                        umma_bf16(d_tmem, sdesc(line, Q_BOX + 16, Q_LINE_PITCH, SWZ_NONE),
                                  sdesc(b_addr + m * C::SLAB, C::N * 16, 128, SWZ_NONE), C::IDESC,
                                  (kd | kh) ? 1u : 0u);
                        umma_bf16(d_tmem, sdesc(line + 16, Q_BOX - 16, Q_LINE_PITCH, SWZ_NONE),
                                  sdesc(b_addr + (m + 1) * C::SLAB, C::N * 16, 128, SWZ_NONE), C::IDESC, 1u);
                    }
                umma_commit(&empty[s]);
                umma_commit(&tfull[a]);
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!ok) {
                umma_commit(&drain[pl]);
                mbar_wait_timed(&drain[pl], 0, p.wait_ns);
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: lane quarter q, channels 16*hf .. 16*hf + 15
        const int q = warp & 3, hf = (warp - 4) >> 2;
        const int m = q * 32 + lane;
        const int g = m >> 3, i = m & 7;  // output line of the tile, quad of the line
        const int dh = g & 1;             // the lane 8 away holds the other line of the window
        const bool active = hf * 16 < CO;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + hf * 16;
        float bias[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
            bias[c] = (active && p.bias != nullptr) ? __ldg(p.bias + hf * 16 + c) : 0.f;
        const int D2 = p.D >> 1, H2 = p.H >> 1, W2 = p.W >> 1;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t a = local & 1, use = local >> 1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&tfull[a], use & 1, abort_flag, p.wait_ns, p.status, WAIT_EPI_TMEM_FULL)))
                break;
            tc_fence_after();
            if (!active) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[a]);
                continue;
            }
            const QTile t = quad_decode(p, tile);
            // per window w2 (phases 2*w2, 2*w2 + 1) and channel: first maximum over
            // (plane dd, phase dw) in code order dd*4 + dh*2 + dw
            float mx[2][16];
            int kx[2][16];
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
                uint32_t r00[32], r01[32], r10[32], r11[32];
                const uint32_t c0 = lane_addr + a * C::ACC + (2 * w2) * CO;
                tmem_ld16(c0, r00);
                tmem_ld16(c0 + CO, r01);
                tmem_ld16(c0 + C::N, r10);
                tmem_ld16(c0 + C::N + CO, r11);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float v = __uint_as_float(r00[c]);
                    int k = dh * 2;
                    const float v1 = __uint_as_float(r01[c]), v2 = __uint_as_float(r10[c]),
                                v3 = __uint_as_float(r11[c]);
                    if (v1 > v) {
                        v = v1;
                        k = dh * 2 + 1;
                    }
                    if (v2 > v) {
                        v = v2;
                        k = 4 + dh * 2;
                    }
                    if (v3 > v) {
                        v = v3;
                        k = 4 + dh * 2 + 1;
                    }
                    mx[w2][c] = v;
                    kx[w2][c] = k;
                }
            }
            // the accumulator is in registers: hand it back before the exchange and stores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
            // lane pair (dh = 0, 1): this lane finalises window dh and takes the
            // partner's values for it
            float y[16];
            uint32_t codes[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float v = dh ? mx[1][c] : mx[0][c];
                int k = dh ? kx[1][c] : kx[0][c];
                const float ov = __shfl_xor_sync(0xffffffffu, dh ? mx[0][c] : mx[1][c], 8);
                const int ok2 = __shfl_xor_sync(0xffffffffu, dh ? kx[0][c] : kx[1][c], 8);
                pool_combine(v, k, ov, ok2);
                y[c] = lrelu(v + bias[c], p.slope);
                codes[c >> 2] |= (uint32_t)k << (8 * (c & 3));
            }
            const int pd = t.d0 >> 1, phh = (t.h0 >> 1) + (g >> 1), pw = (t.w0 >> 1) + 2 * i + dh;
            const int64_t po = ((((int64_t)t.n * D2 + pd) * H2 + phh) * W2 + pw) * CO + hf * 16;
            uint4* yo = reinterpret_cast<uint4*>(p.y + po);
            yo[0] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                               pack_bf16x2(y[6], y[7]));
            yo[1] = make_uint4(pack_bf16x2(y[8], y[9]), pack_bf16x2(y[10], y[11]), pack_bf16x2(y[12], y[13]),
                               pack_bf16x2(y[14], y[15]));
            if (p.idx != nullptr)
                *reinterpret_cast<uint4*>(p.idx + po) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 3) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

bool quad_path_supported(int64_t d, int64_t h, int64_t w, int c_in, int c_out) {
    return c_in == 4 && (c_out == 16 || c_out == 32) && d % QT_D == 0 && h % QT_H == 0 && w % QT_W == 0;
}

// The input as (8 elements, W/4 quads of 32 bytes, H, D, N), from `base`
// (x for the even pairs, x + 16 bytes for the odd ones); box 8 x 9 x 18 x 4.
static bool make_quad_map(CUtensorMap* m, const void* base, int64_t n, int64_t d, int64_t h, int64_t w) {
    const uint64_t dims[5] = {8u, (uint64_t)(w / 4), (uint64_t)h, (uint64_t)d, (uint64_t)n};
    const uint64_t str[4] = {32u, (uint64_t)w * 8, (uint64_t)(h * w * 8), (uint64_t)(d * h * w * 8)};
    const uint32_t box[5] = {8u, (uint32_t)Q_QUADS, (uint32_t)Q_LINES, (uint32_t)Q_PLANES, 1u};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int CO>
static cf_status run_quad(const LaunchCtx& ctx, const QuadParams& p, const uint16_t* x) {
    using C = QuadCfg<CO>;
    CUtensorMap te, to;
    if (!make_quad_map(&te, x, p.N, p.D, p.H, p.W) ||
        !make_quad_map(&to, reinterpret_cast<const uint8_t*>(x) + 16, p.N, p.D, p.H, p.W))
        return CF_ERR_CUDA;
    auto kern = conv_quad_kernel<CO>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return CF_ERR_CUDA;
    const int grid = grid_for(kern, C::SMEM, 384, ctx.num_sms, p.num_tiles, C::TMEM_COLS);
    kern<<<grid, 384, C::SMEM, ctx.stream>>>(te, to, p);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

cf_status launch_conv_quad(const LaunchCtx& ctx, int64_t n, int64_t d, int64_t h, int64_t w, int c_out,
                           const uint16_t* x, const uint16_t* wk, uint16_t* y, uint8_t* idx, const float* bias,
                           float slope) {
    if (!quad_path_supported(d, h, w, 4, c_out)) return CF_ERR_UNSUPPORTED;
    QuadParams p;
    p.N = (int)n;
    p.D = (int)d;
    p.H = (int)h;
    p.W = (int)w;
    p.tiles_w = (int)(w / QT_W);
    p.tiles_h = (int)(h / QT_H);
    p.tiles_d = (int)(d / QT_D);
    const int64_t tiles = n * p.tiles_d * p.tiles_h * p.tiles_w;
    if (tiles > INT32_MAX) return CF_ERR_UNSUPPORTED;
    p.num_tiles = (int)tiles;
    p.fd_w = FastDiv::make((uint32_t)p.tiles_w);
    p.fd_h = FastDiv::make((uint32_t)p.tiles_h);
    p.fd_d = FastDiv::make((uint32_t)p.tiles_d);
    p.w = wk;
    p.bias = bias;
    p.slope = slope;
    p.y = y;
    p.idx = idx;
    p.status = ctx.status;
    p.wait_ns = ctx.wait_ns;
    return c_out == 32 ? run_quad<32>(ctx, p, x) : run_quad<16>(ctx, p, x);
}

}  // namespace cf
