// cf_noalloc.cu -- cf_bias_lrelu_pool_bwd_noalloc: the pool/leaky-ReLU backward
// for callers that cannot allocate device memory, e.g. an operator plugged
// into a host framework that owns every device allocation and gives its
// plug-ins no allocator and no workspace.  The bias-gradient partial sums that
// cf_bias_lrelu_pool_bwd keeps in a caller workspace live here in a
// file-scope device array instead.
//
// The array is a fixed 1 MiB per device (every GPU that loads the library
// holds it until the process exits).  It is shared by all calls and keeps the
// last call's contents; this operation overwrites every partial it reads, so
// nothing needs clearing between calls.  Calls whose work overlaps on the GPU
// (two streams, or two host threads) race on the array.
#include <mutex>

#include "cf_internal.h"

namespace cf {

constexpr size_t kNoallocScratchBytes = 1u << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

namespace {
std::mutex g_na_mu;
float* g_na_ptr[64] = {nullptr};
int g_na_sms[64] = {0};
}  // namespace

}  // namespace cf

using namespace cf;

extern "C" cf_status cf_bias_lrelu_pool_bwd_noalloc(int64_t n, int64_t d, int64_t h, int64_t w, int32_t c,
                                                    const uint16_t* dy, const uint16_t* y, const uint8_t* idx,
                                                    float slope, uint16_t* dz, uint16_t* dy_pre, float* dbias,
                                                    void* stream) {
    if (n <= 0 || d <= 0 || h <= 0 || w <= 0 || c <= 0 || dy == nullptr) return CF_ERR_INVALID_ARG;
    if (dz != nullptr && idx == nullptr) return CF_ERR_INVALID_ARG;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(dy) || (y && !aligned16(y)) || (idx && !aligned16(idx)) || (dz && !aligned16(dz)) ||
        (dy_pre && !aligned16(dy_pre)) || (dbias && !aligned16(dbias)))
        return CF_ERR_INVALID_ARG;
    if (c % 8 != 0 || c > 2048 || ((d | h | w) & 1)) return CF_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CF_ERR_CUDA;
    float* scratch = nullptr;
    int sms = 0;
    {
        // First call on a device: look up the array's device address (with that
        // device current) and the SM count; later calls reuse them.
        std::lock_guard<std::mutex> lock(g_na_mu);
        if (g_na_ptr[dev] == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CF_ERR_CUDA;
            if (cudaDeviceGetAttribute(&g_na_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return CF_ERR_CUDA;
            g_na_ptr[dev] = static_cast<float*>(p);
        }
        scratch = g_na_ptr[dev];
        sms = g_na_sms[dev];
    }
    // The partials need (blocks x c) floats; beyond the array's size the call
    // is refused before anything is launched.
    if (dbias != nullptr && pool_bwd_workspace_bytes(sms, c) > kNoallocScratchBytes) return CF_ERR_WORKSPACE;
    return cf_bias_lrelu_pool_bwd(n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, dbias, scratch,
                                  kNoallocScratchBytes, stream);
}
