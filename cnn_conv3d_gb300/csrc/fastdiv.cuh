// fastdiv.cuh -- unsigned division by a divisor fixed at launch time.
#pragma once

#include <cstdint>

namespace cf {

// Division by a divisor fixed at launch, by multiply and shifts (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", 1994,
// the unsigned N-bit algorithm of their figure 4.1 with N = 32): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
//   q = (t + ((x - t) >> min(l, 1))) >> max(l - 1, 0),  t = mulhi(m, x),
// equals floor(x / d) for every 32-bit x.  Tile decoders run it once per
// tile in every epilogue thread, where an integer division costs about 20
// instructions.
struct FastDiv {
    uint32_t d, m, s1, s2;
    static FastDiv make(uint32_t d) {
        uint32_t l = 0;
        while (l < 32 && (1ull << l) < d) ++l;
        FastDiv f;
        f.d = d;
        f.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
        f.s1 = l ? 1u : 0u;
        f.s2 = l ? l - 1 : 0u;
        return f;
    }
    __device__ __forceinline__ uint32_t div(uint32_t x) const {
        const uint32_t t = __umulhi(x, m);
        return (t + ((x - t) >> s1)) >> s2;
    }
};

}  // namespace cf
