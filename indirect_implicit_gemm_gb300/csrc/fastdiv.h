// fastdiv.h -- division of non-negative int32 values by a run-time invariant
// divisor with one multiply-high, an add and a shift (Granlund & Montgomery,
// "Division by Invariant Integers using Multiplication", PLDI 1994, the
// round-up multiplier of their section 4).  Valid for dividends in [0, 2^31).
#pragma once

#include <stdint.h>

namespace convgb {

struct FastDiv {
    uint32_t d;      // divisor, >= 1
    uint32_t mult;   // m' = floor(2^32 * (2^l - d) / d) + 1
    uint32_t shift;  // l = ceil(log2(d))

    FastDiv() = default;
    __host__ explicit FastDiv(uint32_t divisor) : d(divisor)
    {
        uint32_t l = 0;
        while ((1ull << l) < divisor) ++l;
        shift = l;
        uint64_t num = (1ull << 32) * ((1ull << l) - divisor);
        mult = static_cast<uint32_t>(num / divisor + 1);
    }

    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        return (__umulhi(n, mult) + n) >> shift;
    }
    // q = n / d, r = n - q*d
    __device__ __forceinline__ void divmod(uint32_t n, uint32_t& q, uint32_t& r) const
    {
        q = div(n);
        r = n - q * d;
    }
};

}  // namespace convgb
