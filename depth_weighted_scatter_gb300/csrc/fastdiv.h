// fastdiv.h -- unsigned division by a run-time constant, for n < 2^31.
//
// The round-up method of Granlund & Montgomery, "Division by Invariant
// Integers using Multiplication" (PLDI 1994): with l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1,
//     n / d = (umulhi(m, n) + n) >> l      for 0 <= n < 2^31, d >= 1,
// where the sum is formed in 64 bits.  Plain C++ (host and device) so the
// CPU tests can check it against ordinary division.
#pragma once

#include <stdint.h>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#ifndef __forceinline__
#define __forceinline__ inline
#endif
#endif

namespace bevpool {

struct FastDiv {
    uint32_t d = 1, m = 1, l = 0;
    FastDiv() = default;
    __host__ __device__ explicit FastDiv(uint32_t divisor) : d(divisor) {
        l = 0;
        while ((1ull << l) < d) ++l;
        m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    }
    __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
        const uint32_t t = __umulhi(m, n);
#else
        const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(m) * n) >> 32);
#endif
        return static_cast<uint32_t>((static_cast<uint64_t>(t) + n) >> l);
    }
};

}  // namespace bevpool
