// Division of 32-bit unsigned integers by a run-time invariant divisor with a
// multiply-high and shifts, following T. Granlund and P. L. Montgomery,
// "Division by Invariant Integers using Multiplication" (PLDI 1994), §4
// (unsigned division, the variant that keeps every intermediate in 32 bits):
//   l  = ceil(log2 d)
//   m' = floor(2^32 * (2^l - d) / d) + 1
//   t1 = mulhi(m', n);  q = (t1 + ((n - t1) >> min(l, 1))) >> max(l - 1, 0)
// exact for every 0 <= n < 2^32 and 1 <= d < 2^32.  The kernels use it to split
// a row index into (query position, head, batch) without hardware division.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SMS_HD __host__ __device__ __forceinline__
#else
#define SMS_HD inline
#endif

namespace sms {

struct FastDiv {
    uint32_t d;    // divisor
    uint32_t m;    // m'
    uint32_t s1;   // min(l, 1)
    uint32_t s2;   // max(l - 1, 0)

    SMS_HD FastDiv() : d(1), m(1), s1(0), s2(0) {}
    explicit FastDiv(uint32_t div)
    {
        d = div ? div : 1;
        uint32_t l = 0;
        while (l < 32 && (uint64_t(1) << l) < d) ++l;  // ceil(log2 d)
        const uint64_t two_l = uint64_t(1) << l;
        m = uint32_t(((uint64_t(1) << 32) * (two_l - d)) / d + 1);
        s1 = l < 1 ? l : 1;
        s2 = l > 1 ? l - 1 : 0;
    }

    SMS_HD uint32_t div(uint32_t n) const
    {
#if defined(__CUDA_ARCH__)
        const uint32_t t1 = __umulhi(m, n);
#else
        const uint32_t t1 = uint32_t((uint64_t(m) * n) >> 32);
#endif
        return (t1 + ((n - t1) >> s1)) >> s2;
    }
};

}  // namespace sms
