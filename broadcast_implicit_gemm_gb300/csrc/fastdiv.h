// fastdiv.h -- unsigned division by a divisor fixed for a launch, as one
// multiply-high, one add and one shift.  The method is the round-up variant of
// Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication" (PLDI 1994): with l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1, the quotient n / d equals
// (mulhi(m, n) + n) >> l for every dividend 0 <= n < 2^31.  The host computes
// (m, l) once per plan; kernels divide tile and unit indices with it instead of
// the much longer integer-division sequence.
//
// No CUDA dependency on the host side, so that a plain C++ test can check it.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define BIGEMM_FD_HD __host__ __device__ __forceinline__
#else
#define BIGEMM_FD_HD inline
#endif

namespace bigemm {

struct FastDiv {
    uint32_t d;   // the divisor, 1 <= d < 2^31
    uint32_t m;   // magic multiplier
    uint32_t l;   // shift, ceil(log2 d)
};

// Returns the divisor's constants; d = 0 is mapped to 1 (callers never divide by 0).
inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    if (d == 0) d = 1;
    uint32_t l = 0;
    while (l < 31 && (1u << l) < d) ++l;
    f.d = d;
    f.l = l;
    f.m = (uint32_t)(((((uint64_t)1) << 32) * ((((uint64_t)1) << l) - d)) / d + 1);
    return f;
}

// n / f.d for 0 <= n < 2^31.
BIGEMM_FD_HD uint32_t fd_div(uint32_t n, const FastDiv &f)
{
#if defined(__CUDA_ARCH__)
    const uint32_t t = __umulhi(n, f.m);
#else
    const uint32_t t = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
    return (t + n) >> f.l;
}

// n / f.d and n % f.d.
BIGEMM_FD_HD uint32_t fd_divmod(uint32_t n, const FastDiv &f, uint32_t *rem)
{
    const uint32_t q = fd_div(n, f);
    *rem = n - q * f.d;
    return q;
}

}  // namespace bigemm
