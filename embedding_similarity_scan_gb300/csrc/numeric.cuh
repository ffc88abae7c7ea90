// numeric.cuh — fp32 and integer building blocks shared by the kernels:
// warp reductions, a compensated sum, power-of-two row scaling, and an exact
// fixed-point representation for sums that must not depend on the order of
// their terms.  None of them uses 64-bit floating point: GB300's FP64 rate is
// a small fraction of its fp32 rate, and a conversion to or from double runs
// at that rate.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dseq {

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ int warp_or_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Compensated (Kahan) fp32 sum: error about 2 ulp of the total whatever the
// number of terms.  Norms are taken as sums of squares of values scaled into
// [0, 1) by a power of two, so nothing overflows.
struct KahanSum {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float term) {
        const float y = term - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ float total() const { return s - c; }
};

// max |v| over a row (one warp), and whether every entry is finite
__device__ __forceinline__ float row_absmax(const float *src, int D, int lane, int &bad) {
    float mx = 0.0f;
    int b = 0;
    for (int k = lane; k < D; k += 32) {
        const float v = src[k];
        if (!isfinite(v)) b = 1;
        mx = fmaxf(mx, fabsf(v));
    }
    bad = warp_or_i(b);
    return warp_max_f(mx);
}

// exponent e with max |v| = f 2^e, f in [0.5, 1): v * 2^-e lies in (-1, 1)
__device__ __forceinline__ int scale_exponent(float mx) {
    int e = 0;
    if (mx > 0.0f) frexpf(mx, &e);
    return e;
}

// ---- fixed point: v = trunc(x 2^F) in 64-bit two's complement ----------------
// With every |x| < 2^E and at most 2^L terms, F = 62 - E - L keeps any sum
// below 2^62: integer sums are then exact and independent of term order.

// trunc(x 2^F) from the bits of x (integer operations only; exact)
__device__ __forceinline__ long long to_fixed(float x, int F) {
    const uint32_t b = __float_as_uint(x);
    int ef = (int)((b >> 23) & 0xffu);
    uint32_t m = b & 0x7fffffu;
    if (ef == 0) {
        if (m == 0) return 0;
        ef = 1;  // subnormal: no implicit bit
    } else {
        m |= 0x800000u;
    }
    const int s = ef - 150 + F;  // x = m 2^(ef - 150)
    unsigned long long u;
    if (s >= 0)
        u = (unsigned long long)m << s;
    else if (s > -32)
        u = (unsigned long long)(m >> (-s));
    else
        u = 0;
    return (b >> 31) ? -(long long)u : (long long)u;
}

// 2^-F as two normal fp32 factors (|F| up to about 250)
__device__ __forceinline__ void fixed_unscale(int F, float &s1, float &s2) {
    const int f1 = F / 2, f2 = F - f1;
    s1 = __int_as_float((127 - f1) << 23);
    s2 = __int_as_float((127 - f2) << 23);
}

// v 2^-F in fp32 (two 32-bit conversions; relative error below 2^-22)
__device__ __forceinline__ float from_fixed(long long v, float s1, float s2) {
    const unsigned long long u = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
    float f = fmaf(__uint2float_rn((unsigned)(u >> 32)), 4294967296.0f,
                   __uint2float_rn((unsigned)(u & 0xffffffffu)));
    f = (f * s1) * s2;
    return v < 0 ? -f : f;
}

}  // namespace dseq
