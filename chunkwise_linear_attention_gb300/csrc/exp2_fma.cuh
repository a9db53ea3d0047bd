// exp2_fma.cuh -- 2^x evaluated on the FMA pipe (integer/fraction split and a
// fitted polynomial), for kernels whose exponentials must be more accurate
// than the special-function unit's (the selective scan's decays).
#pragma once

#include <cuda_runtime.h>

namespace cla {
namespace {

// 2^x on the FMA pipe, for the selective scan's per-step decays
// a = exp(delta A).  Along a
// channel with long memory (decays near 1) the error of every factor of a
// product of many decays adds up, so the hardware approximation (about 2 ulp)
// is not accurate enough there.  Method: split x = k + f with k = rint(x) and
// |f| <= 1/2, evaluate 2^f by a degree-6 polynomial with p(0) = 1 fitted for
// the least maximum relative error (Lawson's reweighted least squares; fit
// error 2e-9, within 0.66 ulp in fp32 Horner form; exp2_poly.py beside this
// file derives the coefficients and checks both figures), and scale by 2^k by
// building the float with exponent field k + 127.
// Results below 2^-126 are returned as 0 (a decay that small is 0 to fp32).
// k is rounded to nearest-even by adding and removing 1.5 * 2^23 (exact for
// |x| <= 2^22, which the clamp ensures), and the low bits of x + 1.5 * 2^23
// are k itself, so the exponent field is one shift-add of them.
// coefficients c1..c6 of 2^f ~ 1 + c1 f + ... + c6 f^6 on [-1/2, 1/2] (exp2_poly.py)
constexpr float kP1 = 6.931471825e-01f, kP2 = 2.402264774e-01f, kP3 = 5.550332367e-02f, kP4 = 9.618437849e-03f,
                kP5 = 1.339887269e-03f, kP6 = 1.535334159e-04f;
__device__ __forceinline__ float exp2_fma(float x) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    x = fminf(fmaxf(x, -127.f), 127.f);
    const float km = x + kMagic;
    const float k = km - kMagic;
    const float f = x - k;
    float p = kP6;
    p = fmaf(p, f, kP5);
    p = fmaf(p, f, kP4);
    p = fmaf(p, f, kP3);
    p = fmaf(p, f, kP2);
    p = fmaf(p, f, kP1);
    p = fmaf(p, f, 1.0f);
    // k + 127 in [0, 254]; 0 gives the float 0 (results below 2^-126 are 0)
    const int e = (__float_as_int(km) - __float_as_int(kMagic)) + 127;
    return p * __int_as_float(e << 23);
}

// The same 2^x on two arguments at once: the paired FP32 instructions
// (add / mul / fma on float2) round each lane exactly as the scalar ones, so
// the results equal exp2_fma's; the instruction count is about halved.
// CLAMP = false: the caller guarantees |x| <= 126 (then the clamp changes nothing).
__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <bool CLAMP = true>
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
    constexpr float kMagic = 12582912.0f;
    if (CLAMP) {
        x.x = fminf(fmaxf(x.x, -127.f), 127.f);
        x.y = fminf(fmaxf(x.y, -127.f), 127.f);
    }
    const float2 km = __fadd2_rn(x, make_float2(kMagic, kMagic));
    const float2 k = __fadd2_rn(km, make_float2(-kMagic, -kMagic));
    const float2 f = __ffma2_rn(k, make_float2(-1.f, -1.f), x);  // x - k, exact
    float2 p = make_float2(kP6, kP6);
    p = __ffma2_rn(p, f, make_float2(kP5, kP5));
    p = __ffma2_rn(p, f, make_float2(kP4, kP4));
    p = __ffma2_rn(p, f, make_float2(kP3, kP3));
    p = __ffma2_rn(p, f, make_float2(kP2, kP2));
    p = __ffma2_rn(p, f, make_float2(kP1, kP1));
    p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
    if (!CLAMP) {
        // |k| <= 126: add k to p's exponent field (p in [2^-1/2, 2^1/2]).  The low bits of
        // km hold k; shifted left by 23 the rest of km's bits leave the word.  Exact, as the
        // multiply by 2^k below is, except that results under 2^-126 come out as subnormals
        // read from the wrong field (absolute error below 2^-126).
        // One integer multiply-add per lane: km * 2^23 + p (the same bits as the shift and add).
        return make_float2(__uint_as_float(mad_u32(__float_as_uint(km.x), 1u << 23, __float_as_uint(p.x))),
                           __uint_as_float(mad_u32(__float_as_uint(km.y), 1u << 23, __float_as_uint(p.y))));
    }
    const int ex = (__float_as_int(km.x) - __float_as_int(kMagic)) + 127;
    const int ey = (__float_as_int(km.y) - __float_as_int(kMagic)) + 127;
    return __fmul2_rn(p, make_float2(__int_as_float(ex << 23), __int_as_float(ey << 23)));
}
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

}  // namespace
}  // namespace cla
