// qk_codes.cuh -- the quantizers' integer codes q = clamp(round(u / d), lo,
// hi) (round half away from zero, IEEE fp32 quotient, a NaN quotient giving
// lo), for a group of values that share one divisor d, without a division
// per value.
//
// Each value is multiplied by an approximate reciprocal of d (the hardware
// reciprocal, relative error at most one unit in the last place), clamped
// to [lo, hi] and rounded to the nearest integer by an add of 1.5 * 2^23.
// For an unclamped y = u * (1/d)~ the distance to the correctly rounded
// quotient fl(u / d) is below |u / d| (2^-22 + 2^-24 + 2^-24) < |y| 2^-21;
// when y lies farther than |y| 2^-20 from every half-integer, its code equals
// the one the division gives (and no exact tie can occur).  A clamped y is
// the same code as its quotient's (both are beyond the end of the range or
// within the error of it, far less than a half).  A NaN or infinite
// numerator gives the division's code too (lo for NaN, the end of its sign
// for an infinity).  A group with a value that fails the test (a value does
// so with probability about |y| 2^-19), or whose d is not a normal number
// with 1/d normal, is computed again with the division.
#pragma once
#include <cstdint>

namespace qk {

// clamp(round(v), lo, hi): round half away from zero, clamp as a float (a
// NaN goes to lo), then convert.
__device__ __forceinline__ int cr(float v, int lo, int hi) {
    float r = roundf(v);
    if (!(r >= (float)lo)) r = (float)lo;
    if (r > (float)hi) r = (float)hi;
    return (int)r;
}

// An approximation of 1/d good to one unit in the last place (the hardware
// reciprocal), usable for the codes only when rcp_usable(d): 1/d safely
// inside the normal range (not for a zero, subnormal, huge, infinite or NaN
// d; those take the division).
__device__ __forceinline__ float approx_rcp(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}
__device__ __forceinline__ bool rcp_usable(float d) {
    const float ad = fabsf(d);
    return ad >= 0x1p-120f && ad <= 0x1p120f;
}

// The codes cr(u[l] / d, LO, HI) + OFF of N values (d > 0 or d < 0,
// finite, non-zero; any other d is the caller's special case), as the low
// byte of cb[l] (two's complement for a negative code; the higher bits are
// not defined).  For a code range within +-16 the test takes the group's
// largest rounding distance against the bound at |y| = 16 (one instruction
// fewer per value; a group then fails with probability about 32 N 2^-20).
template <int N, int LO, int HI, int OFF>
__device__ __forceinline__ void group_codes(const float (&u)[N], float d, uint32_t (&cb)[N]) {
    constexpr int kM = (-LO > HI) ? -LO : HI;
    constexpr bool kWide = kM > 16;
    const float rd = approx_rcp(d);
    const float magic = 12582912.0f + (float)OFF;   // 1.5 * 2^23 + OFF
    float worst = 0.0f;
#pragma unroll
    for (int l = 0; l < N; ++l) {
        const float y = fminf(fmaxf(__fmul_rn(u[l], rd), (float)LO), (float)HI);
        const float r = __fadd_rn(y, magic);
        cb[l] = __float_as_uint(r);
        const float dist = fabsf(__fsub_rn(y, __fsub_rn(r, magic)));
        worst = fmaxf(worst, kWide ? __fmaf_rn(fabsf(y), 0x1p-20f, dist) : dist);
    }
    const float limit = kWide ? 0.5f : 0.5f - (float)kM * 0x1p-20f;
    if (!(rcp_usable(d) && worst < limit)) {
#pragma unroll
        for (int l = 0; l < N; ++l) cb[l] = (uint32_t)(cr(__fdiv_rn(u[l], d), LO, HI) + OFF);
    }
}

// Bytes 0 of a, b, c, e as one word (a in the low byte).
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t e) {
    return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, e, 0x0040u), 0x5410u);
}

}  // namespace qk
