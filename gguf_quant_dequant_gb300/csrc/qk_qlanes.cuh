// qk_qlanes.cuh -- block assembly of the quantizers, one lane per 32
// consecutive weights (a warp covers 32 groups of 32: four super-blocks of a
// K type, or 32 blocks of Q8_0 / Q5_0 / Q4_0).
//
// The quantizers differ only in where the per-group scale s (and min m)
// come from: the plain min/max scheme (plain_params) or the importance-
// weighted search.  From those the block is assembled the same way for both
// (every quotient with the IEEE fp32 division's rounding, every code
// clamp(round-half-away(quotient))):
//   Q4_K, per 32-weight sub-block j: d = fp16(max s / 63), dmin = fp16(max m /
//        63); sc = cr(s / d, 0, 63), m' = cr(m / dmin, 0, 63);
//        q = cr((w + dmin*m') / (d*sc), 0, 15).
//   Q5_K, the same with codes 0..31.
//   Q2_K, per 16 weights: d = fp16(max s / 15), dmin = fp16(max m / 15), 4-bit
//        sc and m', codes 0..3.
//   Q3_K, per 16 weights: d = fp16(max s / 31); sc = cr(s / d, -32, 31);
//        q = cr(w / (d*sc), -4, 3).
//   Q6_K, per 16 weights: d = fp16(max s / 127); sc = cr(s / d, -128, 127);
//        q = cr(w / (d*sc), -32, 31) + 32.
//   Q8_0 / Q5_0 / Q4_0, per 32 weights: d = fp16(s); q = cr(w / d, ...) + 0,
//        16, 8.
// A zero divisor gives the offset code (0 for the codes, scales and mins of
// the types with a min).  Maxima treat NaN as absent; a NaN quotient takes
// the lowest code.  The per-weight codes come from group_codes (one
// reciprocal per group, the division's rounding reproduced exactly).
#pragma once
#include <cuda_fp16.h>

#include "qk_codes.cuh"
#include "qk_formats.cuh"

namespace qk {
namespace ql {

constexpr unsigned kFull = 0xffffffffu;

// Groups of one lane: 1 (32-weight groups) or 2 (16-weight groups).
template <int T> struct LaneGeo {
    static constexpr int G = (T == T_Q6_K || T == T_Q3_K || T == T_Q2_K) ? 16 : 32;
    static constexpr int NG = 32 / G;
    static constexpr bool K = T == T_Q4_K || T == T_Q6_K || T == T_Q5_K || T == T_Q2_K || T == T_Q3_K;
};

// Largest of the values that are > 0 across the 2^k lanes of an aligned
// group (0 when none is): the sequential "if (v > best) best = v" from 0.
template <int LANES>
__device__ __forceinline__ float group_max_pos(float v) {
    float b = v > 0.0f ? v : 0.0f;
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) {
        const float t = __shfl_xor_sync(kFull, b, o);
        b = t > b ? t : b;
    }
    return b;
}

__device__ __forceinline__ uint32_t half_bits(float v) { return (uint32_t)__half_as_ushort(__float2half_rn(v)); }
__device__ __forceinline__ float half_val(uint32_t bits) { return __half2float(__ushort_as_half((unsigned short)bits)); }

// The low bytes of four codes -> a word.
__device__ __forceinline__ uint32_t bytes4(const uint32_t* q) { return pack4(q[0], q[1], q[2], q[3]); }

__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) { *reinterpret_cast<uint16_t*>(p) = (uint16_t)v; }
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

// Codes of a min type's group: cr((w + dm) / ds, 0, TOP) in the low bytes
// of q, 0 when ds <= 0.
template <int N, int TOP>
__device__ __forceinline__ void min_codes(const float* v, float dm, float ds, uint32_t* q) {
    if (ds > 0.0f) {
        float u[N];
        uint32_t c[N];
#pragma unroll
        for (int l = 0; l < N; ++l) u[l] = __fadd_rn(v[l], dm);
        group_codes<N, 0, TOP, 0>(u, ds, c);
#pragma unroll
        for (int l = 0; l < N; ++l) q[l] = c[l];
    } else {
#pragma unroll
        for (int l = 0; l < N; ++l) q[l] = 0;
    }
}
// Codes of a symmetric group: cr(w / ds, LO, HI) + OFF in the low bytes of
// q, OFF when ds == 0.
template <int N, int LO, int HI, int OFF>
__device__ __forceinline__ void sym_codes(const float* v, float ds, uint32_t* q) {
    if (ds != 0.0f) {
        float u[N];
        uint32_t c[N];
#pragma unroll
        for (int l = 0; l < N; ++l) u[l] = v[l];
        group_codes<N, LO, HI, OFF>(u, ds, c);
#pragma unroll
        for (int l = 0; l < N; ++l) q[l] = c[l];
    } else {
#pragma unroll
        for (int l = 0; l < N; ++l) q[l] = (uint32_t)OFF;
    }
}

// The plain scheme's group parameters of the lane's weights:
//   Q4_K / Q5_K / Q2_K: lo = min(0, min w), hi = max w, s = (hi - lo) / (15,
//   31, 3), m = -lo;  Q6_K / Q3_K: s = max|w| / (32, 4);  Q8_0 / Q5_0 / Q4_0:
//   s = max|w| / (127, 15, 7).
// The scans are the sequential "if (x < lo) lo = x" from 0 and "if (x > hi)
// hi = x" from the first weight: fminf / fmaxf chains give the same values
// (both skip NaN), except that hi stays NaN when the first weight is NaN.
// Signed zeros may come out the other way round, which no code or scale
// depends on.
template <int T>
__device__ __forceinline__ void plain_params(const float (&v)[32], float (&s)[2], float (&m)[2]) {
    constexpr int G = LaneGeo<T>::G;
    s[1] = m[1] = m[0] = 0.0f;
#pragma unroll
    for (int e = 0; e < LaneGeo<T>::NG; ++e) {
        if constexpr (T == T_Q4_K || T == T_Q5_K || T == T_Q2_K) {
            constexpr float kDiv = T == T_Q4_K ? 15.0f : (T == T_Q5_K ? 31.0f : 3.0f);
            float lo = 0.0f, hi = v[G * e];
#pragma unroll
            for (int l = 0; l < G; ++l) {
                lo = fminf(lo, v[G * e + l]);
                hi = fmaxf(hi, v[G * e + l]);
            }
            if (v[G * e] != v[G * e]) hi = v[G * e];   // a NaN first weight: the scan keeps it
            s[e] = __fdiv_rn(__fsub_rn(hi, lo), kDiv);
            m[e] = -lo;
        } else {
            constexpr float kDiv = T == T_Q6_K ? 32.0f : T == T_Q3_K ? 4.0f
                                 : T == T_Q8_0 ? 127.0f : (T == T_Q5_0 ? 15.0f : 7.0f);
            float a = 0.0f;
#pragma unroll
            for (int l = 0; l < G; ++l) a = fmaxf(a, fabsf(v[G * e + l]));
            s[e] = __fdiv_rn(a, kDiv);
        }
    }
}

// Q4_K / Q5_K: lane j = lane % 8 holds sub-block j of its super-block
// (bytes at `blk`, 4-byte aligned in shared memory).  Codes: byte 16 + 32c +
// l (Q5_K: 48 + ...) holds sub-block 2c's low four bits of code l (low
// nibble) and sub-block 2c+1's (high nibble); Q5_K's fifth bit of sub-block
// j's code l is bit j of qh[l] (byte 16 + l).  Scales and mins: bytes b,
// 4 + b and 8 + b come from sub-blocks b and b + 4.
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

template <int T>
__device__ __forceinline__ void lane_k45(const float (&v)[32], const float (&sp)[2], const float (&mp)[2], int lane,
                                         bool live, uint8_t* blk) {
    constexpr bool five = T == T_Q5_K;
    const int j = lane & 7;
    const float scf = sp[0], mf = mp[0];
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(scf), 63.0f));
    const uint32_t dmb = half_bits(__fdiv_rn(group_max_pos<8>(mf), 63.0f));
    const float d = half_val(db), dmin = half_val(dmb);
    const int s = d > 0.0f ? cr(__fdiv_rn(scf, d), 0, 63) : 0;
    const int m = dmin > 0.0f ? cr(__fdiv_rn(mf, dmin), 0, 63) : 0;
    const float ds = __fmul_rn(d, (float)s), dm = __fmul_rn(dmin, (float)m);
    uint32_t q[32];
    min_codes<32, five ? 31 : 15>(v, dm, ds, q);
    uint32_t wd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t mine = bytes4(&q[4 * k]) & 0x0F0F0F0Fu;
        const uint32_t odd = __shfl_down_sync(kFull, mine, 1);
        wd[k] = mine | (odd << 4);
    }
    uint32_t qhw = 0;
    if constexpr (five) {
        uint32_t hb = 0;
#pragma unroll
        for (int l = 0; l < 32; ++l) hb |= ((q[l] >> 4) & 1u) << l;
#pragma unroll
        for (int jp = 0; jp < 8; ++jp) {
            const uint32_t t = __shfl_sync(kFull, hb, (lane & ~7) + jp);
            qhw |= spread4((t >> (4 * j)) & 15u) << jp;
        }
    }
    const int s4 = __shfl_down_sync(kFull, s, 4), m4 = __shfl_down_sync(kFull, m, 4);
    if (!live) return;
    constexpr int qs = five ? 48 : 16;
    if ((j & 1) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) st_u32(blk + qs + 16 * j + 4 * k, wd[k]);   // qs + 32 (j / 2)
    }
    if constexpr (five) st_u32(blk + 16 + 4 * j, qhw);
    if (j < 4) {
        blk[4 + j] = (uint8_t)(s | ((s4 >> 4) << 6));
        blk[8 + j] = (uint8_t)(m | ((m4 >> 4) << 6));
        blk[12 + j] = (uint8_t)((s4 & 15) | ((m4 & 15) << 4));
    }
    if (j == 0) st_u32(blk, db | (dmb << 16));
}

// Q2_K / Q3_K: lane j = lane % 8 holds weights 32j .. 32j+31 of its
// super-block (groups 2j, 2j+1), whose 2-bit fields are bits 2(j%4).. of code
// bytes 32(j/4) .. +31: the four lanes that share those bytes OR their
// fields together.  Q3_K's mask bit of weight 32j + l is bit j of hmask[l]
// (gathered as Q5_K's fifth bits).  `blk` is 4-byte (Q2_K) or 2-byte (Q3_K)
// aligned.
__device__ __forceinline__ void plane_words(const uint32_t (&q)[32], int j, uint32_t (&wd)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t w = bytes4(&q[4 * k]) << (2 * (j & 3));
        w |= __shfl_xor_sync(kFull, w, 1);
        w |= __shfl_xor_sync(kFull, w, 2);
        wd[k] = w;
    }
}

__device__ __forceinline__ void lane_q2k(const float (&v)[32], const float (&scf)[2], const float (&mf)[2], int lane,
                                         bool live, uint8_t* blk) {
    const int j = lane & 7;
    const float c0 = scf[0] > 0.0f ? scf[0] : 0.0f, c1 = scf[1] > 0.0f ? scf[1] : 0.0f;
    const float n0 = mf[0] > 0.0f ? mf[0] : 0.0f, n1 = mf[1] > 0.0f ? mf[1] : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 15.0f));
    const uint32_t dmb = half_bits(__fdiv_rn(group_max_pos<8>(n1 > n0 ? n1 : n0), 15.0f));
    const float d = half_val(db), dmin = half_val(dmb);
    uint32_t q[32];
    uint32_t sm = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int s = d > 0.0f ? cr(__fdiv_rn(scf[e], d), 0, 15) : 0;
        const int m = dmin > 0.0f ? cr(__fdiv_rn(mf[e], dmin), 0, 15) : 0;
        const float ds = __fmul_rn(d, (float)s), dm = __fmul_rn(dmin, (float)m);
        min_codes<16, 3>(v + 16 * e, dm, ds, q + 16 * e);
        sm |= (uint32_t)(s | (m << 4)) << (8 * e);
    }
    uint32_t wd[8];
    plane_words(q, j, wd);
    if (!live) return;
    if ((j & 3) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) st_u32(blk + 16 + 32 * (j >> 2) + 4 * k, wd[k]);
    }
    st_u16(blk + 2 * j, sm);
    if (j == 0) st_u32(blk + 80, db | (dmb << 16));
}

__device__ __forceinline__ void lane_q3k(const float (&v)[32], const float (&sf)[2], int lane, bool live,
                                         uint8_t* blk) {
    const int j = lane & 7;
    const float c0 = sf[0] > 0.0f ? sf[0] : 0.0f, c1 = sf[1] > 0.0f ? sf[1] : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 31.0f));
    const float d = half_val(db);
    uint32_t q[32], lo2[32];
    int sv[2];
    uint32_t hb = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int s = d > 0.0f ? cr(__fdiv_rn(sf[e], d), -32, 31) : 0;
        const float ds = __fmul_rn(d, (float)s);
        sym_codes<16, -4, 3, 0>(v + 16 * e, ds, q + 16 * e);
        sv[e] = s + 32;
    }
    // A code in -4..3 as a byte: its two low bits are q (q >= 0) or q + 4,
    // and bit 2 is set exactly when q < 0.
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        lo2[l] = q[l] & 3u;
        hb |= (((q[l] >> 2) & 1u) ^ 1u) << l;
    }
    uint32_t wd[8];
    plane_words(lo2, j, wd);
    // hmask bytes 4j .. 4j+3: bit j' of byte l from lane j'.
    uint32_t hmw = 0;
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
        const uint32_t t = __shfl_sync(kFull, hb, (lane & ~7) + jp);
        hmw |= spread4((t >> (4 * j)) & 15u) << jp;
    }
    // Scales of groups g = 2j + e (value + 32): low nibble g/8 of byte g%8
    // (lanes j and j + 4 share bytes 2j, 2j+1), high bits at 2(g/4) of byte
    // 8 + g%4 (all eight lanes share bytes 8..11).
    const int up0 = __shfl_down_sync(kFull, sv[0], 4), up1 = __shfl_down_sync(kFull, sv[1], 4);
    uint32_t hi2 = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) hi2 |= (uint32_t)(sv[e] >> 4) << (8 * (2 * (j & 1) + e) + 2 * (j >> 1));
    hi2 |= __shfl_xor_sync(kFull, hi2, 1);
    hi2 |= __shfl_xor_sync(kFull, hi2, 2);
    hi2 |= __shfl_xor_sync(kFull, hi2, 4);
    if (!live) return;
    if ((j & 3) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            st_u16(blk + 32 + 32 * (j >> 2) + 4 * k, wd[k]);
            st_u16(blk + 34 + 32 * (j >> 2) + 4 * k, wd[k] >> 16);
        }
    }
    st_u16(blk + 4 * j, hmw);
    st_u16(blk + 4 * j + 2, hmw >> 16);
    if (j < 4)
        st_u16(blk + 96 + 2 * j, (uint32_t)((sv[0] & 15) | ((up0 & 15) << 4)) |
                                     ((uint32_t)((sv[1] & 15) | ((up1 & 15) << 4)) << 8));
    if (j == 0) {
        st_u16(blk + 104, hi2);
        st_u16(blk + 106, hi2 >> 16);
        st_u16(blk + 108, db);
    }
}

// Q6_K: lane t = lane % 8 holds weights 32t .. 32t+31 of its super-block,
// i.e. half h = t / 4, group g = t % 4, and scale groups 2t, 2t+1.  Bytes at
// `blk` (2-byte aligned).
__device__ __forceinline__ void lane_q6k(const float (&v)[32], const float (&sf)[2], int lane, bool live,
                                         uint8_t* blk) {
    const int t = lane & 7, h = t >> 2, g = t & 3;
    const float c0 = sf[0] > 0.0f ? sf[0] : 0.0f, c1 = sf[1] > 0.0f ? sf[1] : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 127.0f));
    const float d = half_val(db);
    const int s0 = d > 0.0f ? cr(__fdiv_rn(sf[0], d), -128, 127) : 0;
    const int s1 = d > 0.0f ? cr(__fdiv_rn(sf[1], d), -128, 127) : 0;
    const float ds0 = __fmul_rn(d, (float)s0), ds1 = __fmul_rn(d, (float)s1);
    uint32_t q[32];
    sym_codes<16, -32, 31, 32>(v, ds0, q);
    sym_codes<16, -32, 31, 32>(v + 16, ds1, q + 16);
    // Low 4 bits: ql[64h + 32(g & 1) + l], low nibble for g < 2, high for g >= 2
    // (lanes t and t + 2 share the bytes).  High 2 bits: qh[32h + l] bits 2g,
    // 2g + 1 (the four lanes of a half share the bytes).
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w4 = bytes4(&q[4 * k]);   // codes 0..63
        const uint32_t l4 = w4 & 0x0F0F0F0Fu;
        uint32_t h2 = (w4 >> 4) & 0x03030303u;
        const uint32_t up = __shfl_down_sync(kFull, l4, 2);
        lo[k] = l4 | (up << 4);
        h2 <<= 2 * g;
        h2 |= __shfl_xor_sync(kFull, h2, 1);
        h2 |= __shfl_xor_sync(kFull, h2, 2);
        hi[k] = h2;
    }
    if (!live) return;
    if (g < 2) {
        uint8_t* p = blk + 64 * h + 32 * g;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            st_u16(p + 4 * k, lo[k] & 0xFFFFu);
            st_u16(p + 4 * k + 2, lo[k] >> 16);
        }
    }
    if (g == 0) {
        uint8_t* p = blk + 128 + 32 * h;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            st_u16(p + 4 * k, hi[k] & 0xFFFFu);
            st_u16(p + 4 * k + 2, hi[k] >> 16);
        }
    }
    st_u16(blk + 192 + 2 * t, (uint32_t)(uint8_t)(int8_t)s0 | ((uint32_t)(uint8_t)(int8_t)s1 << 8));
    if (t == 0) st_u16(blk + 208, db);
}

// Q8_0 / Q5_0 / Q4_0: the lane holds one whole block (bytes at `blk`, 2-byte
// aligned).
template <int T>
__device__ __forceinline__ void lane_small(const float (&v)[32], float s, bool live, uint8_t* blk) {
    constexpr int kOff = T == T_Q8_0 ? 0 : (T == T_Q5_0 ? 16 : 8);
    constexpr int kLo = T == T_Q8_0 ? -128 : 0;
    constexpr int kHi = T == T_Q8_0 ? 127 : (T == T_Q5_0 ? 31 : 15);
    const uint32_t db = half_bits(s);
    const float d = half_val(db);
    uint32_t q[32];
    if (d > 0.0f) {
        sym_codes<32, kLo - kOff, kHi - kOff, kOff>(v, d, q);
    } else {
#pragma unroll
        for (int l = 0; l < 32; ++l) q[l] = (uint32_t)kOff;
    }
    if (!live) return;
    st_u16(blk, db);
    if constexpr (T == T_Q8_0) {
#pragma unroll
        for (int l = 0; l < 32; l += 4) {
            const uint32_t w4 = bytes4(&q[l]);
            st_u16(blk + 2 + l, w4 & 0xFFFFu);
            st_u16(blk + 4 + l, w4 >> 16);
        }
    } else {
        uint8_t* qs = blk + (T == T_Q5_0 ? 6 : 2);
        if constexpr (T == T_Q5_0) {
            uint32_t qh = 0;
#pragma unroll
            for (int l = 0; l < 32; ++l) qh |= ((q[l] >> 4) & 1u) << l;
            st_u16(blk + 2, qh & 0xFFFFu);
            st_u16(blk + 4, qh >> 16);
        }
        // Byte j: element j in the low nibble, element j + 16 in the high one.
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const uint32_t w4 = (bytes4(&q[j]) & 0x0F0F0F0Fu) | ((bytes4(&q[j + 16]) & 0x0F0F0F0Fu) << 4);
            st_u16(qs + j, w4 & 0xFFFFu);
            st_u16(qs + j + 2, w4 >> 16);
        }
    }
}

// The lane's part of its block from the group parameters (s, m); `blk` is
// the block's bytes (the lane's own for Q8_0 / Q5_0 / Q4_0, its
// super-block's for the K types).
template <int T>
__device__ __forceinline__ void assemble(const float (&v)[32], const float (&s)[2], const float (&m)[2], int lane,
                                         bool live, uint8_t* blk) {
    if constexpr (T == T_Q4_K || T == T_Q5_K) lane_k45<T>(v, s, m, lane, live, blk);
    else if constexpr (T == T_Q2_K) lane_q2k(v, s, m, lane, live, blk);
    else if constexpr (T == T_Q3_K) lane_q3k(v, s, lane, live, blk);
    else if constexpr (T == T_Q6_K) lane_q6k(v, s, lane, live, blk);
    else lane_small<T>(v, s[0], live, blk);
}

}  // namespace ql
}  // namespace qk
