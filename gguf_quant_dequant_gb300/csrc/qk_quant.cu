// qk_quant.cu -- the write side: fp32 weights -> packed GGUF blocks.
//
// The pages name the k-quant quantizer ("Quantization formats", the
// quantize_row_q4_K reference) without giving it; this is the plain min/max
// scheme, every quotient an IEEE fp32 division and every code
// clamp(round-half-away(quotient)), in this order:
//   Q4_K, per 32-weight sub-block j: lo = min(0, min w), hi = max w,
//        sc_f = (hi - lo) / 15, m_f = -lo; d = fp16(max sc_f / 63),
//        dmin = fp16(max m_f / 63); sc = cr(sc_f / d, 0, 63),
//        m = cr(m_f / dmin, 0, 63); q = cr((w + dmin*m) / (d*sc), 0, 15).
//   Q5_K, the same with 31 in place of 15 (codes 0..31).
//   Q2_K, per 16 weights: the Q4_K scheme with 3 steps, d = fp16(max sc_f /
//        15), dmin = fp16(max m_f / 15), 4-bit sc and m, codes 0..3.
//   Q3_K, per 16 weights: s = max|w| / 4; d = fp16(max s / 31);
//        sc = cr(s / d, -32, 31); q = cr(w / (d*sc), -4, 3).
//   Q6_K, per 16 weights: s = max|w| / 32; d = fp16(max s / 127);
//        sc = cr(s / d, -128, 127); q = cr(w / (d*sc), -32, 31) + 32.
//   Q8_0 / Q5_0 / Q4_0, per 32 weights: d = fp16(max|w| / 127, 15, 7);
//        q = cr(w / d, ...) + 0, 16, 8.
// A zero divisor gives the offset code (0 for Q4_K's codes, scales and mins).
// Maxima treat NaN as absent; a NaN quotient takes the lowest code.
//
// One warp quantizes 32 consecutive 32-weight groups (1024 weights): four
// super-blocks for the K types, 32 blocks otherwise.  Each lane loads its 32
// weights (eight 16-byte streaming loads), the per-super-block maxima and the
// nibble / bit packing cross lanes with shuffles, and the packed bytes are
// staged in shared memory and written out as 4-byte words.  The work is
// HBM-bound: 4 bytes read and BB/BE bytes written per weight.
#include <cuda_fp16.h>

#include "qk_formats.cuh"
#include "qk_internal.h"

namespace qk {
namespace qz {

constexpr int kWarps = 8;                    // per CTA
constexpr int kBufWords = 32 * 34 / 4;      // largest warp output: 32 Q8_0 blocks = 1088 bytes
constexpr unsigned kFull = 0xffffffffu;

// clamp(round(v), lo, hi): round half away from zero, clamp as a float (a
// NaN goes to lo), then convert.
__device__ __forceinline__ int cr(float v, int lo, int hi) {
    float r = roundf(v);
    if (!(r >= (float)lo)) r = (float)lo;
    if (r > (float)hi) r = (float)hi;
    return (int)r;
}

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

// Four codes (one per byte, low bits) -> a word.
__device__ __forceinline__ uint32_t bytes4(const int* q) {
    return (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2] << 16) | ((uint32_t)q[3] << 24);
}

__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) { *reinterpret_cast<uint16_t*>(p) = (uint16_t)v; }
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

// Q4_K: lane j = lane % 8 holds sub-block j of super-block `sb` (bytes at
// `blk`, 4-byte aligned in shared memory).
__device__ __forceinline__ void lane_q4k(const float (&v)[32], int lane, bool live, uint8_t* blk) {
    const int j = lane & 7;
    float lo = 0.0f, hi = v[0];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        if (v[l] < lo) lo = v[l];
        if (v[l] > hi) hi = v[l];
    }
    const float scf = __fdiv_rn(__fsub_rn(hi, lo), 15.0f), mf = -lo;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(scf), 63.0f));
    const uint32_t dmb = half_bits(__fdiv_rn(group_max_pos<8>(mf), 63.0f));
    const float d = half_val(db), dmin = half_val(dmb);
    const int s = d > 0.0f ? cr(__fdiv_rn(scf, d), 0, 63) : 0;
    const int m = dmin > 0.0f ? cr(__fdiv_rn(mf, dmin), 0, 63) : 0;
    const float ds = __fmul_rn(d, (float)s), dm = __fmul_rn(dmin, (float)m);
    int q[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) q[l] = ds > 0.0f ? cr(__fdiv_rn(__fadd_rn(v[l], dm), ds), 0, 15) : 0;
    // Codes: byte 16 + 32c + l holds sub-block 2c's code l (low nibble) and
    // sub-block 2c+1's (high nibble).
    uint32_t wd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t mine = bytes4(&q[4 * k]);
        const uint32_t odd = __shfl_down_sync(kFull, mine, 1);
        wd[k] = mine | (odd << 4);
    }
    // Scales and mins: bytes b, 4 + b and 8 + b come from sub-blocks b and b + 4.
    const int s4 = __shfl_down_sync(kFull, s, 4), m4 = __shfl_down_sync(kFull, m, 4);
    if (!live) return;
    if ((j & 1) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) st_u32(blk + 16 + 16 * j + 4 * k, wd[k]);   // 16 + 32 (j / 2)
    }
    if (j < 4) {
        blk[4 + j] = (uint8_t)(s | ((s4 >> 4) << 6));
        blk[8 + j] = (uint8_t)(m | ((m4 >> 4) << 6));
        blk[12 + j] = (uint8_t)((s4 & 15) | ((m4 & 15) << 4));
    }
    if (j == 0) st_u32(blk, db | (dmb << 16));
}

// Q5_K: as Q4_K with 31 steps; the low 4 bits of each code go where Q4_K's
// codes go (from byte 48), the fifth bit of sub-block j's code l is bit j of
// qh[l] (byte 16 + l).  Lane j writes qh bytes 4j .. 4j+3, gathering bit j'
// of each from lane j' of its super-block.
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

__device__ __forceinline__ void lane_q5k(const float (&v)[32], int lane, bool live, uint8_t* blk) {
    const int j = lane & 7;
    float lo = 0.0f, hi = v[0];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        if (v[l] < lo) lo = v[l];
        if (v[l] > hi) hi = v[l];
    }
    const float scf = __fdiv_rn(__fsub_rn(hi, lo), 31.0f), mf = -lo;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(scf), 63.0f));
    const uint32_t dmb = half_bits(__fdiv_rn(group_max_pos<8>(mf), 63.0f));
    const float d = half_val(db), dmin = half_val(dmb);
    const int s = d > 0.0f ? cr(__fdiv_rn(scf, d), 0, 63) : 0;
    const int m = dmin > 0.0f ? cr(__fdiv_rn(mf, dmin), 0, 63) : 0;
    const float ds = __fmul_rn(d, (float)s), dm = __fmul_rn(dmin, (float)m);
    int q[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) q[l] = ds > 0.0f ? cr(__fdiv_rn(__fadd_rn(v[l], dm), ds), 0, 31) : 0;
    uint32_t wd[8], hb = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t mine = bytes4(&q[4 * k]) & 0x0F0F0F0Fu;
        const uint32_t odd = __shfl_down_sync(kFull, mine, 1);
        wd[k] = mine | (odd << 4);
    }
#pragma unroll
    for (int l = 0; l < 32; ++l) hb |= (uint32_t)(q[l] >> 4) << l;
    uint32_t qhw = 0;
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
        const uint32_t t = __shfl_sync(kFull, hb, (lane & ~7) + jp);
        qhw |= spread4((t >> (4 * j)) & 15u) << jp;
    }
    const int s4 = __shfl_down_sync(kFull, s, 4), m4 = __shfl_down_sync(kFull, m, 4);
    if (!live) return;
    if ((j & 1) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) st_u32(blk + 48 + 16 * j + 4 * k, wd[k]);   // 48 + 32 (j / 2)
    }
    st_u32(blk + 16 + 4 * j, qhw);
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
__device__ __forceinline__ void plane_words(const int (&q)[32], int j, uint32_t (&wd)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t w = bytes4(&q[4 * k]) << (2 * (j & 3));
        w |= __shfl_xor_sync(kFull, w, 1);
        w |= __shfl_xor_sync(kFull, w, 2);
        wd[k] = w;
    }
}

__device__ __forceinline__ void lane_q2k(const float (&v)[32], int lane, bool live, uint8_t* blk) {
    const int j = lane & 7;
    float scf[2], mf[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float lo = 0.0f, hi = v[16 * e];
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            if (v[16 * e + l] < lo) lo = v[16 * e + l];
            if (v[16 * e + l] > hi) hi = v[16 * e + l];
        }
        scf[e] = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
        mf[e] = -lo;
    }
    const float c0 = scf[0] > 0.0f ? scf[0] : 0.0f, c1 = scf[1] > 0.0f ? scf[1] : 0.0f;
    const float n0 = mf[0] > 0.0f ? mf[0] : 0.0f, n1 = mf[1] > 0.0f ? mf[1] : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 15.0f));
    const uint32_t dmb = half_bits(__fdiv_rn(group_max_pos<8>(n1 > n0 ? n1 : n0), 15.0f));
    const float d = half_val(db), dmin = half_val(dmb);
    int q[32];
    uint32_t sm = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int s = d > 0.0f ? cr(__fdiv_rn(scf[e], d), 0, 15) : 0;
        const int m = dmin > 0.0f ? cr(__fdiv_rn(mf[e], dmin), 0, 15) : 0;
        const float ds = __fmul_rn(d, (float)s), dm = __fmul_rn(dmin, (float)m);
#pragma unroll
        for (int l = 0; l < 16; ++l)
            q[16 * e + l] = ds > 0.0f ? cr(__fdiv_rn(__fadd_rn(v[16 * e + l], dm), ds), 0, 3) : 0;
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

__device__ __forceinline__ void lane_q3k(const float (&v)[32], int lane, bool live, uint8_t* blk) {
    const int j = lane & 7;
    float sf[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float a = 0.0f;
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const float x = fabsf(v[16 * e + l]);
            if (x > a) a = x;
        }
        sf[e] = __fdiv_rn(a, 4.0f);
    }
    const float c0 = sf[0] > 0.0f ? sf[0] : 0.0f, c1 = sf[1] > 0.0f ? sf[1] : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 31.0f));
    const float d = half_val(db);
    int q[32], lo2[32], sv[2];
    uint32_t hb = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int s = d > 0.0f ? cr(__fdiv_rn(sf[e], d), -32, 31) : 0;
        const float ds = __fmul_rn(d, (float)s);
#pragma unroll
        for (int l = 0; l < 16; ++l) q[16 * e + l] = ds != 0.0f ? cr(__fdiv_rn(v[16 * e + l], ds), -4, 3) : 0;
        sv[e] = s + 32;
    }
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        lo2[l] = q[l] >= 0 ? q[l] : q[l] + 4;
        hb |= (uint32_t)(q[l] >= 0) << l;
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

// Q6_K: lane t = lane % 8 holds weights 32t .. 32t+31 of super-block `sb`,
// i.e. half h = t / 4, group g = t % 4, and scale groups 2t, 2t+1.  Bytes at
// `blk` (2-byte aligned).
__device__ __forceinline__ void lane_q6k(const float (&v)[32], int lane, bool live, uint8_t* blk) {
    const int t = lane & 7, h = t >> 2, g = t & 3;
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        const float x0 = fabsf(v[l]), x1 = fabsf(v[16 + l]);
        if (x0 > a0) a0 = x0;
        if (x1 > a1) a1 = x1;
    }
    const float sf0 = __fdiv_rn(a0, 32.0f), sf1 = __fdiv_rn(a1, 32.0f);
    const float c0 = sf0 > 0.0f ? sf0 : 0.0f, c1 = sf1 > 0.0f ? sf1 : 0.0f;
    const uint32_t db = half_bits(__fdiv_rn(group_max_pos<8>(c1 > c0 ? c1 : c0), 127.0f));
    const float d = half_val(db);
    const int s0 = d > 0.0f ? cr(__fdiv_rn(sf0, d), -128, 127) : 0;
    const int s1 = d > 0.0f ? cr(__fdiv_rn(sf1, d), -128, 127) : 0;
    const float ds0 = __fmul_rn(d, (float)s0), ds1 = __fmul_rn(d, (float)s1);
    int q[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const float ds = l < 16 ? ds0 : ds1;
        q[l] = ds != 0.0f ? cr(__fdiv_rn(v[l], ds), -32, 31) + 32 : 32;
    }
    // Low 4 bits: ql[64h + 32(g & 1) + l], low nibble for g < 2, high for g >= 2
    // (lanes t and t + 2 share the bytes).  High 2 bits: qh[32h + l] bits 2g,
    // 2g + 1 (the four lanes of a half share the bytes).
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int* qk4 = &q[4 * k];
        uint32_t l4 = 0, h2 = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            l4 |= (uint32_t)(qk4[b] & 15) << (8 * b);
            h2 |= (uint32_t)((qk4[b] >> 4) & 3) << (8 * b);
        }
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
__device__ __forceinline__ void lane_small(const float (&v)[32], bool live, uint8_t* blk) {
    constexpr float kDiv = T == T_Q8_0 ? 127.0f : (T == T_Q5_0 ? 15.0f : 7.0f);
    constexpr int kOff = T == T_Q8_0 ? 0 : (T == T_Q5_0 ? 16 : 8);
    constexpr int kLo = T == T_Q8_0 ? -128 : 0;
    constexpr int kHi = T == T_Q8_0 ? 127 : (T == T_Q5_0 ? 31 : 15);
    float a = 0.0f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const float x = fabsf(v[l]);
        if (x > a) a = x;
    }
    const uint32_t db = half_bits(__fdiv_rn(a, kDiv));
    const float d = half_val(db);
    int q[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) q[l] = d > 0.0f ? cr(__fdiv_rn(v[l], d), kLo - kOff, kHi - kOff) + kOff : kOff;
    if (!live) return;
    st_u16(blk, db);
    if constexpr (T == T_Q8_0) {
#pragma unroll
        for (int l = 0; l < 32; l += 2) st_u16(blk + 2 + l, (uint32_t)(q[l] & 0xFF) | ((uint32_t)(q[l + 1] & 0xFF) << 8));
    } else {
        uint8_t* qs = blk + (T == T_Q5_0 ? 6 : 2);
        if constexpr (T == T_Q5_0) {
            uint32_t qh = 0;
#pragma unroll
            for (int l = 0; l < 32; ++l) qh |= (uint32_t)((q[l] >> 4) & 1) << l;
            st_u16(blk + 2, qh & 0xFFFFu);
            st_u16(blk + 4, qh >> 16);
        }
        // Byte j: element j in the low nibble, element j + 16 in the high one.
#pragma unroll
        for (int j = 0; j < 16; j += 2)
            st_u16(qs + j, (uint32_t)((q[j] & 15) | ((q[j + 16] & 15) << 4)) |
                               ((uint32_t)((q[j + 1] & 15) | ((q[j + 17] & 15) << 4)) << 8));
    }
}

template <int T>
__global__ void __launch_bounds__(kWarps * 32) quantize_kernel(const float* __restrict__ w, int64_t ngroups,
                                                                uint8_t* __restrict__ out) {
    constexpr bool kK = T == T_Q4_K || T == T_Q6_K || T == T_Q5_K || T == T_Q2_K || T == T_Q3_K;
    constexpr int kBB = Fmt<T>::BB;
    __shared__ uint32_t buf[kWarps][kBufWords];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g0 = ((int64_t)blockIdx.x * kWarps + warp) * 32;   // first 32-weight group of this warp
    if (g0 >= ngroups) return;   // whole warp
    const int64_t left = ngroups - g0;
    const int ng = left < 32 ? (int)left : 32;   // a multiple of 8 for the K types
    const bool live = lane < ng;
    float v[32];
    if (live) {
        const float4* src = reinterpret_cast<const float4*>(w + (g0 + lane) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = __ldcs(src + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int l = 0; l < 32; ++l) v[l] = 0.0f;
    }
    uint8_t* sb = reinterpret_cast<uint8_t*>(buf[warp]);
    if constexpr (T == T_Q4_K) lane_q4k(v, lane, live, sb + (lane >> 3) * kBB);
    else if constexpr (T == T_Q5_K) lane_q5k(v, lane, live, sb + (lane >> 3) * kBB);
    else if constexpr (T == T_Q2_K) lane_q2k(v, lane, live, sb + (lane >> 3) * kBB);
    else if constexpr (T == T_Q3_K) lane_q3k(v, lane, live, sb + (lane >> 3) * kBB);
    else if constexpr (T == T_Q6_K) lane_q6k(v, lane, live, sb + (lane >> 3) * kBB);
    else lane_small<T>(v, live, sb + lane * kBB);
    __syncwarp();
    // This warp's bytes: [g0 * BB / groups-per-block, + nb), 4-byte aligned
    // (every warp but the last covers a multiple of 4 bytes).
    const int64_t ob = (kK ? g0 / 8 : g0) * kBB;
    const int nb = (kK ? ng / 8 : ng) * kBB;
    uint8_t* dst = out + ob;
    for (int i = lane; i < nb / 4; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = buf[warp][i];
    if (lane < (nb & 3)) dst[(nb & ~3) + lane] = sb[(nb & ~3) + lane];
}

template <int T>
static cudaError_t launch_t(const float* w, int64_t ngroups, uint8_t* out, cudaStream_t s) {
    const int64_t warps = (ngroups + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quantize_kernel<T><<<(unsigned)blocks, kWarps * 32, 0, s>>>(w, ngroups, out);
    return cudaGetLastError();
}

}  // namespace qz

cudaError_t launch_quantize(int type, const float* w, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t s) {
    const int64_t ngroups = rows * (cols / 32);
    switch (type) {
    case T_Q4_K: return qz::launch_t<T_Q4_K>(w, ngroups, out, s);
    case T_Q6_K: return qz::launch_t<T_Q6_K>(w, ngroups, out, s);
    case T_Q8_0: return qz::launch_t<T_Q8_0>(w, ngroups, out, s);
    case T_Q5_0: return qz::launch_t<T_Q5_0>(w, ngroups, out, s);
    case T_Q4_0: return qz::launch_t<T_Q4_0>(w, ngroups, out, s);
    case T_Q5_K: return qz::launch_t<T_Q5_K>(w, ngroups, out, s);
    case T_Q2_K: return qz::launch_t<T_Q2_K>(w, ngroups, out, s);
    case T_Q3_K: return qz::launch_t<T_Q3_K>(w, ngroups, out, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
