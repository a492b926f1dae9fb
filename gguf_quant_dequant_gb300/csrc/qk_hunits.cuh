// qk_hunits.cuh -- per-type unit decoders of the tensor-core decode GEMV.
//
// Arithmetic ("Local LLM inference", "The mmap backend": the blocks are
// dequantized inside the dot product).  The dot products run on the fp16
// warp MMA (mma.sync m16n8k16, fp32 accumulation):
//   * A (16 weight rows x 16 k) holds integer codes minus an integer offset,
//     q - o, exact in fp16 (|q - o| <= 63).  A code is placed in the mantissa
//     of a magic fp16 value (1024 + q, or 64 + q when the code sits in the
//     high nibble of its byte) and the offset is removed with one exact
//     fp16 add of -(1024 + o) or -(64 + o).
//   * B (16 k x 8 columns) holds x as two fp16 terms per element,
//     x' = x * 2^-e (e chosen per 32-element block so that x' fits fp16),
//     hi = fp16(x'), lo = fp16(x' - hi): about 22 significant bits relative
//     to each element, whatever the other elements of the block are.
//   * The code offset o is the type's own (Q6_K 32, Q5_0 16, Q4_0 8, Q3_K 4,
//     Q8_0 0).  For the types with a min (Q4_K, Q5_K, Q2_K),
//     w = d*sc*q - dmin*m = d*sc*(q - o) - r with o = the code nearest to
//     dmin*m / (d*sc) and r = dmin*m - d*sc*o; r is applied to the fp32 sum
//     of the block's x.  A weight that is exactly zero therefore contributes
//     exactly zero (its q - o is 0 and r is 0), and |r| never exceeds any
//     |w| of the group, so no term of the sum is larger than the weights and
//     activations it stands for (no cancellation of large terms).
// Work of one warp on one unit (16 rows x 256 weights): thread (g, t) of the
// MMA layout (g = lane / 4, t = lane % 4) supplies the A fragments of rows
// g and g + 8 for the two 32-weight x-blocks X0(t), X1(t) of its "group" t;
// the B columns 2t (hi) and 2t + 1 (lo) are non-zero only at the k slots of
// group t, so the C columns of thread t hold exactly the sums of its own
// group and the scales of a group are applied by the thread that decoded it.
// Within a group, step i of an x-block uses code word i (weights 4i .. 4i+3
// of the block): bytes 0 and 2 form the k pair (2t, 2t+1), bytes 1 and 3 the
// pair (2t+8, 2t+9); the prepared x uses the same order.
#pragma once
#include <cstdint>

#include "qk_formats.cuh"

namespace qk {
namespace hm {

// D = A * B + D, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a & m) | c and (a & m) ^ c as one three-input logic instruction each (the
// compiler otherwise emits two).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
    return d;
}

// Two fp16 adds (round to nearest; exact for the integer operands used here).
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// N little-endian words from a 2-byte-aligned shared address: aligned loads
// joined by funnel shifts (the slot has slack past the segment).
template <int N>
__device__ __forceinline__ void words_a2(const uint8_t* p, uint32_t (&w)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8;
    uint32_t prev = lds32(b);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t next = lds32(b + 4 * (i + 1));
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

// Byte k of v as an exact fp32 (0..255).
__device__ __forceinline__ float ubyte_f(uint32_t v, int k) {
    return __uint_as_float(__byte_perm(v, 0x4B000000u, (uint32_t)k | 0x7440u)) - 8388608.0f;
}

// half2 with both halves = the fp16 bit pattern h.
__device__ __forceinline__ uint32_t dup16(uint32_t h) { return h * 0x00010001u; }

// half2 (v, v) from an fp32 value exactly representable in fp16.
__device__ __forceinline__ uint32_t h2dup(float v) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    return d;
}

// The B fragments of one thread for one x-block: 8 words x (b0, b1).
struct XB {
    uint32_t b[16];
};
__device__ __forceinline__ void load_xb(const uint8_t* p, XB& x) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 v = lds128(p + 16 * q);
        x.b[4 * q] = v.x;
        x.b[4 * q + 1] = v.y;
        x.b[4 * q + 2] = v.z;
        x.b[4 * q + 3] = v.w;
    }
}

// Every unit decoder takes the unit's bytes of rows g (r0) and g + 8 (r1),
// the B fragments of the thread's x-blocks (zero unless the thread owns the
// B column), the sums and scales of its group's x-blocks, its group t, and
// nvb = the blocks of 32 weights present in the unit (8 except in a short
// last unit of the 32-weight types), and adds its rows' sums to y0, y1.

// Row sums of one unit for rows g and g + 8: C columns (hi, lo) of group t.
__device__ __forceinline__ float csum_g(const float (&c)[4]) { return c[0] + c[1]; }
__device__ __forceinline__ float csum_g8(const float (&c)[4]) { return c[2] + c[3]; }

// The code nearest to mu = dm / ds, clamped to 0..qmax (any code gives a
// correct result; the nearest one makes the residual r the smallest), as
// o + 1.5 * 2^23 in fp32: its low mantissa bits are the integer o.  The
// clamp is the multiply's saturation and the rounding the add of 1.5 * 2^23
// (round to nearest even), both on the FMA pipe.
__device__ __forceinline__ float nearest_code_m(float dm, float ds, float qmax) {
    float rc, u;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(ds));
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(u) : "f"(dm * rc), "f"(1.0f / qmax));
    return fmaf(u, qmax, 12582912.0f);
}
// half2 (-(B + o), -(B + o)) with o from nearest_code_m's result m and B the
// magic of the code's position: B = 1024 (code in bits 0..), the fp16 bits
// 0xE400 | o; B = 64 (code in bits 4..), 0xD400 | o << 4.  One integer
// multiply-add on the float's bits, 0x4B400000 + o.
__device__ __forceinline__ uint32_t neg_magic1024(float m) {
    return __float_as_uint(m) * 0x00010001u + (0xE400E400u - 0x4B400000u * 0x00010001u);
}
__device__ __forceinline__ uint32_t neg_magic64(float m) {
    return __float_as_uint(m) * 0x00100010u + (0xD400D400u - 0x4B400000u * 0x00100010u);
}

template <int T> struct HU;

// ---------------------------------------------------------------- Q4_K --
// Group t = code bytes qs[32t .. 32t+31]: low nibbles are sub-block 2t
// (x-block X0 = 2t), high nibbles sub-block 2t+1 (X1 = 2t+1).
template <> struct HU<T_Q4_K> {
    static constexpr int UB = 144;   // bytes per unit per row
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    // [sc(2t), sc(2t+1), m(2t), m(2t+1)] as bytes, from the 12 scale bytes
    // (h.y = s0..3, h.z = s4..7, h.w = s8..11).
    __device__ static __forceinline__ uint32_t fields(const uint4& h, int t) {
        const int j = 2 * (t & 1);
        const uint32_t sel_yz = (uint32_t)(j | ((j + 1) << 4) | ((4 + j) << 8) | ((5 + j) << 12));
        const uint32_t sel_w = (uint32_t)(j | ((j + 1) << 4) | (j << 8) | ((j + 1) << 12));
        const uint32_t p = __byte_perm(h.y, h.z, sel_yz);   // [s_j, s_j+1, s_j+4, s_j+5]
        const uint32_t q = __byte_perm(h.w, 0, sel_w);       // [s_j+8, s_j+9, s_j+8, s_j+9]
        const uint32_t split = (q & 0x00000F0Fu) | ((q >> 4) & 0x0F0F0000u) | ((p >> 2) & 0x30303030u);
        return t >= 2 ? split : (p & 0x3F3F3F3Fu);
    }
    struct Row {
        uint32_t clo, chi;   // half2 offsets -(1024 + o_lo), -(64 + o_hi)
        float ds_lo, ds_hi, r_lo, r_hi;
    };
    __device__ static __forceinline__ Row row_params(const uint4& h, int t) {
        const uint32_t f = fields(h, t);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        Row r;
        r.ds_lo = d * ubyte_f(f, 0);
        r.ds_hi = d * ubyte_f(f, 1);
        const float dm_lo = dmin * ubyte_f(f, 2), dm_hi = dmin * ubyte_f(f, 3);
        const float m_lo = nearest_code_m(dm_lo, r.ds_lo, 15.0f), m_hi = nearest_code_m(dm_hi, r.ds_hi, 15.0f);
        r.r_lo = fmaf(-r.ds_lo, m_lo - 12582912.0f, dm_lo);
        r.r_hi = fmaf(-r.ds_hi, m_hi - 12582912.0f, dm_hi);
        r.clo = neg_magic1024(m_lo);
        r.chi = neg_magic64(m_hi);
        return r;
    }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const uint4 h0 = lds128(r0), h1 = lds128(r1);
        const uint4 a0 = lds128(r0 + 16 + 32 * t), a1 = lds128(r0 + 32 + 32 * t);
        const uint4 b0 = lds128(r1 + 16 + 32 * t), b1 = lds128(r1 + 32 + 32 * t);
        const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const Row p0 = row_params(h0, t), p1 = row_params(h1, t);
        // Two accumulator chains per sub-block (even and odd steps) for more
        // independent MMAs in flight.
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t u0 = w0[i] >> 8, u1 = w1[i] >> 8;
            mma16816(c[i & 1], hadd2(and_or(w0[i], 0x000F000Fu, 0x64006400u), p0.clo),
                     hadd2(and_or(w1[i], 0x000F000Fu, 0x64006400u), p1.clo),
                     hadd2(and_or(u0, 0x000F000Fu, 0x64006400u), p0.clo), hadd2(and_or(u1, 0x000F000Fu, 0x64006400u), p1.clo),
                     xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[2 + (i & 1)], hadd2(and_or(w0[i], 0x00F000F0u, 0x54005400u), p0.chi),
                     hadd2(and_or(w1[i], 0x00F000F0u, 0x54005400u), p1.chi),
                     hadd2(and_or(u0, 0x00F000F0u, 0x54005400u), p0.chi), hadd2(and_or(u1, 0x00F000F0u, 0x54005400u), p1.chi),
                     xb1.b[2 * i], xb1.b[2 * i + 1]);
        }
        const float tl0 = csum_g(c[0]) + csum_g(c[1]), th0 = csum_g(c[2]) + csum_g(c[3]);
        const float tl1 = csum_g8(c[0]) + csum_g8(c[1]), th1 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += fmaf(p0.ds_lo * xm0.y, tl0, -p0.r_lo * xm0.x) + fmaf(p0.ds_hi * xm1.y, th0, -p0.r_hi * xm1.x);
        y1 += fmaf(p1.ds_lo * xm0.y, tl1, -p1.r_lo * xm0.x) + fmaf(p1.ds_hi * xm1.y, th1, -p1.r_hi * xm1.x);
    }
};

// ---------------------------------------------------------------- Q6_K --
// Group t: half th = t/2 of the super-block, code bytes ql[64 th + 32 gl + l]
// (gl = t%2) and qh[32 th + l], l = 0..31.  Low nibbles with qh bits 2gl are
// 32-block (th, gl) (x-block X0 = 4th + gl), high nibbles with qh bits
// 2gl + 4 are 32-block (th, gl + 2) (X1 = X0 + 2).  Words 0-3 of a block are
// its first 16-weight group, words 4-7 the second; w = d * sc * (q - 32).
template <> struct HU<T_Q6_K> {
    static constexpr int UB = 210;
    __device__ static __forceinline__ int X0(int t) { return 4 * (t >> 1) + (t & 1); }
    __device__ static __forceinline__ int X1(int t) { return 4 * (t >> 1) + (t & 1) + 2; }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const int th = t >> 1, gl = t & 1;
        uint32_t ql0[8], qh0[8], ql1[8], qh1[8];
        words_a2<8>(r0 + 64 * th + 32 * gl, ql0);
        words_a2<8>(r0 + 128 + 32 * th, qh0);
        words_a2<8>(r1 + 64 * th + 32 * gl, ql1);
        words_a2<8>(r1 + 128 + 32 * th, qh1);
        // int8 scales of the four 16-weight groups: sc[8th + 2gl + {0, 1}]
        // (block X0) and sc[8th + 2gl + 4 + {0, 1}] (block X1).
        const uint32_t s0 = ld_u16(r0 + 192 + 8 * th + 2 * gl) | (ld_u16(r0 + 196 + 8 * th + 2 * gl) << 16);
        const uint32_t s1 = ld_u16(r1 + 192 + 8 * th + 2 * gl) | (ld_u16(r1 + 196 + 8 * th + 2 * gl) << 16);
        const float d0 = h2f(ld_u16(r0 + 208)), d1 = h2f(ld_u16(r1 + 208));
        const int sh = 4 - 2 * gl;   // qh bits 2gl -> bits 4-5 of a byte, bits 2gl+4 -> bits 8-9 of a half
        float c[4][4] = {};
        const uint32_t CLO = dup16(0xE420u), CHI = dup16(0xD600u);   // -(1024 + 32), -(64 + 32)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v0 = qh0[i] << sh, v1 = qh1[i] << sh;
            // Bytes 1 and 3: shift down first, so that byte 3's bits stay in the word.
            const uint32_t u0 = ql0[i] >> 8, u1 = ql1[i] >> 8, e0 = (qh0[i] >> 8) << sh, e1 = (qh1[i] >> 8) << sh;
            const int a = i >> 2;   // first or second 16-weight group of the block
            // (low code bits & m1) | (high code bits & m2) | magic: two logic ops.
            auto cv = [](uint32_t lo, uint32_t m1, uint32_t hi, uint32_t m2, uint32_t mg) {
                return and_or(lo, m1, and_or(hi, m2, mg));
            };
            mma16816(c[a], hadd2(cv(ql0[i], 0x000F000Fu, v0, 0x00300030u, 0x64006400u), CLO),
                     hadd2(cv(ql1[i], 0x000F000Fu, v1, 0x00300030u, 0x64006400u), CLO),
                     hadd2(cv(u0, 0x000F000Fu, e0, 0x00300030u, 0x64006400u), CLO),
                     hadd2(cv(u1, 0x000F000Fu, e1, 0x00300030u, 0x64006400u), CLO), xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[2 + a], hadd2(cv(ql0[i], 0x00F000F0u, v0, 0x03000300u, 0x54005400u), CHI),
                     hadd2(cv(ql1[i], 0x00F000F0u, v1, 0x03000300u, 0x54005400u), CHI),
                     hadd2(cv(u0, 0x00F000F0u, e0, 0x03000300u, 0x54005400u), CHI),
                     hadd2(cv(u1, 0x00F000F0u, e1, 0x03000300u, 0x54005400u), CHI), xb1.b[2 * i], xb1.b[2 * i + 1]);
        }
        const float f00 = d0 * xm0.y, f01 = d0 * xm1.y, f10 = d1 * xm0.y, f11 = d1 * xm1.y;
        auto sc = [](uint32_t s, int k) { return (float)(int8_t)((s >> (8 * k)) & 0xFFu); };
        y0 += f00 * fmaf(sc(s0, 0), csum_g(c[0]), sc(s0, 1) * csum_g(c[1])) +
              f01 * fmaf(sc(s0, 2), csum_g(c[2]), sc(s0, 3) * csum_g(c[3]));
        y1 += f10 * fmaf(sc(s1, 0), csum_g8(c[0]), sc(s1, 1) * csum_g8(c[1])) +
              f11 * fmaf(sc(s1, 2), csum_g8(c[2]), sc(s1, 3) * csum_g8(c[3]));
    }
};

// ---------------------------------------------------------------- Q8_0 --
// A unit is 8 blocks of 32; group t = blocks 2t (X0) and 2t+1 (X1), 68
// consecutive bytes.  w = d * q, q signed: the magic holds q + 128.
template <> struct HU<T_Q8_0> {
    static constexpr int UB = 8 * 34;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const uint8_t* p0 = r0 + 68 * t;
        const uint8_t* p1 = r1 + 68 * t;
        uint32_t q00[8], q01[8], q10[8], q11[8];
        words_a2<8>(p0 + 2, q00);
        words_a2<8>(p0 + 36, q01);
        words_a2<8>(p1 + 2, q10);
        words_a2<8>(p1 + 36, q11);
        const float d00 = h2f(ld_u16(p0)), d01 = h2f(ld_u16(p0 + 34)), d10 = h2f(ld_u16(p1)), d11 = h2f(ld_u16(p1 + 34));
        const uint32_t C = dup16(0xE480u);   // -(1024 + 128)
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mma16816(c[i & 1], hadd2(and_xor(q00[i], 0x00FF00FFu, 0x64806480u), C), hadd2(and_xor(q10[i], 0x00FF00FFu, 0x64806480u), C),
                     hadd2(and_xor(q00[i] >> 8, 0x00FF00FFu, 0x64806480u), C),
                     hadd2(and_xor(q10[i] >> 8, 0x00FF00FFu, 0x64806480u), C), xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[2 + (i & 1)], hadd2(and_xor(q01[i], 0x00FF00FFu, 0x64806480u), C), hadd2(and_xor(q11[i], 0x00FF00FFu, 0x64806480u), C),
                     hadd2(and_xor(q01[i] >> 8, 0x00FF00FFu, 0x64806480u), C),
                     hadd2(and_xor(q11[i] >> 8, 0x00FF00FFu, 0x64806480u), C), xb1.b[2 * i], xb1.b[2 * i + 1]);
        }
        // Blocks past the end of a short last unit hold stale bytes: skipped.
        const bool v0 = 2 * t < nvb, v1 = 2 * t + 1 < nvb;
        const float t00 = csum_g(c[0]) + csum_g(c[1]), t01 = csum_g(c[2]) + csum_g(c[3]);
        const float t10 = csum_g8(c[0]) + csum_g8(c[1]), t11 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += (v0 ? d00 * xm0.y * t00 : 0.0f) + (v1 ? d01 * xm1.y * t01 : 0.0f);
        y1 += (v0 ? d10 * xm0.y * t10 : 0.0f) + (v1 ? d11 * xm1.y * t11 : 0.0f);
    }
};

// ---------------------------------------------------------------- Q4_0 --
// A unit is 8 blocks of 32 (18 bytes: fp16 d, 16 bytes of nibbles); group t
// = blocks 2t (X0) and 2t+1 (X1).  Element e < 16 is the low nibble of qs[e],
// element 16 + e its high nibble: words 0-3 of a block are the low nibbles
// of its four code words, words 4-7 the high nibbles.  w = d * (q - 8).
template <> struct HU<T_Q4_0> {
    static constexpr int UB = 8 * 18;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const uint8_t* p0 = r0 + 36 * t;
        const uint8_t* p1 = r1 + 36 * t;
        uint32_t q00[4], q01[4], q10[4], q11[4];
        words_a2<4>(p0 + 2, q00);
        words_a2<4>(p0 + 20, q01);
        words_a2<4>(p1 + 2, q10);
        words_a2<4>(p1 + 20, q11);
        const float d00 = h2f(ld_u16(p0)), d01 = h2f(ld_u16(p0 + 18)), d10 = h2f(ld_u16(p1)), d11 = h2f(ld_u16(p1 + 18));
        const uint32_t CL = dup16(0xE408u), CH = dup16(0xD480u);   // -(1024 + 8), -(64 + 8)
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a0 = q00[i] >> 8, a1 = q10[i] >> 8, b0 = q01[i] >> 8, b1 = q11[i] >> 8;
            mma16816(c[0], hadd2(and_or(q00[i], 0x000F000Fu, 0x64006400u), CL), hadd2(and_or(q10[i], 0x000F000Fu, 0x64006400u), CL),
                     hadd2(and_or(a0, 0x000F000Fu, 0x64006400u), CL), hadd2(and_or(a1, 0x000F000Fu, 0x64006400u), CL),
                     xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[1], hadd2(and_or(q00[i], 0x00F000F0u, 0x54005400u), CH), hadd2(and_or(q10[i], 0x00F000F0u, 0x54005400u), CH),
                     hadd2(and_or(a0, 0x00F000F0u, 0x54005400u), CH), hadd2(and_or(a1, 0x00F000F0u, 0x54005400u), CH),
                     xb0.b[8 + 2 * i], xb0.b[8 + 2 * i + 1]);
            mma16816(c[2], hadd2(and_or(q01[i], 0x000F000Fu, 0x64006400u), CL), hadd2(and_or(q11[i], 0x000F000Fu, 0x64006400u), CL),
                     hadd2(and_or(b0, 0x000F000Fu, 0x64006400u), CL), hadd2(and_or(b1, 0x000F000Fu, 0x64006400u), CL),
                     xb1.b[2 * i], xb1.b[2 * i + 1]);
            mma16816(c[3], hadd2(and_or(q01[i], 0x00F000F0u, 0x54005400u), CH), hadd2(and_or(q11[i], 0x00F000F0u, 0x54005400u), CH),
                     hadd2(and_or(b0, 0x00F000F0u, 0x54005400u), CH), hadd2(and_or(b1, 0x00F000F0u, 0x54005400u), CH),
                     xb1.b[8 + 2 * i], xb1.b[8 + 2 * i + 1]);
        }
        const bool v0 = 2 * t < nvb, v1 = 2 * t + 1 < nvb;
        const float t00 = csum_g(c[0]) + csum_g(c[1]), t01 = csum_g(c[2]) + csum_g(c[3]);
        const float t10 = csum_g8(c[0]) + csum_g8(c[1]), t11 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += (v0 ? d00 * xm0.y * t00 : 0.0f) + (v1 ? d01 * xm1.y * t01 : 0.0f);
        y1 += (v0 ? d10 * xm0.y * t10 : 0.0f) + (v1 ? d11 * xm1.y * t11 : 0.0f);
    }
};

// ---------------------------------------------------------------- Q5_0 --
// Blocks of 22 bytes (fp16 d, a 32-bit word of fifth bits, 16 bytes of
// nibbles placed as Q4_0's); group t = blocks 2t (X0) and 2t+1 (X1).  The
// code of element e is its nibble plus 16 * bit e of the fifth-bit word;
// w = d * (q - 16).
template <> struct HU<T_Q5_0> {
    static constexpr int UB = 8 * 22;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    // Four bits z (bit k = fifth bit of byte k) -> 0x10 in each byte whose bit is set.
    __device__ static __forceinline__ uint32_t spread(uint32_t z) { return ((z & 15u) * 0x02040810u) & 0x10101010u; }
    // One block's 8 steps for rows g (word arrays a) and g + 8 (b): code bytes
    // = nibble | fifth bit << 4, then the two byte pairs of a word.
    __device__ static __forceinline__ void block(const uint32_t (&a)[5], const uint32_t (&b)[5], const XB& xb, float (&c)[4],
                                                 float (&c2)[4]) {
        const uint32_t C = dup16(0xE410u);   // -(1024 + 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int w = i & 3, h = i >> 2;   // code word, nibble
            const uint32_t ca = and_or(h ? a[1 + w] >> 4 : a[1 + w], 0x0F0F0F0Fu, spread(a[0] >> (4 * i)));
            const uint32_t cb = and_or(h ? b[1 + w] >> 4 : b[1 + w], 0x0F0F0F0Fu, spread(b[0] >> (4 * i)));
            mma16816(h ? c2 : c, hadd2(and_or(ca, 0x001F001Fu, 0x64006400u), C), hadd2(and_or(cb, 0x001F001Fu, 0x64006400u), C),
                     hadd2(and_or(ca >> 8, 0x001F001Fu, 0x64006400u), C), hadd2(and_or(cb >> 8, 0x001F001Fu, 0x64006400u), C),
                     xb.b[2 * i], xb.b[2 * i + 1]);
        }
    }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const uint8_t* p0 = r0 + 44 * t;
        const uint8_t* p1 = r1 + 44 * t;
        uint32_t a0[5], a1[5], b0[5], b1[5];   // fifth-bit word, then the four code words
        words_a2<5>(p0 + 2, a0);
        words_a2<5>(p0 + 24, a1);
        words_a2<5>(p1 + 2, b0);
        words_a2<5>(p1 + 24, b1);
        const float d00 = h2f(ld_u16(p0)), d01 = h2f(ld_u16(p0 + 22)), d10 = h2f(ld_u16(p1)), d11 = h2f(ld_u16(p1 + 22));
        float c[4][4] = {};
        block(a0, b0, xb0, c[0], c[1]);
        block(a1, b1, xb1, c[2], c[3]);
        const bool v0 = 2 * t < nvb, v1 = 2 * t + 1 < nvb;
        const float t00 = csum_g(c[0]) + csum_g(c[1]), t01 = csum_g(c[2]) + csum_g(c[3]);
        const float t10 = csum_g8(c[0]) + csum_g8(c[1]), t11 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += (v0 ? d00 * xm0.y * t00 : 0.0f) + (v1 ? d01 * xm1.y * t01 : 0.0f);
        y1 += (v0 ? d10 * xm0.y * t10 : 0.0f) + (v1 ? d11 * xm1.y * t11 : 0.0f);
    }
};

// ---------------------------------------------------------------- Q5_K --
// Q4_K's header and code placement (group t = qs[32t .. 32t+31] at byte 48:
// low nibbles sub-block 2t, high nibbles 2t+1) with the fifth code bits in
// qh[l] (byte 16 + l): bit 2t for the low nibble's code, bit 2t+1 for the
// high nibble's.  w = (d*sc)*q - dmin*m, q in 0..31.
template <> struct HU<T_Q5_K> {
    static constexpr int UB = 176;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    __device__ static __forceinline__ HU<T_Q4_K>::Row row_params(const uint4& h, int t) {
        const uint32_t f = HU<T_Q4_K>::fields(h, t);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        HU<T_Q4_K>::Row r;
        r.ds_lo = d * ubyte_f(f, 0);
        r.ds_hi = d * ubyte_f(f, 1);
        const float dm_lo = dmin * ubyte_f(f, 2), dm_hi = dmin * ubyte_f(f, 3);
        const float m_lo = nearest_code_m(dm_lo, r.ds_lo, 31.0f), m_hi = nearest_code_m(dm_hi, r.ds_hi, 31.0f);
        r.r_lo = fmaf(-r.ds_lo, m_lo - 12582912.0f, dm_lo);
        r.r_hi = fmaf(-r.ds_hi, m_hi - 12582912.0f, dm_hi);
        r.clo = neg_magic1024(m_lo);
        r.chi = neg_magic1024(m_hi);
        return r;
    }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const uint4 h0 = lds128(r0), h1 = lds128(r1);
        const uint4 a0 = lds128(r0 + 48 + 32 * t), a1 = lds128(r0 + 64 + 32 * t);
        const uint4 b0 = lds128(r1 + 48 + 32 * t), b1 = lds128(r1 + 64 + 32 * t);
        const uint4 e0 = lds128(r0 + 16), e1 = lds128(r0 + 32), f0 = lds128(r1 + 16), f1 = lds128(r1 + 32);
        const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t v0[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const uint32_t v1[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
        const HU<T_Q4_K>::Row p0 = row_params(h0, t), p1 = row_params(h1, t);
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // Code bytes (0..31) of the low and the high nibbles, then the pairs.
            const uint32_t u0 = v0[i] >> (2 * t), u1 = v1[i] >> (2 * t);
            const uint32_t l0 = and_or(w0[i], 0x0F0F0F0Fu, (u0 << 4) & 0x10101010u);
            const uint32_t l1 = and_or(w1[i], 0x0F0F0F0Fu, (u1 << 4) & 0x10101010u);
            const uint32_t k0 = and_or(w0[i] >> 4, 0x0F0F0F0Fu, (u0 << 3) & 0x10101010u);
            const uint32_t k1 = and_or(w1[i] >> 4, 0x0F0F0F0Fu, (u1 << 3) & 0x10101010u);
            mma16816(c[i & 1], hadd2(and_or(l0, 0x001F001Fu, 0x64006400u), p0.clo),
                     hadd2(and_or(l1, 0x001F001Fu, 0x64006400u), p1.clo),
                     hadd2(and_or(l0 >> 8, 0x001F001Fu, 0x64006400u), p0.clo),
                     hadd2(and_or(l1 >> 8, 0x001F001Fu, 0x64006400u), p1.clo), xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[2 + (i & 1)], hadd2(and_or(k0, 0x001F001Fu, 0x64006400u), p0.chi),
                     hadd2(and_or(k1, 0x001F001Fu, 0x64006400u), p1.chi),
                     hadd2(and_or(k0 >> 8, 0x001F001Fu, 0x64006400u), p0.chi),
                     hadd2(and_or(k1 >> 8, 0x001F001Fu, 0x64006400u), p1.chi), xb1.b[2 * i], xb1.b[2 * i + 1]);
        }
        const float tl0 = csum_g(c[0]) + csum_g(c[1]), th0 = csum_g(c[2]) + csum_g(c[3]);
        const float tl1 = csum_g8(c[0]) + csum_g8(c[1]), th1 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += fmaf(p0.ds_lo * xm0.y, tl0, -p0.r_lo * xm0.x) + fmaf(p0.ds_hi * xm1.y, th0, -p0.r_hi * xm1.x);
        y1 += fmaf(p1.ds_lo * xm0.y, tl1, -p1.r_lo * xm0.x) + fmaf(p1.ds_hi * xm1.y, th1, -p1.r_hi * xm1.x);
    }
};

// ---------------------------------------------------------------- Q2_K --
// 84-byte blocks: sixteen (scale, min) bytes (scale in the low nibble), 64
// bytes of 2-bit codes, fp16 d, fp16 dmin.  Weight 128t' + 32j + l has code
// (qs[32t' + l] >> 2j) & 3; group t = weights 64t .. 64t+63 = code bytes
// qs[32(t/2) ..] with j = 2(t%2) (x-block X0 = 2t) and j + 1 (X1 = 2t+1), and
// the 16-weight groups 4t .. 4t+3 (words 0-3 / 4-7 of each x-block).  A code
// at bits 2j of a byte sits in the mantissa of the magic 2^(10 - 2j) with
// unit weight.  w = (d*sc)*q - dmin*m per 16-weight group, with the code
// offset o = the code nearest dmin*m / (d*sc) as for Q4_K.
template <> struct HU<T_Q2_K> {
    static constexpr int UB = 84;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    struct Row {
        uint32_t cst[4];   // half2 -(magic + o) of the four groups
        float ds[4], r[4];
    };
    __device__ static __forceinline__ Row row_params(const uint8_t* r, int t, float magic0, float magic1) {
        const uint32_t sm = lds32(r + 4 * t);   // (scale, min) bytes of groups 4t .. 4t+3
        const uint32_t dd = lds32(r + 80);
        const float d = h2f(dd & 0xFFFFu), dmin = h2f(dd >> 16);
        const uint32_t scb = sm & 0x0F0F0F0Fu, mb = (sm >> 4) & 0x0F0F0F0Fu;
        Row w;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.ds[k] = d * ubyte_f(scb, k);
            const float dm = dmin * ubyte_f(mb, k);
            const float m = nearest_code_m(dm, w.ds[k], 3.0f);
            const float o = m - 12582912.0f;
            w.r[k] = fmaf(-w.ds[k], o, dm);
            w.cst[k] = h2dup(-((k < 2 ? magic0 : magic1) + o));
        }
        return w;
    }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const int j0 = 2 * (t & 1);
        // Masks and magics of the two code positions: j0 = 0 -> bits 0-1 (1024),
        // j0 = 2 -> bits 4-5 (64); j0 + 1 -> bits 2-3 (256) or 6-7 (16).
        const uint32_t M0 = j0 ? 0x00300030u : 0x00030003u, G0 = j0 ? 0x54005400u : 0x64006400u;
        const uint32_t M1 = j0 ? 0x00C000C0u : 0x000C000Cu, G1 = j0 ? 0x4C004C00u : 0x5C005C00u;
        const float mg0 = j0 ? 64.0f : 1024.0f, mg1 = j0 ? 16.0f : 256.0f;
        // 84-byte blocks are 4-byte aligned (not 16): word loads.
        uint32_t w0[8], w1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w0[i] = lds32(r0 + 16 + 32 * (t >> 1) + 4 * i);
            w1[i] = lds32(r1 + 16 + 32 * (t >> 1) + 4 * i);
        }
        const Row p0 = row_params(r0, t, mg0, mg1), p1 = row_params(r1, t, mg0, mg1);
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = i >> 2;   // 16-weight group within the x-block
            const uint32_t u0 = w0[i] >> 8, u1 = w1[i] >> 8;
            mma16816(c[k], hadd2(and_or(w0[i], M0, G0), p0.cst[k]), hadd2(and_or(w1[i], M0, G0), p1.cst[k]),
                     hadd2(and_or(u0, M0, G0), p0.cst[k]), hadd2(and_or(u1, M0, G0), p1.cst[k]), xb0.b[2 * i],
                     xb0.b[2 * i + 1]);
            mma16816(c[2 + k], hadd2(and_or(w0[i], M1, G1), p0.cst[2 + k]), hadd2(and_or(w1[i], M1, G1), p1.cst[2 + k]),
                     hadd2(and_or(u0, M1, G1), p0.cst[2 + k]), hadd2(and_or(u1, M1, G1), p1.cst[2 + k]), xb1.b[2 * i],
                     xb1.b[2 * i + 1]);
        }
        // Groups 4t, 4t+1 (x-block X0 halves) and 4t+2, 4t+3 (X1 halves).
        y0 += fmaf(p0.ds[0] * xm0.y, csum_g(c[0]), -p0.r[0] * xm0.z) + fmaf(p0.ds[1] * xm0.y, csum_g(c[1]), -p0.r[1] * xm0.w) +
              fmaf(p0.ds[2] * xm1.y, csum_g(c[2]), -p0.r[2] * xm1.z) + fmaf(p0.ds[3] * xm1.y, csum_g(c[3]), -p0.r[3] * xm1.w);
        y1 += fmaf(p1.ds[0] * xm0.y, csum_g8(c[0]), -p1.r[0] * xm0.z) + fmaf(p1.ds[1] * xm0.y, csum_g8(c[1]), -p1.r[1] * xm0.w) +
              fmaf(p1.ds[2] * xm1.y, csum_g8(c[2]), -p1.r[2] * xm1.z) + fmaf(p1.ds[3] * xm1.y, csum_g8(c[3]), -p1.r[3] * xm1.w);
    }
};

// ---------------------------------------------------------------- Q3_K --
// 110-byte blocks: hmask[32], 64 bytes of 2-bit codes (placed as Q2_K's),
// twelve bytes of sixteen 6-bit scales stored + 32, fp16 d.  Weight
// 128t' + 32j + l has u = ((qs[32t' + l] >> 2j) & 3) + 4 * ((hmask[l] >>
// (4t' + j)) & 1) and q = u - 4; w = d*sc*q per 16-weight group.  Group t as
// for Q2_K (X0 = 2t with j = 2(t%2), X1 = 2t+1 with j + 1).  u sits at bits
// 2j .. 2j+2 of a byte, in the mantissa of the magic 2^(10 - 2j) with unit
// weight, the mask bit moved to bit 2j + 2.  Scale of group 4t + k: low four
// bits = nibble t/2 of byte 96 + 4(t%2) + k, high two = bits 2t.. of byte
// 104 + k.
template <> struct HU<T_Q3_K> {
    static constexpr int UB = 110;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    __device__ static __forceinline__ void unit(const uint8_t* r0, const uint8_t* r1, const XB& xb0, const XB& xb1,
                                                float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
        const int tp = t >> 1, j0 = 2 * (t & 1), j1 = j0 + 1;
        // Code bits 2j, 2j+1 and the mask bit moved from bit 4t' + j to 2j + 2,
        // per 16-bit half; magic 2^(10 - 2j).
        const uint32_t M0 = 0x00030003u << (2 * j0), M1 = 0x00030003u << (2 * j1);
        const uint32_t B0 = 0x00040004u << (2 * j0), B1 = 0x00040004u << (2 * j1);
        const uint32_t G0 = j0 ? 0x54005400u : 0x64006400u, G1 = j0 ? 0x4C004C00u : 0x5C005C00u;
        // -(magic + 4): 1028 = 0x6404 -> 0xE404 (j = 0); 260 = 0x5C10 -> 0xDC10 (j = 1);
        // 68 = 0x5440 -> 0xD440 (j = 2); 20 = 0x4D00 -> 0xCD00 (j = 3).
        const uint32_t CC0 = j0 ? dup16(0xD440u) : dup16(0xE404u), CC1 = j0 ? dup16(0xCD00u) : dup16(0xDC10u);
        const int hs0 = 4 * tp + j0, hs1 = 4 * tp + j1;   // mask bit positions
        const int sh0 = 2 * j0 + 2 - hs0, sh1 = 2 * j1 + 2 - hs1;   // shift to place it (may be negative)
        uint32_t q0[8], q1[8], m0[8], m1[8];
        words_a2<8>(r0 + 32 + 32 * tp, q0);
        words_a2<8>(r1 + 32 + 32 * tp, q1);
        words_a2<8>(r0, m0);
        words_a2<8>(r1, m1);
        auto shl = [](uint32_t v, int s) { return s >= 0 ? v << s : v >> (-s); };
        float c[4][4] = {};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = i >> 2;
            const uint32_t qa = q0[i], qb = q1[i], qa8 = q0[i] >> 8, qb8 = q1[i] >> 8;
            const uint32_t ma = m0[i], mb = m1[i], ma8 = m0[i] >> 8, mb8 = m1[i] >> 8;
            mma16816(c[k], hadd2(and_or(qa, M0, and_or(shl(ma, sh0), B0, G0)), CC0),
                     hadd2(and_or(qb, M0, and_or(shl(mb, sh0), B0, G0)), CC0),
                     hadd2(and_or(qa8, M0, and_or(shl(ma8, sh0), B0, G0)), CC0),
                     hadd2(and_or(qb8, M0, and_or(shl(mb8, sh0), B0, G0)), CC0), xb0.b[2 * i], xb0.b[2 * i + 1]);
            mma16816(c[2 + k], hadd2(and_or(qa, M1, and_or(shl(ma, sh1), B1, G1)), CC1),
                     hadd2(and_or(qb, M1, and_or(shl(mb, sh1), B1, G1)), CC1),
                     hadd2(and_or(qa8, M1, and_or(shl(ma8, sh1), B1, G1)), CC1),
                     hadd2(and_or(qb8, M1, and_or(shl(mb8, sh1), B1, G1)), CC1), xb1.b[2 * i], xb1.b[2 * i + 1]);
        }
        // Scales of groups 4t .. 4t+3 (signed, stored + 32).
        uint32_t l0[1], l1[1], u0[1], u1[1];
        words_a2<1>(r0 + 96 + 4 * (t & 1), l0);
        words_a2<1>(r1 + 96 + 4 * (t & 1), l1);
        words_a2<1>(r0 + 104, u0);
        words_a2<1>(r1 + 104, u1);
        const uint32_t S0 = ((l0[0] >> (4 * tp)) & 0x0F0F0F0Fu) | (((u0[0] >> (2 * t)) & 0x03030303u) << 4);
        const uint32_t S1 = ((l1[0] >> (4 * tp)) & 0x0F0F0F0Fu) | (((u1[0] >> (2 * t)) & 0x03030303u) << 4);
        const float d0 = h2f(ld_u16(r0 + 108)), d1 = h2f(ld_u16(r1 + 108));
        auto sc = [](uint32_t S, int k) { return ubyte_f(S, k) - 32.0f; };
        y0 += d0 * (xm0.y * fmaf(sc(S0, 0), csum_g(c[0]), sc(S0, 1) * csum_g(c[1])) +
                    xm1.y * fmaf(sc(S0, 2), csum_g(c[2]), sc(S0, 3) * csum_g(c[3])));
        y1 += d1 * (xm0.y * fmaf(sc(S1, 0), csum_g8(c[0]), sc(S1, 1) * csum_g8(c[1])) +
                    xm1.y * fmaf(sc(S1, 2), csum_g8(c[2]), sc(S1, 3) * csum_g8(c[3])));
    }
};

}  // namespace hm
}  // namespace qk
