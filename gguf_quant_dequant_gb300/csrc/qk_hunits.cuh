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

// D = A * B with zero accumulators: the first step of a sum, without
// clearing four registers first.
__device__ __forceinline__ void mma16816_z(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
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

// Every unit decoder HU<T> provides:
//   Ctx                        the unit's code words and scales of rows g, g + 8
//   load(ctx, r0, r1, t)       read them from the unit's bytes of the two rows
//   conv(ctx, i, t, A)         A fragments of step i: A[0..3] for x-block X0
//                              (row g bytes 0/2, row g+8 bytes 0/2, row g
//                              bytes 1/3, row g+8 bytes 1/3), A[4..7] for X1
//   epi(ctx, c, xm0, xm1, t, nvb, y0, y1)   scale the accumulators of one
//                              token (c[0..1] X0, c[2..3] X1: the two halves
//                              of each x-block for the 16-weight-group types;
//                              otherwise c[0] X0 and c[2] X1, with c[1] and
//                              c[3] zero) and add the rows'
//                              sums; nvb = blocks of 32 weights present in
//                              the unit (8 except in a short last unit).

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
    static constexpr bool kGroup16 = false;
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
        uint32_t clo, chi;   // half2 offsets -(magic + o) of the low and high nibble codes
        float2 ds;           // d*sc of the low and high sub-block
        float2 nr;           // -r = d*sc*o - dmin*m of each
    };
    // The per-sub-block factors d*sc and dmin*m, the nearest code o of their
    // ratio and the residual r = dmin*m - d*sc*o; the high codes use magic
    // 64 (hi_magic64) or 1024 (codes moved down first, as Q5_K's).  The two
    // sub-blocks go through packed fp32 pair operations (each lane rounds as
    // the scalar operation would).
    template <bool hi_magic64>
    __device__ static __forceinline__ Row row_params(const uint4& h, int t, float qmax) {
        const uint32_t f = fields(h, t);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        constexpr float kM = 8388608.0f, kR = 12582912.0f;   // 2^23, 1.5 * 2^23
        const float2 sc = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(f, 0x4B000000u, 0x7650)),
                                                 __uint_as_float(__byte_perm(f, 0x4B000000u, 0x7651))),
                                     make_float2(-kM, -kM));
        const float2 mm = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(f, 0x4B000000u, 0x7652)),
                                                 __uint_as_float(__byte_perm(f, 0x4B000000u, 0x7653))),
                                     make_float2(-kM, -kM));
        Row r;
        r.ds = __fmul2_rn(make_float2(d, d), sc);
        const float2 ndm = __fmul2_rn(make_float2(-dmin, -dmin), mm);   // -dmin*m, exact
        // The nearest code of dm / ds (nearest_code_m, per lane): the ratio's
        // sign is carried by the saturating multiply's factor.
        float rc0, rc1, u0, u1;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc0) : "f"(r.ds.x));
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc1) : "f"(r.ds.y));
        const float2 q = __fmul2_rn(ndm, make_float2(rc0, rc1));
        asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(u0) : "f"(q.x), "f"(-1.0f / qmax));
        asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(u1) : "f"(q.y), "f"(-1.0f / qmax));
        const float2 m = __ffma2_rn(make_float2(u0, u1), make_float2(qmax, qmax), make_float2(kR, kR));
        const float2 o = __fadd2_rn(m, make_float2(-kR, -kR));
        r.nr = __ffma2_rn(r.ds, o, ndm);
        r.clo = neg_magic1024(m.x);
        r.chi = hi_magic64 ? neg_magic64(m.y) : neg_magic1024(m.y);
        return r;
    }
    // y0, y1 += the unit's sums of rows g, g + 8 (low / high sub-block sums
    // of group t in c[0] / c[2], each the hi and lo columns): ds*2^e*t - r*X
    // per sub-block.
    __device__ static __forceinline__ void epi_min(const Row& p0, const Row& p1, const float (&c)[4][4], float4 xm0,
                                                   float4 xm1, float& y0, float& y1) {
        y0 += fmaf(p0.ds.x * xm0.y, c[0][0] + c[0][1], p0.nr.x * xm0.x) +
              fmaf(p0.ds.y * xm1.y, c[2][0] + c[2][1], p0.nr.y * xm1.x);
        y1 += fmaf(p1.ds.x * xm0.y, c[0][2] + c[0][3], p1.nr.x * xm0.x) +
              fmaf(p1.ds.y * xm1.y, c[2][2] + c[2][3], p1.nr.y * xm1.x);
    }
    struct Ctx {
        uint32_t w0[8], w1[8];
        Row p0, p1;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const uint4 h0 = lds128(r0), h1 = lds128(r1);
        const uint4 a0 = lds128(r0 + 16 + 32 * t), a1 = lds128(r0 + 32 + 32 * t);
        const uint4 b0 = lds128(r1 + 16 + 32 * t), b1 = lds128(r1 + 32 + 32 * t);
        x.w0[0] = a0.x; x.w0[1] = a0.y; x.w0[2] = a0.z; x.w0[3] = a0.w;
        x.w0[4] = a1.x; x.w0[5] = a1.y; x.w0[6] = a1.z; x.w0[7] = a1.w;
        x.w1[0] = b0.x; x.w1[1] = b0.y; x.w1[2] = b0.z; x.w1[3] = b0.w;
        x.w1[4] = b1.x; x.w1[5] = b1.y; x.w1[6] = b1.z; x.w1[7] = b1.w;
        x.p0 = row_params<true>(h0, t, 15.0f);
        x.p1 = row_params<true>(h1, t, 15.0f);
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int, uint32_t (&A)[8]) {
        const uint32_t u0 = x.w0[i] >> 8, u1 = x.w1[i] >> 8;
        A[0] = hadd2(and_or(x.w0[i], 0x000F000Fu, 0x64006400u), x.p0.clo);
        A[1] = hadd2(and_or(x.w1[i], 0x000F000Fu, 0x64006400u), x.p1.clo);
        A[2] = hadd2(and_or(u0, 0x000F000Fu, 0x64006400u), x.p0.clo);
        A[3] = hadd2(and_or(u1, 0x000F000Fu, 0x64006400u), x.p1.clo);
        A[4] = hadd2(and_or(x.w0[i], 0x00F000F0u, 0x54005400u), x.p0.chi);
        A[5] = hadd2(and_or(x.w1[i], 0x00F000F0u, 0x54005400u), x.p1.chi);
        A[6] = hadd2(and_or(u0, 0x00F000F0u, 0x54005400u), x.p0.chi);
        A[7] = hadd2(and_or(u1, 0x00F000F0u, 0x54005400u), x.p1.chi);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int, int,
                                               float& y0, float& y1) {
        epi_min(x.p0, x.p1, c, xm0, xm1, y0, y1);
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
    static constexpr bool kGroup16 = true;
    __device__ static __forceinline__ int X0(int t) { return 4 * (t >> 1) + (t & 1); }
    __device__ static __forceinline__ int X1(int t) { return 4 * (t >> 1) + (t & 1) + 2; }
    struct Ctx {
        uint32_t ql0[8], qh0[8], ql1[8], qh1[8];
        uint32_t s0, s1;   // int8 scales of the four 16-weight groups, rows g and g + 8
        float d0, d1;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const int th = t >> 1, gl = t & 1;
        words_a2<8>(r0 + 64 * th + 32 * gl, x.ql0);
        words_a2<8>(r0 + 128 + 32 * th, x.qh0);
        words_a2<8>(r1 + 64 * th + 32 * gl, x.ql1);
        words_a2<8>(r1 + 128 + 32 * th, x.qh1);
        // sc[8th + 2gl + {0, 1}] (block X0) and sc[8th + 2gl + 4 + {0, 1}] (block X1).
        x.s0 = ld_u16(r0 + 192 + 8 * th + 2 * gl) | (ld_u16(r0 + 196 + 8 * th + 2 * gl) << 16);
        x.s1 = ld_u16(r1 + 192 + 8 * th + 2 * gl) | (ld_u16(r1 + 196 + 8 * th + 2 * gl) << 16);
        x.d0 = h2f(ld_u16(r0 + 208));
        x.d1 = h2f(ld_u16(r1 + 208));
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int t, uint32_t (&A)[8]) {
        const int sh = 4 - 2 * (t & 1);   // qh bits 2gl -> bits 4-5 of a byte, bits 2gl+4 -> bits 8-9 of a half
        const uint32_t v0 = x.qh0[i] << sh, v1 = x.qh1[i] << sh;
        // Bytes 1 and 3: one right shift puts their qh bits where v has those
        // of bytes 0 and 2 (the other bits it moves are masked off).
        const uint32_t u0 = x.ql0[i] >> 8, u1 = x.ql1[i] >> 8, e0 = x.qh0[i] >> (8 - sh), e1 = x.qh1[i] >> (8 - sh);
        const uint32_t CLO = dup16(0xE420u), CHI = dup16(0xD600u);   // -(1024 + 32), -(64 + 32)
        // (low code bits & m1) | (high code bits & m2) | magic: two logic ops.
        auto cv = [](uint32_t lo, uint32_t m1, uint32_t hi, uint32_t m2, uint32_t mg) {
            return and_or(lo, m1, and_or(hi, m2, mg));
        };
        A[0] = hadd2(cv(x.ql0[i], 0x000F000Fu, v0, 0x00300030u, 0x64006400u), CLO);
        A[1] = hadd2(cv(x.ql1[i], 0x000F000Fu, v1, 0x00300030u, 0x64006400u), CLO);
        A[2] = hadd2(cv(u0, 0x000F000Fu, e0, 0x00300030u, 0x64006400u), CLO);
        A[3] = hadd2(cv(u1, 0x000F000Fu, e1, 0x00300030u, 0x64006400u), CLO);
        A[4] = hadd2(cv(x.ql0[i], 0x00F000F0u, v0, 0x03000300u, 0x54005400u), CHI);
        A[5] = hadd2(cv(x.ql1[i], 0x00F000F0u, v1, 0x03000300u, 0x54005400u), CHI);
        A[6] = hadd2(cv(u0, 0x00F000F0u, e0, 0x03000300u, 0x54005400u), CHI);
        A[7] = hadd2(cv(u1, 0x00F000F0u, e1, 0x03000300u, 0x54005400u), CHI);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int, int,
                                               float& y0, float& y1) {
        // The four int8 scales of a row as exact floats: each byte with its sign
        // bit flipped (b + 128) in the mantissa of 2^23, less 2^23 + 128.
        auto scales = [](uint32_t s, float (&f)[4]) {
            const uint32_t u = s ^ 0x80808080u;
            const float2 lo = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)),
                                                     __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651))),
                                         make_float2(-8388736.0f, -8388736.0f));
            const float2 hi = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)),
                                                     __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653))),
                                         make_float2(-8388736.0f, -8388736.0f));
            f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
        };
        float a[4], b[4];
        scales(x.s0, a);
        scales(x.s1, b);
        y0 += x.d0 * (xm0.y * fmaf(a[0], csum_g(c[0]), a[1] * csum_g(c[1])) +
                      xm1.y * fmaf(a[2], csum_g(c[2]), a[3] * csum_g(c[3])));
        y1 += x.d1 * (xm0.y * fmaf(b[0], csum_g8(c[0]), b[1] * csum_g8(c[1])) +
                      xm1.y * fmaf(b[2], csum_g8(c[2]), b[3] * csum_g8(c[3])));
    }
};

// ---------------------------------------------------------------- Q8_0 --
// A unit is 8 blocks of 32; group t = blocks 2t (X0) and 2t+1 (X1), 68
// consecutive bytes.  w = d * q, q signed: the magic holds q + 128.
template <> struct HU<T_Q8_0> {
    static constexpr int UB = 8 * 34;
    static constexpr bool kGroup16 = false;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    struct Ctx {
        uint32_t q00[8], q01[8], q10[8], q11[8];
        float d00, d01, d10, d11;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const uint8_t* p0 = r0 + 68 * t;
        const uint8_t* p1 = r1 + 68 * t;
        words_a2<8>(p0 + 2, x.q00);
        words_a2<8>(p0 + 36, x.q01);
        words_a2<8>(p1 + 2, x.q10);
        words_a2<8>(p1 + 36, x.q11);
        x.d00 = h2f(ld_u16(p0));
        x.d01 = h2f(ld_u16(p0 + 34));
        x.d10 = h2f(ld_u16(p1));
        x.d11 = h2f(ld_u16(p1 + 34));
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int, uint32_t (&A)[8]) {
        const uint32_t C = dup16(0xE480u);   // -(1024 + 128)
        A[0] = hadd2(and_xor(x.q00[i], 0x00FF00FFu, 0x64806480u), C);
        A[1] = hadd2(and_xor(x.q10[i], 0x00FF00FFu, 0x64806480u), C);
        A[2] = hadd2(and_xor(x.q00[i] >> 8, 0x00FF00FFu, 0x64806480u), C);
        A[3] = hadd2(and_xor(x.q10[i] >> 8, 0x00FF00FFu, 0x64806480u), C);
        A[4] = hadd2(and_xor(x.q01[i], 0x00FF00FFu, 0x64806480u), C);
        A[5] = hadd2(and_xor(x.q11[i], 0x00FF00FFu, 0x64806480u), C);
        A[6] = hadd2(and_xor(x.q01[i] >> 8, 0x00FF00FFu, 0x64806480u), C);
        A[7] = hadd2(and_xor(x.q11[i] >> 8, 0x00FF00FFu, 0x64806480u), C);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int t,
                                               int nvb, float& y0, float& y1) {
        // Blocks past the end of a short last unit hold stale bytes: skipped.
        const bool v0 = 2 * t < nvb, v1 = 2 * t + 1 < nvb;
        const float t00 = csum_g(c[0]) + csum_g(c[1]), t01 = csum_g(c[2]) + csum_g(c[3]);
        const float t10 = csum_g8(c[0]) + csum_g8(c[1]), t11 = csum_g8(c[2]) + csum_g8(c[3]);
        y0 += (v0 ? x.d00 * xm0.y * t00 : 0.0f) + (v1 ? x.d01 * xm1.y * t01 : 0.0f);
        y1 += (v0 ? x.d10 * xm0.y * t10 : 0.0f) + (v1 ? x.d11 * xm1.y * t11 : 0.0f);
    }
};

// Epilogue of the two-block types (Q8_0, Q4_0, Q5_0): y += d * 2^e * T per block.
struct Epi2 {
    __device__ static __forceinline__ void run(float d00, float d01, float d10, float d11, const float (&c)[4][4],
                                               float4 xm0, float4 xm1, int t, int nvb, float& y0, float& y1) {
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
// element 16 + e its high nibble: steps 0-3 of a block are the low nibbles
// of its four code words, steps 4-7 the high nibbles.  w = d * (q - 8).
template <> struct HU<T_Q4_0> {
    static constexpr int UB = 8 * 18;
    static constexpr bool kGroup16 = false;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    struct Ctx {
        uint32_t q00[4], q01[4], q10[4], q11[4];
        float d00, d01, d10, d11;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const uint8_t* p0 = r0 + 36 * t;
        const uint8_t* p1 = r1 + 36 * t;
        words_a2<4>(p0 + 2, x.q00);
        words_a2<4>(p0 + 20, x.q01);
        words_a2<4>(p1 + 2, x.q10);
        words_a2<4>(p1 + 20, x.q11);
        x.d00 = h2f(ld_u16(p0));
        x.d01 = h2f(ld_u16(p0 + 18));
        x.d10 = h2f(ld_u16(p1));
        x.d11 = h2f(ld_u16(p1 + 18));
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int, uint32_t (&A)[8]) {
        const int w = i & 3;
        // Low nibbles: magic 1024, -(1024 + 8); high nibbles: magic 64, -(64 + 8).
        const uint32_t M = i < 4 ? 0x000F000Fu : 0x00F000F0u, G = i < 4 ? 0x64006400u : 0x54005400u;
        const uint32_t C = i < 4 ? dup16(0xE408u) : dup16(0xD480u);
        A[0] = hadd2(and_or(x.q00[w], M, G), C);
        A[1] = hadd2(and_or(x.q10[w], M, G), C);
        A[2] = hadd2(and_or(x.q00[w] >> 8, M, G), C);
        A[3] = hadd2(and_or(x.q10[w] >> 8, M, G), C);
        A[4] = hadd2(and_or(x.q01[w], M, G), C);
        A[5] = hadd2(and_or(x.q11[w], M, G), C);
        A[6] = hadd2(and_or(x.q01[w] >> 8, M, G), C);
        A[7] = hadd2(and_or(x.q11[w] >> 8, M, G), C);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int t,
                                               int nvb, float& y0, float& y1) {
        Epi2::run(x.d00, x.d01, x.d10, x.d11, c, xm0, xm1, t, nvb, y0, y1);
    }
};

// ---------------------------------------------------------------- Q5_0 --
// Blocks of 22 bytes (fp16 d, a 32-bit word of fifth bits, 16 bytes of
// nibbles placed as Q4_0's); group t = blocks 2t (X0) and 2t+1 (X1).  The
// code of element e is its nibble plus 16 * bit e of the fifth-bit word;
// w = d * (q - 16).
template <> struct HU<T_Q5_0> {
    static constexpr int UB = 8 * 22;
    static constexpr bool kGroup16 = false;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    // Four bits z (bit k = fifth bit of byte k) -> 0x10 in each byte whose bit is set.
    __device__ static __forceinline__ uint32_t spread(uint32_t z) { return ((z & 15u) * 0x02040810u) & 0x10101010u; }
    struct Ctx {
        uint32_t a0[5], a1[5], b0[5], b1[5];   // fifth-bit word, then the four code words
        float d00, d01, d10, d11;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const uint8_t* p0 = r0 + 44 * t;
        const uint8_t* p1 = r1 + 44 * t;
        words_a2<5>(p0 + 2, x.a0);
        words_a2<5>(p0 + 24, x.a1);
        words_a2<5>(p1 + 2, x.b0);
        words_a2<5>(p1 + 24, x.b1);
        x.d00 = h2f(ld_u16(p0));
        x.d01 = h2f(ld_u16(p0 + 22));
        x.d10 = h2f(ld_u16(p1));
        x.d11 = h2f(ld_u16(p1 + 22));
    }
    // Code bytes (0..31) of step i: nibble | fifth bit << 4.
    __device__ static __forceinline__ uint32_t codes(const uint32_t (&q)[5], int i) {
        const int w = i & 3;
        return and_or(i < 4 ? q[1 + w] : q[1 + w] >> 4, 0x0F0F0F0Fu, spread(q[0] >> (4 * i)));
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int, uint32_t (&A)[8]) {
        const uint32_t C = dup16(0xE410u);   // -(1024 + 16)
        const uint32_t ca = codes(x.a0, i), cb = codes(x.b0, i), cc = codes(x.a1, i), cd = codes(x.b1, i);
        A[0] = hadd2(and_or(ca, 0x001F001Fu, 0x64006400u), C);
        A[1] = hadd2(and_or(cb, 0x001F001Fu, 0x64006400u), C);
        A[2] = hadd2(and_or(ca >> 8, 0x001F001Fu, 0x64006400u), C);
        A[3] = hadd2(and_or(cb >> 8, 0x001F001Fu, 0x64006400u), C);
        A[4] = hadd2(and_or(cc, 0x001F001Fu, 0x64006400u), C);
        A[5] = hadd2(and_or(cd, 0x001F001Fu, 0x64006400u), C);
        A[6] = hadd2(and_or(cc >> 8, 0x001F001Fu, 0x64006400u), C);
        A[7] = hadd2(and_or(cd >> 8, 0x001F001Fu, 0x64006400u), C);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int t,
                                               int nvb, float& y0, float& y1) {
        Epi2::run(x.d00, x.d01, x.d10, x.d11, c, xm0, xm1, t, nvb, y0, y1);
    }
};

// ---------------------------------------------------------------- Q5_K --
// Q4_K's header and code placement (group t = qs[32t .. 32t+31] at byte 48:
// low nibbles sub-block 2t, high nibbles 2t+1) with the fifth code bits in
// qh[l] (byte 16 + l): bit 2t for the low nibble's code, bit 2t+1 for the
// high nibble's.  Both codes are moved to bits 0-4 (magic 1024).
// w = (d*sc)*q - dmin*m, q in 0..31.
template <> struct HU<T_Q5_K> {
    static constexpr int UB = 176;
    static constexpr bool kGroup16 = false;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    struct Ctx {
        uint32_t w0[8], w1[8], v0[8], v1[8];
        HU<T_Q4_K>::Row p0, p1;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const uint4 h0 = lds128(r0), h1 = lds128(r1);
        const uint4 a0 = lds128(r0 + 48 + 32 * t), a1 = lds128(r0 + 64 + 32 * t);
        const uint4 b0 = lds128(r1 + 48 + 32 * t), b1 = lds128(r1 + 64 + 32 * t);
        const uint4 e0 = lds128(r0 + 16), e1 = lds128(r0 + 32), f0 = lds128(r1 + 16), f1 = lds128(r1 + 32);
        const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t v0[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const uint32_t v1[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x.w0[i] = w0[i];
            x.w1[i] = w1[i];
            x.v0[i] = v0[i] >> (2 * t);   // bit 0 of each byte: low code's fifth bit, bit 1: high code's
            x.v1[i] = v1[i] >> (2 * t);
        }
        x.p0 = HU<T_Q4_K>::row_params<false>(h0, t, 31.0f);
        x.p1 = HU<T_Q4_K>::row_params<false>(h1, t, 31.0f);
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int, uint32_t (&A)[8]) {
        const uint32_t l0 = and_or(x.w0[i], 0x0F0F0F0Fu, (x.v0[i] << 4) & 0x10101010u);
        const uint32_t l1 = and_or(x.w1[i], 0x0F0F0F0Fu, (x.v1[i] << 4) & 0x10101010u);
        const uint32_t k0 = and_or(x.w0[i] >> 4, 0x0F0F0F0Fu, (x.v0[i] << 3) & 0x10101010u);
        const uint32_t k1 = and_or(x.w1[i] >> 4, 0x0F0F0F0Fu, (x.v1[i] << 3) & 0x10101010u);
        A[0] = hadd2(and_or(l0, 0x001F001Fu, 0x64006400u), x.p0.clo);
        A[1] = hadd2(and_or(l1, 0x001F001Fu, 0x64006400u), x.p1.clo);
        A[2] = hadd2(and_or(l0 >> 8, 0x001F001Fu, 0x64006400u), x.p0.clo);
        A[3] = hadd2(and_or(l1 >> 8, 0x001F001Fu, 0x64006400u), x.p1.clo);
        A[4] = hadd2(and_or(k0, 0x001F001Fu, 0x64006400u), x.p0.chi);
        A[5] = hadd2(and_or(k1, 0x001F001Fu, 0x64006400u), x.p1.chi);
        A[6] = hadd2(and_or(k0 >> 8, 0x001F001Fu, 0x64006400u), x.p0.chi);
        A[7] = hadd2(and_or(k1 >> 8, 0x001F001Fu, 0x64006400u), x.p1.chi);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int, int,
                                               float& y0, float& y1) {
        HU<T_Q4_K>::epi_min(x.p0, x.p1, c, xm0, xm1, y0, y1);
    }
};

// ---------------------------------------------------------------- Q2_K --
// 84-byte blocks: sixteen (scale, min) bytes (scale in the low nibble), 64
// bytes of 2-bit codes, fp16 d, fp16 dmin.  Weight 128t' + 32j + l has code
// (qs[32t' + l] >> 2j) & 3; group t = weights 64t .. 64t+63 = code bytes
// qs[32(t/2) ..] with j = 2(t%2) (x-block X0 = 2t) and j + 1 (X1 = 2t+1), and
// the 16-weight groups 4t .. 4t+3 (steps 0-3 / 4-7 of each x-block).  A code
// at bits 2j of a byte sits in the mantissa of the magic 2^(10 - 2j) with
// unit weight.  w = (d*sc)*q - dmin*m per 16-weight group, with the code
// offset o = the code nearest dmin*m / (d*sc) as for Q4_K.
template <> struct HU<T_Q2_K> {
    static constexpr int UB = 84;
    static constexpr bool kGroup16 = true;
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
            const float o = nearest_code_m(dm, w.ds[k], 3.0f) - 12582912.0f;
            w.r[k] = fmaf(-w.ds[k], o, dm);
            w.cst[k] = h2dup(-((k < 2 ? magic0 : magic1) + o));
        }
        return w;
    }
    struct Ctx {
        uint32_t w0[8], w1[8];
        Row p0, p1;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const int j0 = 2 * (t & 1);
        // 84-byte blocks are 4-byte aligned (not 16): word loads.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x.w0[i] = lds32(r0 + 16 + 32 * (t >> 1) + 4 * i);
            x.w1[i] = lds32(r1 + 16 + 32 * (t >> 1) + 4 * i);
        }
        const float mg0 = j0 ? 64.0f : 1024.0f, mg1 = j0 ? 16.0f : 256.0f;
        x.p0 = row_params(r0, t, mg0, mg1);
        x.p1 = row_params(r1, t, mg0, mg1);
    }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int t, uint32_t (&A)[8]) {
        const int j0 = 2 * (t & 1), k = i >> 2;
        // Masks and magics of the two code positions: j0 = 0 -> bits 0-1 (1024),
        // j0 = 2 -> bits 4-5 (64); j0 + 1 -> bits 2-3 (256) or 6-7 (16).
        const uint32_t M0 = j0 ? 0x00300030u : 0x00030003u, G0 = j0 ? 0x54005400u : 0x64006400u;
        const uint32_t M1 = j0 ? 0x00C000C0u : 0x000C000Cu, G1 = j0 ? 0x4C004C00u : 0x5C005C00u;
        const uint32_t u0 = x.w0[i] >> 8, u1 = x.w1[i] >> 8;
        A[0] = hadd2(and_or(x.w0[i], M0, G0), x.p0.cst[k]);
        A[1] = hadd2(and_or(x.w1[i], M0, G0), x.p1.cst[k]);
        A[2] = hadd2(and_or(u0, M0, G0), x.p0.cst[k]);
        A[3] = hadd2(and_or(u1, M0, G0), x.p1.cst[k]);
        A[4] = hadd2(and_or(x.w0[i], M1, G1), x.p0.cst[2 + k]);
        A[5] = hadd2(and_or(x.w1[i], M1, G1), x.p1.cst[2 + k]);
        A[6] = hadd2(and_or(u0, M1, G1), x.p0.cst[2 + k]);
        A[7] = hadd2(and_or(u1, M1, G1), x.p1.cst[2 + k]);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int, int,
                                               float& y0, float& y1) {
        // Groups 4t, 4t+1 (x-block X0 halves) and 4t+2, 4t+3 (X1 halves).
        y0 += fmaf(x.p0.ds[0] * xm0.y, csum_g(c[0]), -x.p0.r[0] * xm0.z) +
              fmaf(x.p0.ds[1] * xm0.y, csum_g(c[1]), -x.p0.r[1] * xm0.w) +
              fmaf(x.p0.ds[2] * xm1.y, csum_g(c[2]), -x.p0.r[2] * xm1.z) +
              fmaf(x.p0.ds[3] * xm1.y, csum_g(c[3]), -x.p0.r[3] * xm1.w);
        y1 += fmaf(x.p1.ds[0] * xm0.y, csum_g8(c[0]), -x.p1.r[0] * xm0.z) +
              fmaf(x.p1.ds[1] * xm0.y, csum_g8(c[1]), -x.p1.r[1] * xm0.w) +
              fmaf(x.p1.ds[2] * xm1.y, csum_g8(c[2]), -x.p1.r[2] * xm1.z) +
              fmaf(x.p1.ds[3] * xm1.y, csum_g8(c[3]), -x.p1.r[3] * xm1.w);
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
    static constexpr bool kGroup16 = true;
    __device__ static __forceinline__ int X0(int t) { return 2 * t; }
    __device__ static __forceinline__ int X1(int t) { return 2 * t + 1; }
    struct Ctx {
        uint32_t q0[8], q1[8], m0[8], m1[8];
        uint32_t S0, S1;   // the four scales (+ 32) of rows g and g + 8, as bytes
        float d0, d1;
    };
    __device__ static __forceinline__ void load(Ctx& x, const uint8_t* r0, const uint8_t* r1, int t) {
        const int tp = t >> 1;
        words_a2<8>(r0 + 32 + 32 * tp, x.q0);
        words_a2<8>(r1 + 32 + 32 * tp, x.q1);
        words_a2<8>(r0, x.m0);
        words_a2<8>(r1, x.m1);
        uint32_t l0[1], l1[1], u0[1], u1[1];
        words_a2<1>(r0 + 96 + 4 * (t & 1), l0);
        words_a2<1>(r1 + 96 + 4 * (t & 1), l1);
        words_a2<1>(r0 + 104, u0);
        words_a2<1>(r1 + 104, u1);
        x.S0 = ((l0[0] >> (4 * tp)) & 0x0F0F0F0Fu) | (((u0[0] >> (2 * t)) & 0x03030303u) << 4);
        x.S1 = ((l1[0] >> (4 * tp)) & 0x0F0F0F0Fu) | (((u1[0] >> (2 * t)) & 0x03030303u) << 4);
        x.d0 = h2f(ld_u16(r0 + 108));
        x.d1 = h2f(ld_u16(r1 + 108));
    }
    __device__ static __forceinline__ uint32_t shl(uint32_t v, int s) { return s >= 0 ? v << s : v >> (-s); }
    __device__ static __forceinline__ void conv(const Ctx& x, int i, int t, uint32_t (&A)[8]) {
        const int tp = t >> 1, j0 = 2 * (t & 1), j1 = j0 + 1;
        // Code bits 2j, 2j+1 and the mask bit moved from bit 4t' + j to 2j + 2,
        // per 16-bit half; magic 2^(10 - 2j).
        const uint32_t M0 = 0x00030003u << (2 * j0), M1 = 0x00030003u << (2 * j1);
        const uint32_t B0 = 0x00040004u << (2 * j0), B1 = 0x00040004u << (2 * j1);
        const uint32_t G0 = j0 ? 0x54005400u : 0x64006400u, G1 = j0 ? 0x4C004C00u : 0x5C005C00u;
        // -(magic + 4): 1028 = 0x6404 -> 0xE404 (j = 0); 260 = 0x5C10 -> 0xDC10 (j = 1);
        // 68 = 0x5440 -> 0xD440 (j = 2); 20 = 0x4D00 -> 0xCD00 (j = 3).
        const uint32_t C0 = j0 ? dup16(0xD440u) : dup16(0xE404u), C1 = j0 ? dup16(0xCD00u) : dup16(0xDC10u);
        const int sh0 = 2 * j0 + 2 - (4 * tp + j0), sh1 = 2 * j1 + 2 - (4 * tp + j1);   // may be negative
        const uint32_t qa = x.q0[i], qb = x.q1[i], qa8 = qa >> 8, qb8 = qb >> 8;
        const uint32_t ma = x.m0[i], mb = x.m1[i], ma8 = ma >> 8, mb8 = mb >> 8;
        A[0] = hadd2(and_or(qa, M0, and_or(shl(ma, sh0), B0, G0)), C0);
        A[1] = hadd2(and_or(qb, M0, and_or(shl(mb, sh0), B0, G0)), C0);
        A[2] = hadd2(and_or(qa8, M0, and_or(shl(ma8, sh0), B0, G0)), C0);
        A[3] = hadd2(and_or(qb8, M0, and_or(shl(mb8, sh0), B0, G0)), C0);
        A[4] = hadd2(and_or(qa, M1, and_or(shl(ma, sh1), B1, G1)), C1);
        A[5] = hadd2(and_or(qb, M1, and_or(shl(mb, sh1), B1, G1)), C1);
        A[6] = hadd2(and_or(qa8, M1, and_or(shl(ma8, sh1), B1, G1)), C1);
        A[7] = hadd2(and_or(qb8, M1, and_or(shl(mb8, sh1), B1, G1)), C1);
    }
    __device__ static __forceinline__ void epi(const Ctx& x, const float (&c)[4][4], float4 xm0, float4 xm1, int, int,
                                               float& y0, float& y1) {
        auto sc = [](uint32_t S, int k) { return ubyte_f(S, k) - 32.0f; };
        y0 += x.d0 * (xm0.y * fmaf(sc(x.S0, 0), csum_g(c[0]), sc(x.S0, 1) * csum_g(c[1])) +
                      xm1.y * fmaf(sc(x.S0, 2), csum_g(c[2]), sc(x.S0, 3) * csum_g(c[3])));
        y1 += x.d1 * (xm0.y * fmaf(sc(x.S1, 0), csum_g8(c[0]), sc(x.S1, 1) * csum_g8(c[1])) +
                      xm1.y * fmaf(sc(x.S1, 2), csum_g8(c[2]), sc(x.S1, 3) * csum_g8(c[3])));
    }
};

// B fragments of the MT tokens: in registers for one token (the whole
// chunk's steps), from shared memory step by step for more.
struct BRegs {
    XB x0, x1;
    __device__ __forceinline__ uint2 b(int, int X, int i) const {
        return X ? make_uint2(x1.b[2 * i], x1.b[2 * i + 1]) : make_uint2(x0.b[2 * i], x0.b[2 * i + 1]);
    }
};
template <int MT>
struct BSmem {
    const uint8_t* p[MT][2];   // plane of the thread's column in x-blocks X0, X1 of each token
    bool own;
    __device__ __forceinline__ uint2 b(int m, int X, int i) const {
        return own ? lds64(p[m][X] + 8 * i) : make_uint2(0u, 0u);
    }
};

// One unit for MT tokens: each step's A fragments are converted once and
// multiplied with every token's B.  A token's accumulators: the two halves
// of each x-block for the 16-weight-group types (c[0], c[1] for X0, c[2],
// c[3] for X1), else one per x-block (c[0] X0, c[2] X1; c[1] and c[3] stay
// zero and fold away).  The first step of each starts from zero.
template <int T, int MT, class BP>
__device__ __forceinline__ void run_unit(const uint8_t* r0, const uint8_t* r1, const BP& bp, const float4 (&xm0)[MT],
                                         const float4 (&xm1)[MT], int t, int nvb, float (&y0)[MT], float (&y1)[MT]) {
    using U = HU<T>;
    typename U::Ctx cx;
    U::load(cx, r0, r1, t);
    float c[MT][4][4] = {};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t A[8];
        U::conv(cx, i, t, A);
        const int ch = U::kGroup16 ? (i >> 2) : 0;
        const bool first = U::kGroup16 ? (i & 3) == 0 : i == 0;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint2 b0 = bp.b(m, 0, i), b1 = bp.b(m, 1, i);
            if (first) {
                mma16816_z(c[m][ch], A[0], A[1], A[2], A[3], b0.x, b0.y);
                mma16816_z(c[m][2 + ch], A[4], A[5], A[6], A[7], b1.x, b1.y);
            } else {
                mma16816(c[m][ch], A[0], A[1], A[2], A[3], b0.x, b0.y);
                mma16816(c[m][2 + ch], A[4], A[5], A[6], A[7], b1.x, b1.y);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) U::epi(cx, c[m], xm0[m], xm1[m], t, nvb, y0[m], y1[m]);
}

}  // namespace hm
}  // namespace qk
