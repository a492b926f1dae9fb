// qk_formats.cuh -- device-side block geometry and unpackers.
//
// Every block is consumed in "halves": 16 weights whose positions along the
// row are consecutive.  A block of 32 weights has 2 halves; a 256-weight
// super-block has 16, grouped in 8 "units" of two halves that share their
// code bytes.  half(blk, unit, h, w) writes the 16 fp32 weights of half h of
// `unit`; koff(unit, h) is the position of its first weight in the block.
//
// Formats (see include/qk.h for the byte layouts and sources):
//   Q4_K  w = (d*sc)*q - dmin*m        ("Hitchhiker's Guide", 11.2 figure)
//   Q6_K  w = (d*sc)*(q - 32)
//   Q8_0  w = d*q                      ("Hitchhiker's Guide", 11.1)
//   Q5_0  w = d*(q - 16)
//   Q4_0  w = d*(q - 8)                ("Hitchhiker's Guide", 11.1 figure)
//   Q5_K  w = (d*sc)*q - dmin*m, 5-bit q (the GGUF k-quant layout: only the
//         size, 5.5 bits/weight, is on the pages)
//   Q2_K  w = (d*sc)*q - dmin*m per 16 weights, 2-bit q (GGUF layout; the
//         pages give 2.5-2.6 bits/weight)
//   Q3_K  w = (d*sc)*q per 16 weights, q in -4..3, signed 6-bit sc (GGUF
//         layout; the pages give 3.4-4.0 bits/weight)
// Each product before the last rounding is exact in fp32 (an fp16 d has 11
// significant bits, a scale at most 8, a code at most 8), so the weights are
// bit-identical to the formula evaluated in fp32 whatever the contraction.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qk {

enum : int { T_Q4_K = 1, T_Q6_K = 2, T_Q8_0 = 3, T_Q5_0 = 4, T_Q4_0 = 5, T_Q5_K = 6, T_Q2_K = 7, T_Q3_K = 8 };

// 16-bit and 32-bit little-endian loads from a 2-byte-aligned address that
// never touch a byte outside [p, p + size).
__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
    return *reinterpret_cast<const uint16_t*>(p);
}
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {
    return ld_u16(p) | (ld_u16(p + 2) << 16);
}
__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}
__device__ __forceinline__ uint32_t byte_of(const uint32_t (&w)[4], int i) {
    return (w[i >> 2] >> (8 * (i & 3))) & 255u;
}

template <int T> struct Fmt;

// Every type exposes:
//   codes16(blk, u, h, c)  the 16 integer codes of half h of unit u
//   params(blk, u, h, A, B) the fp32 factors with w = A * (code - OFF) - B
// and half() evaluates that formula; A and B are exact fp32 products.
template <int T>
__device__ __forceinline__ void dequant_half(const uint8_t* blk, int u, int h, float (&w)[16]) {
    int c[16];
    float A, B;
    Fmt<T>::codes16(blk, u, h, c);
    Fmt<T>::params(blk, u, h, A, B);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = A * (float)(c[i] - Fmt<T>::OFF) - B;
}

// ---------------------------------------------------------------- Q4_K --
// Bytes 0-1 d, 2-3 dmin, 4-15 scales s[12], 16-143 qs[128].
// Sub-block j (weights 32j..32j+31):
//   j < 4:  sc = s[j] & 63,                          m = s[j+4] & 63
//   j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4
// Weight 64c + 32h + l is nibble h of qs[32c + l].
// Unit u = 2c + hp covers bytes qs[32c + 16hp .. +15]: half 0 is sub-block 2c,
// half 1 sub-block 2c+1.  w = (d*sc)*q - dmin*m.
template <> struct Fmt<T_Q4_K> {
    static constexpr int BB = 144, BE = 256, UPB = 8, OFF = 0;
    __device__ static __forceinline__ int koff(int u, int h) { return 64 * (u >> 1) + 32 * h + 16 * (u & 1); }
    __device__ static __forceinline__ void scale_min(const uint8_t* blk, int j, uint32_t& sc, uint32_t& m) {
        const uint8_t* s = blk + 4;
        if (j < 4) {
            sc = s[j] & 63u;
            m = s[j + 4] & 63u;
        } else {
            sc = (s[j + 4] & 15u) | ((uint32_t)(s[j - 4] >> 6) << 4);
            m = ((uint32_t)s[j + 4] >> 4) | ((uint32_t)(s[j] >> 6) << 4);
        }
    }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int u, int h, int (&c)[16]) {
        const uint4 q4 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * (u >> 1) + 16 * (u & 1));
        const uint32_t q[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = (int)((byte_of(q, i) >> (4 * h)) & 15u);
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int u, int h, float& A, float& B) {
        uint32_t sc, m;
        scale_min(blk, 2 * (u >> 1) + h, sc, m);
        A = h2f(ld_u16(blk)) * (float)sc;
        B = h2f(ld_u16(blk + 2)) * (float)m;
    }
};

// ---------------------------------------------------------------- Q5_K --
// Bytes 0-1 d, 2-3 dmin, 4-15 scales (packed as Q4_K's), 16-47 qh, 48-175 qs.
// Weight 64c + 32h + l: low 4 bits are nibble h of qs[32c + l] (as Q4_K),
// the fifth bit is bit 2c + h of qh[l].  Units and halves as Q4_K's.
template <> struct Fmt<T_Q5_K> {
    static constexpr int BB = 176, BE = 256, UPB = 8, OFF = 0;
    __device__ static __forceinline__ int koff(int u, int h) { return 64 * (u >> 1) + 32 * h + 16 * (u & 1); }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int u, int h, int (&c)[16]) {
        const int cg = u >> 1, hp = u & 1;
        const uint4 q4 = *reinterpret_cast<const uint4*>(blk + 48 + 32 * cg + 16 * hp);
        const uint4 h4 = *reinterpret_cast<const uint4*>(blk + 16 + 16 * hp);
        const uint32_t q[4] = {q4.x, q4.y, q4.z, q4.w};
        const uint32_t hb[4] = {h4.x, h4.y, h4.z, h4.w};
        const int sh = 2 * cg + h;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            c[i] = (int)(((byte_of(q, i) >> (4 * h)) & 15u) | (((byte_of(hb, i) >> sh) & 1u) << 4));
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int u, int h, float& A, float& B) {
        uint32_t sc, m;
        Fmt<T_Q4_K>::scale_min(blk, 2 * (u >> 1) + h, sc, m);
        A = h2f(ld_u16(blk)) * (float)sc;
        B = h2f(ld_u16(blk + 2)) * (float)m;
    }
};

// ---------------------------------------------------------- Q2_K, Q3_K --
// Sixteen 16-weight groups; half i of the super-block (unit i/2, h = i%2) is
// group i, weights 16i..16i+15: t = i/8, j = (i%8)/2, k = i%2, and code l is
// bits 2j..2j+1 of byte 32t + 16k + l of the 2-bit plane.
// Q2_K: bytes 0-15 scale (low nibble) / min (high nibble) per group, 16-79
//       the plane, 80-81 d, 82-83 dmin.  w = (d*sc)*q - dmin*m.
// Q3_K: bytes 0-31 hmask, 32-95 the plane, 96-107 the scales, 108-109 d.  The
//       code's third bit is bit 4t + j of hmask[16k + l]; q = lo2 - 4 when it
//       is clear.  Scale of group g: low 4 bits = nibble g/8 of byte 96 + g%8,
//       high 2 bits = bits 2(g/4).. of byte 104 + g%4; value minus 32.
//       w = (d*sc)*q.
__device__ __forceinline__ int plane_base(int i) { return 32 * (i >> 3) + 16 * (i & 1); }
__device__ __forceinline__ int plane_shift(int i) { return 2 * ((i & 7) >> 1); }

template <> struct Fmt<T_Q2_K> {
    static constexpr int BB = 84, BE = 256, UPB = 8, OFF = 0;
    __device__ static __forceinline__ int koff(int u, int h) { return 32 * u + 16 * h; }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int u, int h, int (&c)[16]) {
        const int i = 2 * u + h;
        const uint8_t* p = blk + 16 + plane_base(i);
        const uint32_t q[4] = {ld_u32_a2(p), ld_u32_a2(p + 4), ld_u32_a2(p + 8), ld_u32_a2(p + 12)};
#pragma unroll
        for (int l = 0; l < 16; ++l) c[l] = (int)((byte_of(q, l) >> plane_shift(i)) & 3u);
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int u, int h, float& A, float& B) {
        const uint32_t sm = blk[2 * u + h];
        A = h2f(ld_u16(blk + 80)) * (float)(sm & 15u);
        B = h2f(ld_u16(blk + 82)) * (float)(sm >> 4);
    }
};

template <> struct Fmt<T_Q3_K> {
    static constexpr int BB = 110, BE = 256, UPB = 8, OFF = 0;
    __device__ static __forceinline__ int koff(int u, int h) { return 32 * u + 16 * h; }
    __device__ static __forceinline__ int scale(const uint8_t* blk, int g) {
        const uint32_t lo4 = (blk[96 + (g & 7)] >> (4 * (g >> 3))) & 15u;
        const uint32_t hi2 = (blk[104 + (g & 3)] >> (2 * (g >> 2))) & 3u;
        return (int)(lo4 | (hi2 << 4)) - 32;
    }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int u, int h, int (&c)[16]) {
        const int i = 2 * u + h;
        const uint8_t* p = blk + 32 + plane_base(i);
        const uint8_t* m = blk + 16 * (i & 1);
        const uint32_t q[4] = {ld_u32_a2(p), ld_u32_a2(p + 4), ld_u32_a2(p + 8), ld_u32_a2(p + 12)};
        const uint32_t hm[4] = {ld_u32_a2(m), ld_u32_a2(m + 4), ld_u32_a2(m + 8), ld_u32_a2(m + 12)};
        const int hb = 4 * (i >> 3) + ((i & 7) >> 1);
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const int lo2 = (int)((byte_of(q, l) >> plane_shift(i)) & 3u);
            c[l] = ((byte_of(hm, l) >> hb) & 1u) ? lo2 : lo2 - 4;
        }
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int u, int h, float& A, float& B) {
        A = h2f(ld_u16(blk + 108)) * (float)scale(blk, 2 * u + h);
        B = 0.0f;
    }
};

// ---------------------------------------------------------------- Q6_K --
// Bytes 0-127 ql, 128-191 qh, 192-207 int8 scales, 208-209 d.
// Weight n = 128t + 32g + l: low 4 bits = nibble (g >= 2) of ql[64t + 32(g&1) + l],
// high 2 bits = bits 2g..2g+1 of qh[32t + l]; scale sc[n / 16].
// Unit u = 4t + 2gp + hp, l = 16hp + i: half h is group g = gp + 2h (both
// halves read the same ql bytes, low then high nibble).  w = (d*sc)*(q - 32).
template <> struct Fmt<T_Q6_K> {
    static constexpr int BB = 210, BE = 256, UPB = 8, OFF = 32;
    __device__ static __forceinline__ int koff(int u, int h) {
        return 128 * (u >> 2) + 32 * (((u >> 1) & 1) + 2 * h) + 16 * (u & 1);
    }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int u, int h, int (&c)[16]) {
        const int t = u >> 2, gp = (u >> 1) & 1, hp = u & 1, g = gp + 2 * h;
        const uint8_t* ql = blk + 64 * t + 32 * gp + 16 * hp;
        const uint8_t* qh = blk + 128 + 32 * t + 16 * hp;
        const uint32_t lw[4] = {ld_u32_a2(ql), ld_u32_a2(ql + 4), ld_u32_a2(ql + 8), ld_u32_a2(ql + 12)};
        const uint32_t hw[4] = {ld_u32_a2(qh), ld_u32_a2(qh + 4), ld_u32_a2(qh + 8), ld_u32_a2(qh + 12)};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t lo = (byte_of(lw, i) >> (4 * h)) & 15u;
            const uint32_t hi = (byte_of(hw, i) >> (2 * g)) & 3u;
            c[i] = (int)(lo | (hi << 4));
        }
    }
    __device__ static __forceinline__ int scale_index(int u, int h) {
        return 8 * (u >> 2) + 2 * (((u >> 1) & 1) + 2 * h) + (u & 1);
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int u, int h, float& A, float& B) {
        A = h2f(ld_u16(blk + 208)) * (float)(int)(int8_t)blk[192 + scale_index(u, h)];
        B = 0.0f;
    }
};

// ---------------------------------------------------------------- Q8_0 --
// Bytes 0-1 d, 2-33 int8 codes.  One unit; half h = codes 16h..16h+15.  w = d*q.
template <> struct Fmt<T_Q8_0> {
    static constexpr int BB = 34, BE = 32, UPB = 1, OFF = 0;
    __device__ static __forceinline__ int koff(int, int h) { return 16 * h; }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int, int h, int (&c)[16]) {
        const uint8_t* p = blk + 2 + 16 * h;
        const uint32_t q[4] = {ld_u32_a2(p), ld_u32_a2(p + 4), ld_u32_a2(p + 8), ld_u32_a2(p + 12)};
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = (int)(int8_t)byte_of(q, i);
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int, int, float& A, float& B) {
        A = h2f(ld_u16(blk));
        B = 0.0f;
    }
};

// ---------------------------------------------------------------- Q5_0 --
// Bytes 0-1 d, 2-5 fifth-bit word qh (bit j = element j), 6-21 qs.
// Element j < 16: low nibble of qs[j]; element j + 16: high nibble of qs[j].
// w = d*(q - 16).
template <> struct Fmt<T_Q5_0> {
    static constexpr int BB = 22, BE = 32, UPB = 1, OFF = 16;
    __device__ static __forceinline__ int koff(int, int h) { return 16 * h; }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int, int h, int (&c)[16]) {
        const uint32_t qh = ld_u32_a2(blk + 2) >> (16 * h);
        const uint8_t* p = blk + 6;
        const uint32_t q[4] = {ld_u32_a2(p), ld_u32_a2(p + 4), ld_u32_a2(p + 8), ld_u32_a2(p + 12)};
#pragma unroll
        for (int i = 0; i < 16; ++i)
            c[i] = (int)(((byte_of(q, i) >> (4 * h)) & 15u) | (((qh >> i) & 1u) << 4));
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int, int, float& A, float& B) {
        A = h2f(ld_u16(blk));
        B = 0.0f;
    }
};

// ---------------------------------------------------------------- Q4_0 --
// Bytes 0-1 d, 2-17 qs.  Element j < 16: low nibble of qs[j]; element j + 16:
// high nibble of qs[j].  w = d*(q - 8).
template <> struct Fmt<T_Q4_0> {
    static constexpr int BB = 18, BE = 32, UPB = 1, OFF = 8;
    __device__ static __forceinline__ int koff(int, int h) { return 16 * h; }
    __device__ static __forceinline__ void codes16(const uint8_t* blk, int, int h, int (&c)[16]) {
        const uint8_t* p = blk + 2;
        const uint32_t q[4] = {ld_u32_a2(p), ld_u32_a2(p + 4), ld_u32_a2(p + 8), ld_u32_a2(p + 12)};
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = (int)((byte_of(q, i) >> (4 * h)) & 15u);
    }
    __device__ static __forceinline__ void params(const uint8_t* blk, int, int, float& A, float& B) {
        A = h2f(ld_u16(blk));
        B = 0.0f;
    }
};

}  // namespace qk
