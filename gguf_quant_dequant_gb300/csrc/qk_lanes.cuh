// qk_lanes.cuh -- the per-lane decoders of the fused dequant-GEMV kernels.
//
// A lane owns 64 weights of one row segment of kKR = 2048 weights (two
// 32-element x-blocks) and forms its share of sum w*x against the 24-bit
// fixed-point limbs of x: x ~= s * (65536a + 256b + c) per 32-block, three
// signed 8-bit limbs per element, so that sum q*x is an exact integer sum of
// dp4a products ("Local LLM inference": dequantize inside the dot product).
// Scales are applied once per 16 or 32 weights; the min / code-offset terms
// use the fp32 sums of x per block half.
#pragma once
#include <cstdint>

#include "qk_formats.cuh"

namespace qk {
namespace gv {

constexpr int kKR = 2048;              // weights per row per stage
constexpr int kXB = kKR / 32;          // x-blocks per stage
constexpr int kXBytes = 112;           // prepped bytes per x-block: a[32] b[32] c[32] + float4
constexpr float kXMax = 8323072.0f;    // 127 * 65536: largest |X| of a 3-limb value

// ---------------------------------------------------------------------------
// dp4a: four signed byte products added to c.
// (The accumulator is an in-place operand, so no register copy is needed.)
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    asm("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}

// The same with unsigned bytes in a (0..255) and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// N little-endian words starting at a 2-byte-aligned shared-memory address:
// aligned 32-bit loads joined by funnel shifts (the slot has slack after the
// segment, so reading one word past the end stays inside the slot).
template <int N>
__device__ __forceinline__ void lds_words_a2(const uint8_t* p, uint32_t (&w)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8;   // 0 or 16
    uint32_t prev = lds32(base);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t next = lds32(base + 4 * (i + 1));
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

// The lane's prepped activations for one activation row: limbs of its two
// x-blocks and their metadata {s, sum lo16, sum hi16, sum 32}.
struct XL {
    uint32_t a[2][8], b[2][8], c[2][8];
    float4 meta[2];
};

// The lane's two x-blocks from the stage's shared-memory copy of the prepped
// activations (x-blocks j0, j1 of the stage).
__device__ __forceinline__ void load_x(const uint8_t* xs, int j0, int j1, XL& x) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint8_t* p = xs + (j == 0 ? j0 : j1) * kXBytes;
        uint4 v[7];
#pragma unroll
        for (int q = 0; q < 7; ++q) v[q] = lds128(p + 16 * q);
        const uint32_t* u = reinterpret_cast<const uint32_t*>(v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x.a[j][i] = u[i];
            x.b[j][i] = u[8 + i];
            x.c[j][i] = u[16 + i];
        }
        x.meta[j] = make_float4(__uint_as_float(u[24]), __uint_as_float(u[25]), __uint_as_float(u[26]),
                                __uint_as_float(u[27]));
    }
}

// Exact integer dot of 4 code words (16 codes) with 16 limb triples, limb
// words w0..w0+3 of x-block j; accumulates into A, B, C.  Every code byte
// fed here is a valid signed byte (Q4_K 0..15, Q6_K 0..63, Q5_0 0..31, Q4_0 0..15, Q8_0
// signed), so the signed x signed form is used throughout.
__device__ __forceinline__ void dot16(const uint32_t (&q)[4], const XL& x, int j, int w0, int& A, int& B, int& C) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        A = dp4a_ss(q[i], x.a[j][w0 + i], A);
        B = dp4a_ss(q[i], x.b[j][w0 + i], B);
        C = dp4a_ss(q[i], x.c[j][w0 + i], C);
    }
}

// 65536A + 256B + C as fp32 (B*256 + C is formed exactly in int32).
__device__ __forceinline__ float limbs_to_f(int A, int B, int C) {
    return fmaf((float)A, 65536.0f, (float)(B * 256 + C));
}

// 65536*Ia + 256*Ib + Ic as fp32, for sums too large to pre-combine in int32.
__device__ __forceinline__ float limbs3_to_f(int A, int B, int C) {
    return fmaf((float)A, 65536.0f, fmaf((float)B, 256.0f, (float)C));
}

// ---------------------------------------------------------------------------
// Lane decoders.  Each returns one lane's share of y[row] for one activation
// row: its 64 weights of the row segment `seg` (the stage's bytes of this row,
// already offset past the alignment remainder) against its limbs x.

template <int T> struct Lane;

// Q4_K: lane l -> super-block sb = l/4 of the stage, code group c = l%4
// (bytes qs[32c..32c+31]): low nibbles are sub-block 2c (x-block 2l), high
// nibbles sub-block 2c+1 (x-block 2l+1).  w = (d*sc)*q - (dmin*m).
template <> struct Lane<T_Q4_K> {
    int sb, c, sh;
    bool hi4;  // c >= 2: sub-blocks 4..7, whose 6-bit fields are split
    __device__ __forceinline__ explicit Lane(int lane) : sb(lane >> 2), c(lane & 3), sh(16 * (lane & 1)), hi4(c >= 2) {}
    __device__ __forceinline__ bool valid(int nblk) const { return sb < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        const uint8_t* blk = seg + sb * 144;
        const uint4 h = lds128(blk);
        const uint4 q0 = lds128(blk + 16 + 32 * c), q1 = lds128(blk + 32 + 32 * c);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint32_t lo[2][4], hi[2][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo[i >> 2][i & 3] = w[i] & 0x0F0F0F0Fu;
            hi[i >> 2][i & 3] = (w[i] >> 4) & 0x0F0F0F0Fu;
        }
        int A0 = 0, B0 = 0, C0 = 0, A1 = 0, B1 = 0, C1 = 0;
        dot16(lo[0], x, 0, 0, A0, B0, C0);
        dot16(lo[1], x, 0, 4, A0, B0, C0);
        dot16(hi[0], x, 1, 0, A1, B1, C1);
        dot16(hi[1], x, 1, 4, A1, B1, C1);
        // 6-bit scales and mins of sub-blocks 2c and 2c+1 (bytes s0..3 = h.y,
        // s4..7 = h.z, s8..11 = h.w).  j < 4: sc = s[j] & 63, m = s[j+4] & 63;
        // j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
        //         m  = (s[j+4] >> 4) | (s[j] >> 6) << 4.
        const uint32_t lsc = hi4 ? h.w : h.y, lm = hi4 ? (h.w >> 4) : h.z;
        const uint32_t lmask = hi4 ? 15u : 63u, hmask = hi4 ? 3u : 0u;
        const uint32_t sc0 = ((lsc >> sh) & lmask) | (((h.y >> (sh + 6)) & hmask) << 4);
        const uint32_t sc1 = ((lsc >> (sh + 8)) & lmask) | (((h.y >> (sh + 14)) & hmask) << 4);
        const uint32_t m0 = ((lm >> sh) & lmask) | (((h.z >> (sh + 6)) & hmask) << 4);
        const uint32_t m1 = ((lm >> (sh + 8)) & lmask) | (((h.z >> (sh + 14)) & hmask) << 4);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        const float f0 = limbs_to_f(A0, B0, C0) * x.meta[0].x;
        const float f1 = limbs_to_f(A1, B1, C1) * x.meta[1].x;
        return d * fmaf((float)sc0, f0, (float)sc1 * f1) - dmin * fmaf((float)m0, x.meta[0].w, (float)m1 * x.meta[1].w);
    }
};

// Q5_K: the Q4_K lane mapping (lane l -> super-block l/4, code group
// c = l%4, x-blocks 2l and 2l+1) with each code's fifth bit merged in from
// the 32-byte plane: bit 2c of qh[k] belongs to the low-nibble code of
// qs[32c + k], bit 2c + 1 to its high-nibble code.  Codes 0..31 are valid
// signed bytes for the signed x signed dp4a.  w = (d*sc)*q - dmin*m.
template <> struct Lane<T_Q5_K> {
    int sb, c, sh;
    bool hi4;  // c >= 2: sub-blocks 4..7, whose 6-bit fields are split
    __device__ __forceinline__ explicit Lane(int lane) : sb(lane >> 2), c(lane & 3), sh(16 * (lane & 1)), hi4(c >= 2) {}
    __device__ __forceinline__ bool valid(int nblk) const { return sb < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        const uint8_t* blk = seg + sb * 176;
        const uint4 h = lds128(blk);
        const uint4 e0 = lds128(blk + 16), e1 = lds128(blk + 32);                    // qh[0..31]
        const uint4 q0 = lds128(blk + 48 + 32 * c), q1 = lds128(blk + 64 + 32 * c);  // qs[32c..32c+31]
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        uint32_t lo[2][4], hi[2][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t b = e[i] >> (2 * c);   // bit 0: low code's fifth bit, bit 1: high code's
            lo[i >> 2][i & 3] = (w[i] & 0x0F0F0F0Fu) | ((b << 4) & 0x10101010u);
            hi[i >> 2][i & 3] = ((w[i] >> 4) & 0x0F0F0F0Fu) | ((b << 3) & 0x10101010u);
        }
        int A0 = 0, B0 = 0, C0 = 0, A1 = 0, B1 = 0, C1 = 0;
        dot16(lo[0], x, 0, 0, A0, B0, C0);
        dot16(lo[1], x, 0, 4, A0, B0, C0);
        dot16(hi[0], x, 1, 0, A1, B1, C1);
        dot16(hi[1], x, 1, 4, A1, B1, C1);
        // Scales and mins of sub-blocks 2c, 2c+1: the Q4_K packing.
        const uint32_t lsc = hi4 ? h.w : h.y, lm = hi4 ? (h.w >> 4) : h.z;
        const uint32_t lmask = hi4 ? 15u : 63u, hmask = hi4 ? 3u : 0u;
        const uint32_t sc0 = ((lsc >> sh) & lmask) | (((h.y >> (sh + 6)) & hmask) << 4);
        const uint32_t sc1 = ((lsc >> (sh + 8)) & lmask) | (((h.y >> (sh + 14)) & hmask) << 4);
        const uint32_t m0 = ((lm >> sh) & lmask) | (((h.z >> (sh + 6)) & hmask) << 4);
        const uint32_t m1 = ((lm >> (sh + 8)) & lmask) | (((h.z >> (sh + 14)) & hmask) << 4);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        const float f0 = limbs3_to_f(A0, B0, C0) * x.meta[0].x;
        const float f1 = limbs3_to_f(A1, B1, C1) * x.meta[1].x;
        return d * fmaf((float)sc0, f0, (float)sc1 * f1) - dmin * fmaf((float)m0, x.meta[0].w, (float)m1 * x.meta[1].w);
    }
};

// Q2_K and Q3_K: lane l -> super-block l/4, c = l%4, x-blocks 2l and 2l+1:
// weights 64c .. 64c+63 = 16-weight groups 4c .. 4c+3.  All of them take
// their 2-bit codes from bytes 32t .. 32t+31 of the code plane (t = c/2):
// x-block e uses bits 2j.. with j = 2(c%2) + e, bytes 0-15 for its first
// group and 16-31 for its second.  Per group the dp4a sums stay separate and
// are weighted by the group's integer scale before the conversion to fp32.
template <> struct Lane<T_Q2_K> {
    int sb, c;
    __device__ __forceinline__ explicit Lane(int lane) : sb(lane >> 2), c(lane & 3) {}
    __device__ __forceinline__ bool valid(int nblk) const { return sb < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    // Blocks are 84 bytes: 4-byte aligned wherever a row starts on 4 bytes.
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        const uint8_t* blk = seg + sb * 84;
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = lds32(blk + 16 + 32 * (c >> 1) + 4 * i);
        const uint32_t sm = lds32(blk + 4 * c);   // (scale, min) bytes of groups 4c .. 4c+3
        const uint32_t dd = lds32(blk + 80);      // d, dmin
        float r = 0.0f, rm = 0.0f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int sh = 2 * (2 * (c & 1) + e);
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo[i] = (q[i] >> sh) & 0x03030303u;
                hi[i] = (q[4 + i] >> sh) & 0x03030303u;
            }
            int A0 = 0, B0 = 0, C0 = 0, A1 = 0, B1 = 0, C1 = 0;
            dot16(lo, x, e, 0, A0, B0, C0);
            dot16(hi, x, e, 4, A1, B1, C1);
            const int s0 = (int)((sm >> (16 * e)) & 15u), s1 = (int)((sm >> (16 * e + 8)) & 15u);
            const float m0 = (float)((sm >> (16 * e + 4)) & 15u), m1 = (float)((sm >> (16 * e + 12)) & 15u);
            const float4 mt = x.meta[e];
            r = fmaf(mt.x, limbs3_to_f(s0 * A0 + s1 * A1, s0 * B0 + s1 * B1, s0 * C0 + s1 * C1), r);
            rm = fmaf(m0, mt.y, fmaf(m1, mt.z, rm));
        }
        return h2f(dd & 0xFFFFu) * r - h2f(dd >> 16) * rm;
    }
};

template <> struct Lane<T_Q3_K> {
    int sb, c;
    __device__ __forceinline__ explicit Lane(int lane) : sb(lane >> 2), c(lane & 3) {}
    __device__ __forceinline__ bool valid(int nblk) const { return sb < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    // Blocks are 110 bytes (2-byte aligned): words through funnel shifts.
    // A code u = lo2 | mask bit << 2 (0..7) is q + 4: sum q x = sum u x - 4 sum x.
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        const uint8_t* blk = seg + sb * 110;
        uint32_t q[8], hm[8], sw[1];
        lds_words_a2<8>(blk + 32 + 32 * (c >> 1), q);
        lds_words_a2<8>(blk, hm);
        lds_words_a2<1>(blk + 96 + 4 * (c & 1), sw);      // low nibbles of groups 4c.. (byte g % 8)
        uint32_t sh2[1];
        lds_words_a2<1>(blk + 104, sh2);                   // high bit pairs (byte 8 + g % 4)
        const uint32_t lo4w = sw[0] >> (4 * (c >> 1));     // nibble g / 8 of bytes 4(c%2) ..
        const float d = h2f(ld_u16(blk + 108));
        float r = 0.0f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * (c & 1) + e, sh = 2 * j, hb = 4 * (c >> 1) + j;
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo[i] = ((q[i] >> sh) & 0x03030303u) | (((hm[i] >> hb) & 0x01010101u) << 2);
                hi[i] = ((q[4 + i] >> sh) & 0x03030303u) | (((hm[4 + i] >> hb) & 0x01010101u) << 2);
            }
            int A0 = 0, B0 = 0, C0 = 0, A1 = 0, B1 = 0, C1 = 0;
            dot16(lo, x, e, 0, A0, B0, C0);
            dot16(hi, x, e, 4, A1, B1, C1);
            // Groups 4c + 2e and 4c + 2e + 1: byte k = 2e (+1) of the words.
            int sc[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int g = 4 * c + 2 * e + k;
                const uint32_t l4 = (lo4w >> (8 * (2 * e + k))) & 15u;
                const uint32_t h2 = (sh2[0] >> (8 * (g & 3) + 2 * (g >> 2))) & 3u;
                sc[k] = (int)(l4 | (h2 << 4)) - 32;
            }
            const float4 mt = x.meta[e];
            const float T = limbs3_to_f(sc[0] * A0 + sc[1] * A1, sc[0] * B0 + sc[1] * B1, sc[0] * C0 + sc[1] * C1);
            r += fmaf(mt.x, T, -4.0f * fmaf((float)sc[0], mt.y, (float)sc[1] * mt.z));
        }
        return d * r;
    }
};

// Byte k of v as an exact fp32 (0..255), via the 2^23 magic constant.
__device__ __forceinline__ float byte_to_f(uint32_t v, uint32_t sel) {
    return __uint_as_float(__byte_perm(v, 0x4B000000u, sel)) - 8388608.0f;
}

// Q4_K, two rows at once (independent instruction streams), lean scale
// decode: one byte permute gathers the four 6-bit fields of this lane's
// sub-blocks 2c and 2c+1 from the 12 scale bytes.
struct Q4KFast {
    uint32_t off_h, off_q;      // byte offsets of the header and of the lane's 32 code bytes
    uint32_t sel_yz, sel_w;     // byte_perm selectors
    bool hi4;
    __device__ __forceinline__ explicit Q4KFast(int lane) {
        const int sb = lane >> 2, c = lane & 3, j = 2 * (c & 1);
        off_h = sb * 144;
        off_q = sb * 144 + 16 + 32 * c;
        hi4 = c >= 2;
        sel_yz = (uint32_t)(j | ((j + 1) << 4) | ((4 + j) << 8) | ((5 + j) << 12));
        sel_w = (uint32_t)(j | ((j + 1) << 4) | (j << 8) | ((j + 1) << 12));
    }
    // [sc0, sc1, m0, m1] as bytes.
    // Both layouts are computed and one is selected (no divergent branch).
    __device__ __forceinline__ uint32_t fields(const uint4& h) const {
        const uint32_t p = __byte_perm(h.y, h.z, sel_yz);   // [s_j, s_j+1, s_j+4, s_j+5]
        const uint32_t q = __byte_perm(h.w, 0, sel_w);       // [s_j+8, s_j+9, s_j+8, s_j+9]
        const uint32_t split = (q & 0x00000F0Fu) | ((q >> 4) & 0x0F0F0000u) | ((p >> 2) & 0x30303030u);
        return hi4 ? split : (p & 0x3F3F3F3Fu);
    }
    __device__ __forceinline__ float one(const uint8_t* seg, const XL& x, float s0, float s1) const {
        const uint4 h = lds128(seg + off_h);
        const uint4 q0 = lds128(seg + off_q), q1 = lds128(seg + off_q + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        int A0 = 0, B0 = 0, C0 = 0, A1 = 0, B1 = 0, C1 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // Low codes 0..15 are valid signed bytes (signed x signed dp4a);
            // the high codes stay in place as 16 * code (unsigned bytes), the
            // factor 16 is taken out of the sum below.
            const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi16 = w[i] & 0xF0F0F0F0u;
            A0 = dp4a_ss(lo, x.a[0][i], A0);
            B0 = dp4a_ss(lo, x.b[0][i], B0);
            C0 = dp4a_ss(lo, x.c[0][i], C0);
            A1 = dp4a_us(hi16, x.a[1][i], A1);
            B1 = dp4a_us(hi16, x.b[1][i], B1);
            C1 = dp4a_us(hi16, x.c[1][i], C1);
        }
        const uint32_t f = fields(h);
        const float sc0 = byte_to_f(f, 0x7440), sc1 = byte_to_f(f, 0x7441);
        const float m0 = byte_to_f(f, 0x7442), m1 = byte_to_f(f, 0x7443);
        const float t0 = limbs_to_f(A0, B0, C0) * s0, t1 = limbs_to_f(A1, B1, C1) * (s1 * 0.0625f);
        const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
        return d * fmaf(sc0, t0, sc1 * t1) - dmin * fmaf(m0, x.meta[0].w, m1 * x.meta[1].w);
    }
};

// Q6_K: lane l -> super-block sb = l/4, u = l%4 = (t = u/2, gp = u%2):
// groups g = gp (low nibbles of ql[64t + 32gp + l'], qh bits 2gp) and
// g = gp + 2 (high nibbles, qh bits 2gp + 4); group g is x-block 4t + g of the
// super-block, with int8 scales sc[8t + 2g] (first 16) and sc[8t + 2g + 1].
// w = d * sc * (q - 32).
template <> struct Lane<T_Q6_K> {
    int sb, t, gp;
    __device__ __forceinline__ explicit Lane(int lane) : sb(lane >> 2), t((lane >> 1) & 1), gp(lane & 1) {}
    __device__ __forceinline__ bool valid(int nblk) const { return sb < nblk; }
    __device__ __forceinline__ void xblocks(int, int& j0, int& j1) const {
        j0 = 8 * sb + 4 * t + gp;
        j1 = j0 + 2;
    }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        const uint8_t* blk = seg + sb * 210;
        uint32_t ql[8], qh[8];
        lds_words_a2<8>(blk + 64 * t + 32 * gp, ql);
        lds_words_a2<8>(blk + 128 + 32 * t, qh);
        const uint32_t s01 = ld_u16(blk + 192 + 8 * t + 2 * gp);      // group gp: lo16, hi16
        const uint32_t s23 = ld_u16(blk + 192 + 8 * t + 2 * gp + 4);  // group gp + 2
        const float d = h2f(ld_u16(blk + 208));
        const int sh = 2 * gp;
        // Bits sh, sh+1 of each qh byte are group gp's high bits, bits sh+4,
        // sh+5 group gp+2's; u = qh >> sh puts them at 0-1 and 4-5.
        uint32_t u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = qh[i] >> sh;
        float r = 0.0f;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint32_t q[2][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo4 = (g == 0 ? ql[i] : (ql[i] >> 4)) & 0x0F0F0F0Fu;
                const uint32_t hi2 = (g == 0 ? (u[i] << 4) : u[i]) & 0x30303030u;
                q[i >> 2][i & 3] = lo4 | hi2;
            }
            int Al = 0, Bl = 0, Cl = 0, Ah = 0, Bh = 0, Ch = 0;
            dot16(q[0], x, g, 0, Al, Bl, Cl);
            dot16(q[1], x, g, 4, Ah, Bh, Ch);
            const uint32_t sw = g == 0 ? s01 : s23;
            const int scl = (int)(int8_t)(sw & 0xFFu), sch = (int)(int8_t)(sw >> 8);
            const float T = limbs3_to_f(scl * Al + sch * Ah, scl * Bl + sch * Bh, scl * Cl + sch * Ch);
            const float4 mt = x.meta[g];
            const float off = 32.0f * fmaf((float)scl, mt.y, (float)sch * mt.z);
            r += fmaf(mt.x, T, -off);
        }
        return d * r;
    }
};

// Q8_0: lane l -> blocks 2l and 2l+1 of the stage (x-blocks 2l, 2l+1).
// w = d * q, q signed.
template <> struct Lane<T_Q8_0> {
    int l;
    __device__ __forceinline__ explicit Lane(int lane) : l(lane) {}
    __device__ __forceinline__ bool valid(int nblk) const { return 2 * l < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        float r = 0.0f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (2 * l + j >= nblk) break;
            const uint8_t* blk = seg + 68 * l + 34 * j;
            uint32_t q[8];
            lds_words_a2<8>(blk + 2, q);
            const uint32_t qa[4] = {q[0], q[1], q[2], q[3]}, qb[4] = {q[4], q[5], q[6], q[7]};
            int A = 0, B = 0, C = 0;
            dot16(qa, x, j, 0, A, B, C);
            dot16(qb, x, j, 4, A, B, C);
            r = fmaf(h2f(ld_u16(blk)) * x.meta[j].x, limbs_to_f(A, B, C), r);
        }
        return r;
    }
};

// Q4_0: lane l -> blocks 2l and 2l+1 (x-blocks 2l, 2l+1).  Element e < 16 is
// the low nibble of qs[e], element e + 16 the high nibble.  w = d * (q - 8).
template <> struct Lane<T_Q4_0> {
    int l;
    __device__ __forceinline__ explicit Lane(int lane) : l(lane) {}
    __device__ __forceinline__ bool valid(int nblk) const { return 2 * l < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        float r = 0.0f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (2 * l + j >= nblk) break;
            const uint8_t* blk = seg + 36 * l + 18 * j;
            uint32_t q[4];
            lds_words_a2<4>(blk + 2, q);
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo[i] = q[i] & 0x0F0F0F0Fu;
                hi[i] = (q[i] >> 4) & 0x0F0F0F0Fu;
            }
            int A = 0, B = 0, C = 0;
            dot16(lo, x, j, 0, A, B, C);
            dot16(hi, x, j, 4, A, B, C);
            const float4 mt = x.meta[j];
            r = fmaf(h2f(ld_u16(blk)), fmaf(mt.x, limbs_to_f(A, B, C), -8.0f * mt.w), r);
        }
        return r;
    }
};

// Q5_0: lane l -> blocks 2l and 2l+1 (x-blocks 2l, 2l+1).  Element e < 16 is
// the low nibble of qs[e], element e + 16 the high nibble; bit e of qh is
// element e's fifth bit.  w = d * (q - 16).
template <> struct Lane<T_Q5_0> {
    int l;
    __device__ __forceinline__ explicit Lane(int lane) : l(lane) {}
    __device__ __forceinline__ bool valid(int nblk) const { return 2 * l < nblk; }
    __device__ __forceinline__ void xblocks(int lane, int& j0, int& j1) const { j0 = 2 * lane; j1 = 2 * lane + 1; }
    // Four bits t (bit i = fifth bit of byte i) -> 0x10 in each byte whose bit is set.
    __device__ static __forceinline__ uint32_t spread(uint32_t t) { return (t * 0x02040810u) & 0x10101010u; }
    __device__ __forceinline__ float dot(const uint8_t* seg, const XL& x, int nblk) const {
        float r = 0.0f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (2 * l + j >= nblk) break;
            const uint8_t* blk = seg + 44 * l + 22 * j;
            uint32_t hq[5];
            lds_words_a2<5>(blk + 2, hq);   // qh, then qs[0..15]
            const uint32_t qh = hq[0];
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo[i] = (hq[1 + i] & 0x0F0F0F0Fu) | spread((qh >> (4 * i)) & 15u);
                hi[i] = ((hq[1 + i] >> 4) & 0x0F0F0F0Fu) | spread((qh >> (16 + 4 * i)) & 15u);
            }
            int A = 0, B = 0, C = 0;
            dot16(lo, x, j, 0, A, B, C);
            dot16(hi, x, j, 4, A, B, C);
            const float4 mt = x.meta[j];
            r = fmaf(h2f(ld_u16(blk)), fmaf(mt.x, limbs_to_f(A, B, C), -16.0f * mt.w), r);
        }
        return r;
    }
};

// One lane's share of y for one row segment: the lean two-stream decoder for
// Q4_K, the generic lane decoder otherwise.
template <int T>
__device__ __forceinline__ float row_dot(const Lane<T>& L, const Q4KFast& F, const uint8_t* seg, const XL& x,
                                         int nblk, float s0, float s1) {
    if constexpr (T == T_Q4_K) {
        (void)L;
        return F.one(seg, x, s0, s1);
    } else {
        (void)F; (void)s0; (void)s1;
        return L.dot(seg, x, nblk);
    }
}

}  // namespace gv
}  // namespace qk
