// qk_gemv.cu -- fused dequant-GEMV: y[m, n] = sum_k w[n, k] x[m, k].
//
// The packed weights are dequantized inside the dot product ("Local LLM
// inference", "The mmap backend"), and every decoded weight is reused across
// the activation rows a CTA holds (the same page: decode each weight once per
// input batch, reuse it across the batch rows).
//
// Arithmetic.  A prep kernel writes each 32-element block of x as three
// signed 8-bit limbs a, b, c and one fp32 scale s, x ~= s * (65536a + 256b + c)
// (24-bit fixed point, error <= s/2 = max|x| * 2^-24 per element), plus the
// fp32 sums of x over each half and the whole block.  The GEMV then forms
// sum q*x exactly in integers with dp4a (4 code bytes times 4 limb bytes per
// instruction), applies the block's fp16 and sub-block scales once per 16 or
// 32 weights in fp32, and subtracts the min / code-offset terms with the
// sums of x:  Q4_K  (d*sc)*s*T - (dmin*m)*sum(x);  Q6_K  d*sc*(s*T - 32 sum x);
// Q8_0  d*s*T;  Q5_0  d*(s*T - 16 sum x), T = sum q*(65536a + 256b + c).
//
// Data flow.  A CTA owns a tile of 16 output rows (4 consumer warps x 4
// rows) and walks K in stages of 2048 weights.  A producer warp streams each
// stage's 16 row segments from HBM into a shared-memory ring with bulk async
// copies (cp.async.bulk; completion counted on a "full" mbarrier, release on
// an "empty" mbarrier that the consumer warps arrive on).  Row segments need
// not be 16-byte aligned (Q6_K rows of 11008 weights are 9030 bytes apart):
// each copy starts at the aligned-down address, the consumer parses from the
// remainder, and the final bytes of the matrix past its last full 16 bytes
// are fetched by the consumer lanes.  Lane l of a consumer warp owns the
// 64 weights that meet x-blocks 2l and 2l+1 of the stage (Q6_K: a permuted
// pair) for all 4 rows of its warp, so its x limbs stay in registers.
// For skinny problems K is split over gridDim.z; the last CTA of a tile to
// finish adds the partials in split order (deterministic).
#include <algorithm>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_ptx.cuh"

namespace qk {
namespace gv {

constexpr int kCW = 8;                 // consumer warps per CTA
constexpr int kRW = 2;                 // rows per consumer warp
constexpr int kRows = kCW * kRW;       // rows per CTA tile
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kKR = 2048;              // weights per row per stage
constexpr int kXB = kKR / 32;          // x-blocks per stage
constexpr int kXBytes = 112;           // prepped bytes per x-block: a[32] b[32] c[32] + float4
constexpr float kXMax = 8323072.0f;    // 127 * 65536: largest |X| of a 3-limb value

// Stage layout: 16 row slots of packed weights, then the stage's prepped
// activations (kXB x-blocks) for each of the MT activation rows.
template <int T, int MT> struct Cfg {
    static constexpr int BB = Fmt<T>::BB, BE = Fmt<T>::BE;
    static constexpr int KB = kKR / BE;                      // blocks per row per stage
    static constexpr int SEG = KB * BB;                      // bytes per row per stage
    static constexpr int SLOT = (SEG + 32 + 15) / 16 * 16;   // with 16-byte alignment slack
    static constexpr int XOFF = kRows * SLOT;
    static constexpr int XBYTES = kXB * kXBytes;             // per activation row
    static constexpr int STAGE = XOFF + MT * XBYTES;
    static constexpr int BUDGET = 110 * 1024;                // two CTAs per SM
    static constexpr int NST = BUDGET / STAGE > 4 ? 4 : (BUDGET / STAGE < 2 ? 2 : BUDGET / STAGE);
    static constexpr int SMEM = NST * STAGE + 2 * NST * 8;
};

struct Args {
    const uint8_t* W;
    int64_t rows, cols, M;
    int64_t row_bytes;
    int64_t total16;        // bytes of W rounded down to 16
    const uint8_t* xp;      // prepped activations [M][cols/32][112]
    float* y;               // [M, rows]
    float* part;            // split partials [splits][M][rows] (splits > 1)
    unsigned* counters;     // one per (row tile, m tile) (splits > 1)
    int splits;
    int stages_per_split;
    unsigned* status;
};

// ---------------------------------------------------------------------------
// dp4a: four signed byte products added to c.
// (The accumulator is an in-place operand, so no register copy is needed.)
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    asm("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
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
// fed here is a valid signed byte (Q4_K 0..15, Q6_K 0..63, Q5_0 0..31, Q8_0
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
            // Codes 0..15 are also valid signed bytes: signed x signed dp4a.
            const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
            A0 = dp4a_ss(lo, x.a[0][i], A0);
            B0 = dp4a_ss(lo, x.b[0][i], B0);
            C0 = dp4a_ss(lo, x.c[0][i], C0);
            A1 = dp4a_ss(hi, x.a[1][i], A1);
            B1 = dp4a_ss(hi, x.b[1][i], B1);
            C1 = dp4a_ss(hi, x.c[1][i], C1);
        }
        const uint32_t f = fields(h);
        const float sc0 = byte_to_f(f, 0x7440), sc1 = byte_to_f(f, 0x7441);
        const float m0 = byte_to_f(f, 0x7442), m1 = byte_to_f(f, 0x7443);
        const float t0 = limbs_to_f(A0, B0, C0) * s0, t1 = limbs_to_f(A1, B1, C1) * s1;
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
        float r = 0.0f;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint32_t q[2][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo4 = (g == 0 ? ql[i] : (ql[i] >> 4)) & 0x0F0F0F0Fu;
                const uint32_t hi2 = ((qh[i] >> (sh + 4 * g)) & 0x03030303u) << 4;
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

// ---------------------------------------------------------------------------
// Activation prep: one warp per (m, 32-block).  Writes the three limbs of
// every element, the scale and the block's sums; also zeroes the split-K
// tile counters of this call.
__global__ void __launch_bounds__(256) xprep_kernel(const float* __restrict__ x, int64_t M, int64_t cols,
                                                    uint8_t* __restrict__ xp, unsigned* counters, int ncounters) {
    pdl_launch_dependents();
    pdl_wait_prior();
    const int lane = threadIdx.x & 31;
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0u;
    const int64_t nxb = cols / 32;
    if (gw >= M * nxb) return;
    const int64_t m = gw / nxb, jb = gw % nxb;
    const float v = x[m * cols + jb * 32 + lane];
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax / kXMax;
    const float inv = amax > 0.0f ? kXMax / amax : 0.0f;
    int X = __float2int_rn(v * inv);
    X = max(-(int)kXMax, min((int)kXMax, X));
    // Balanced base-256 digits: X = 65536a + 256b + c, each in [-128, 127].
    const int c = (int)(int8_t)(X & 255);
    const int X1 = (X - c) >> 8;
    const int b = (int)(int8_t)(X1 & 255);
    const int a = (X1 - b) >> 8;
    uint8_t* o = xp + gw * kXBytes;
    o[lane] = (uint8_t)a;
    o[32 + lane] = (uint8_t)b;
    o[64 + lane] = (uint8_t)c;
    float lo = lane < 16 ? v : 0.0f, hi = lane < 16 ? 0.0f : v;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo += __shfl_xor_sync(0xffffffffu, lo, off);
        hi += __shfl_xor_sync(0xffffffffu, hi, off);
    }
    if (lane == 0)
        *reinterpret_cast<float4*>(o + 96) = make_float4(s, lo, hi, lo + hi);
}

template <int T, int MT>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const Args p) {
    using C = Cfg<T, MT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE);
    uint64_t* empty = full + C::NST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kRows;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    const int64_t nb = p.cols / C::BE;
    const int64_t nst_all = (nb + C::KB - 1) / C::KB;
    const int64_t gs0 = (int64_t)blockIdx.z * p.stages_per_split;
    const int nloc = (int)max((int64_t)0, min((int64_t)p.stages_per_split, nst_all - gs0));

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const int64_t nxb = p.cols / 32;
    if (warp == kCW) {
        // Producer warp: lane r < 16 copies row r's segment of each stage,
        // lanes 16.. copy the stage's prepped activations.  Weights do not
        // depend on the previous kernel, so the first stages' weights go out
        // before the grid-dependency wait; the activations after it.
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        const bool wrow = lane < kRows && row0 + lane < p.rows;
        const int64_t rstart = (row0 + lane) * p.row_bytes + gs0 * C::SEG;  // this lane's row, stage 0
        const bool xlane = lane >= kRows && lane < kRows + MT && m0 + (lane - kRows) < p.M;
        const uint8_t* xsrc = p.xp + ((m0 + (lane - kRows)) * nxb + gs0 * kXB) * kXBytes;
        auto stage_len = [&](int i) -> int64_t {   // weight bytes of every row at local stage i
            return min((int64_t)C::KB, nb - (gs0 + i) * C::KB) * C::BB;
        };
        auto xlen = [&](int i) -> uint32_t {
            return (uint32_t)(min((int64_t)kXB, nxb - (gs0 + i) * kXB) * kXBytes);
        };
        auto wcopy = [&](int i, int slot, bool issue, uint32_t& bytes) {
            const int64_t st = rstart + (int64_t)i * C::SEG;
            const int64_t a = st & ~(int64_t)15;
            const int64_t e = min((st + stage_len(i) + 15) & ~(int64_t)15, p.total16);
            const uint32_t n = (wrow && e > a) ? (uint32_t)(e - a) : 0u;
            bytes = n;
            if (issue && n) bulk_g2s(smem + slot * C::STAGE + lane * C::SLOT, p.W + a, n, &full[slot], pol_w);
        };
        const int pre = min(nloc, C::NST);
        for (int i = 0; i < pre; ++i) {
            uint32_t n;
            wcopy(i, i, false, n);
            const uint32_t tot = __reduce_add_sync(0xffffffffu, n + (xlane ? xlen(i) : 0u));
            if (lane == 0) mbar_arrive_expect_tx(&full[i], tot);
            __syncwarp();
            wcopy(i, i, true, n);
        }
        pdl_wait_prior();
        if (xlane)
            for (int i = 0; i < pre; ++i)
                bulk_g2s(smem + i * C::STAGE + C::XOFF + (lane - kRows) * C::XBYTES,
                         xsrc + (int64_t)i * kXB * kXBytes, xlen(i), &full[i], pol_x);
        for (int i = pre; i < nloc; ++i) {
            const int slot = i % C::NST;
            uint32_t n;
            wcopy(i, slot, false, n);
            const uint32_t tot = __reduce_add_sync(0xffffffffu, n + (xlane ? xlen(i) : 0u));
            int go = 1;
            if (lane == 0) {
                go = mbar_wait_bounded(&empty[slot], (uint32_t)((i / C::NST - 1) & 1), p.status) ? 1 : 0;
                if (go) mbar_arrive_expect_tx(&full[slot], tot);
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) break;
            wcopy(i, slot, true, n);
            if (xlane)
                bulk_g2s(smem + slot * C::STAGE + C::XOFF + (lane - kRows) * C::XBYTES,
                         xsrc + (int64_t)i * kXB * kXBytes, xlen(i), &full[slot], pol_x);
        }
        return;
    }

    const Lane<T> L(lane);
    int j0, j1;
    L.xblocks(lane, j0, j1);
    float acc[kRW][MT];
#pragma unroll
    for (int r = 0; r < kRW; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;
    // Per-row constants: offset of the segment inside its slot (every stage's
    // segment starts at row_start + k*SEG and SEG is a multiple of 16), and
    // whether the row's last bytes lie past the last full 16 bytes of W.
    int roff[kRW];
    bool rtail[kRW], rvalid[kRW];
#pragma unroll
    for (int r = 0; r < kRW; ++r) {
        const int64_t row = row0 + warp * kRW + r;
        rvalid[r] = row < p.rows;
        const int64_t rs = row * p.row_bytes;
        roff[r] = (int)(rs & 15);
        rtail[r] = rvalid[r] && rs + p.row_bytes > p.total16;
    }
    bool ok = true;

    for (int i = 0; i < nloc; ++i) {
        const int slot = i % C::NST;
        const int64_t gs = gs0 + i;
        if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / C::NST) & 1), p.status)) {
            for (int k = i + 1; k < min(nloc, i + C::NST); ++k)
                mbar_wait_bounded(&full[k % C::NST], (uint32_t)((k / C::NST) & 1), p.status);
            ok = false;
            break;
        }
        uint8_t* stage = smem + slot * C::STAGE;
        const int nblk = (int)min((int64_t)C::KB, nb - gs * C::KB);
        if (gs == nst_all - 1) {
            // Bytes past the last full 16 bytes of W: fetched by the owning warp.
            bool wrote = false;
#pragma unroll
            for (int r = 0; r < kRW; ++r) {
                if (!rtail[r]) continue;
                const int64_t row = row0 + warp * kRW + r;
                const int64_t st = row * p.row_bytes + gs * C::SEG;
                const int64_t en = st + (int64_t)nblk * C::BB;
                uint8_t* dst = stage + (warp * kRW + r) * C::SLOT - (st & ~(int64_t)15);
                for (int64_t b = max(st, p.total16) + lane; b < en; b += 32) dst[b] = p.W[b];
                wrote = true;
            }
            if (wrote) fence_proxy_async_smem();
            __syncwarp();
        }
        if (L.valid(nblk)) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m0 + m >= p.M) break;
                XL x;
                load_x(stage + C::XOFF + m * C::XBYTES, j0, j1, x);
#pragma unroll
                for (int r = 0; r < kRW; ++r) {
                    if (!rvalid[r]) break;
                    const uint8_t* seg = stage + (warp * kRW + r) * C::SLOT + roff[r];
                    acc[r][m] += L.dot(seg, x, nblk);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

#pragma unroll
    for (int r = 0; r < kRW; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r][m] = v;
        }

    if (p.splits == 1) {
        if (lane == 0 && ok)
#pragma unroll
            for (int r = 0; r < kRW; ++r) {
                const int64_t row = row0 + warp * kRW + r;
                if (row >= p.rows) break;
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m0 + m < p.M) p.y[(m0 + m) * p.rows + row] = acc[r][m];
            }
        return;
    }

    // Split K: publish this split's partials; the last CTA of the tile sums
    // all splits in order and writes y.  Every consumer warp takes part in
    // the two barriers, even after a timed-out wait (its results are then
    // invalid and the status word says so).
    if (lane == 0 && ok) {
#pragma unroll
        for (int r = 0; r < kRW; ++r) {
            const int64_t row = row0 + warp * kRW + r;
            if (row >= p.rows) break;
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m0 + m < p.M) p.part[((int64_t)blockIdx.z * p.M + m0 + m) * p.rows + row] = acc[r][m];
        }
        __threadfence();
    }
    __shared__ unsigned s_last;
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    if (threadIdx.x == 0) {
        const unsigned tile = blockIdx.y * gridDim.x + blockIdx.x;
        const unsigned old = atomicAdd(&p.counters[tile], 1u);
        s_last = (old == (unsigned)p.splits - 1) ? 1u : 0u;
        if (s_last) p.counters[tile] = 0u;
        __threadfence();
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    if (!s_last) return;
    for (int idx = threadIdx.x; idx < kRows * MT; idx += kCW * 32) {
        const int64_t row = row0 + idx % kRows, m = m0 + idx / kRows;
        if (row >= p.rows || m >= p.M) continue;
        float v = 0.0f;
        for (int z = 0; z < p.splits; ++z) v += __ldcg(&p.part[((int64_t)z * p.M + m) * p.rows + row]);
        p.y[m * p.rows + row] = v;
    }
}

// ---------------------------------------------------------------------------
// Decode kernel for one activation row (M == 1): K-sliced warps.
//
// A CTA owns a contiguous range of output rows (every CTA gets the same
// number of rows, +-1).  K is cut into slices of 2048 weights; warp w works
// on slice group g = w / wps (slices g, g + ngroups, ...) and on the CTA's
// rows r with r % wps == w % wps.  Each lane loads the prepped activations of
// its 64 weights of a slice once and keeps them in registers while the warp
// walks its rows, so the only other traffic is the packed weights.  Each
// warp streams its row segments (the aligned-down 16-byte window of the
// segment) with 16-byte cp.async copies into its own 4-deep shared-memory
// ring and parses them there.  A row's partials from the slice groups meet
// in shared memory and are added in group order after a CTA barrier.

constexpr int kW4 = 8;       // warps per CTA
constexpr int kRCH = 256;    // rows per CTA chunk (partials buffer)

template <int T> struct Cfg4 {
    static constexpr int BB = Fmt<T>::BB, BE = Fmt<T>::BE;
    static constexpr int KB = kKR / BE;
    static constexpr int SEG = KB * BB;
    static constexpr int SLOT = (SEG + 32 + 15) / 16 * 16;   // one row segment
    // Ring depth in row pairs: as deep as fits two CTAs per SM.
    static constexpr int NSW = T == T_Q8_0 ? 2 : (T == T_Q6_K ? 3 : 4);
    static constexpr int WARP = NSW * 2 * SLOT;              // ring of row pairs
    static constexpr int OFF_RED = kW4 * WARP;
    static constexpr int SMEM = OFF_RED + kRCH * kW4 * 4;
};

struct Args4 {
    const uint8_t* W;
    int64_t rows, cols, row_bytes, total16;
    const uint8_t* xp;   // prepped activations [cols/32][112]
    float* y;
    int64_t rows_q;      // rows / gridDim.x
    int rows_r;          // rows % gridDim.x: the first rows_r CTAs take one row more
    int nsl;             // K slices
    int wps_log2;        // warps per slice group = 1 << wps_log2
    int ngroups;         // slice groups
    int nmine0;          // slices of slice group 0 (group g has nmine0 or nmine0 - 1)
};

// The lane's two x-blocks straight from global memory (prepped activations).
__device__ __forceinline__ void load_x_global(const uint8_t* xp, int64_t xb0, int64_t xb1, int64_t nxb, XL& x) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t xb = j == 0 ? xb0 : xb1;
        const uint4* q = reinterpret_cast<const uint4*>(xp + xb * kXBytes);
        uint4 v[7];
#pragma unroll
        for (int k = 0; k < 7; ++k) v[k] = xb < nxb ? __ldg(q + k) : make_uint4(0, 0, 0, 0);
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

template <int T>
__global__ void __launch_bounds__(kW4 * 32, 2) gemv4_kernel(const Args4 p) {
    using C = Cfg4<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wps = 1 << p.wps_log2, g = warp >> p.wps_log2, sub = warp & (wps - 1);
    const bool active = g < p.ngroups;
    uint8_t* ring = smem + warp * C::WARP;
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
    const int bx = (int)blockIdx.x;
    const int64_t r_begin = bx * p.rows_q + min(bx, p.rows_r);
    const int64_t r_end = r_begin + p.rows_q + (bx < p.rows_r ? 1 : 0);
    const int64_t nb = p.cols / C::BE, nxb = p.cols / 32;
    // My slices: g, g + ngroups, ... (nsl = nmine0 * ngroups - extra).
    const int nmine = active ? (g * 1 < p.nsl - (p.nmine0 - 1) * p.ngroups ? p.nmine0 : p.nmine0 - 1) : 0;
    const Lane<T> L(lane);
    const Q4KFast F(lane);
    int j0, j1;
    L.xblocks(lane, j0, j1);
    pdl_launch_dependents();

    constexpr int NCH = (C::SEG + 16 + 15) / 16;          // 16-byte chunks per row window
    constexpr int NIT = (NCH + 31) / 32;                  // copy iterations per lane
    for (int64_t cb = r_begin; cb < r_end; cb += kRCH) {
        const int64_t ce = min(r_end, cb + kRCH);
        const int nr = active ? (int)((ce - cb - sub + wps - 1) >> p.wps_log2) : 0;   // my rows in the chunk
        const int np = (nr + 1) / 2;                                          // row pairs
        const int nst = np * nmine;                                          // stages: slice-major
        // 32-bit byte offsets relative to an aligned base at my first row.
        const int64_t row0_off = (cb + sub) * p.row_bytes;
        const uint8_t* base = p.W + (row0_off & ~(int64_t)15);
        const uint32_t mis0 = (uint32_t)(row0_off & 15);
        const uint32_t rstep = (uint32_t)(wps * p.row_bytes);                // next row of mine
        const int64_t lim64 = p.total16 - (row0_off & ~(int64_t)15);
        const uint32_t lim = lim64 > 0xFFFFFFF0ll ? 0xFFFFFFF0u : (uint32_t)lim64;   // copy limit
        // Issue pointer (slice ik, pair iq) advances one stage per call.
        int ik = 0, iq = 0;
        auto issue = [&](int st) {
            const int sl = g + ik * p.ngroups;
            const uint32_t len = (uint32_t)(min((int64_t)C::KB, nb - (int64_t)sl * C::KB) * C::BB);
            const uint32_t rel0 = mis0 + 2u * iq * rstep + (uint32_t)sl * C::SEG;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (2 * iq + h < nr) {
                    const uint32_t rel = rel0 + h * rstep;
                    const uint32_t a = rel & ~15u;
                    const uint32_t e = min((rel + len + 15u) & ~15u, lim);
                    const int nch = e > a ? (int)((e - a) >> 4) : 0;
                    uint8_t* dst = ring + ((st % C::NSW) * 2 + h) * C::SLOT;
                    const uint8_t* src = base + a;
#pragma unroll
                    for (int it = 0; it < NIT; ++it) {
                        const int ch = lane + 32 * it;
                        if (ch < nch) cp_async16(dst + 16 * ch, src + 16 * ch);
                    }
                }
            }
            if (++iq == np) { iq = 0; ++ik; }
        };
#pragma unroll
        for (int st = 0; st < C::NSW - 1; ++st) {
            if (st < nst) issue(st);
            cp_async_commit();
        }
        if (cb == r_begin) pdl_wait_prior();   // the prepped activations come from the previous kernel
        XL x;
        float s0 = 0.0f, s1 = 0.0f;
        int k = 0, q = 0, nblk = 0, sl = g;
        uint32_t rel_pair = 0;   // offset of this pair's first row, slice sl
        // The first slice's activations load while the first stages are in flight.
        if (nst > 0) load_x_global(p.xp, (int64_t)g * kXB + j0, (int64_t)g * kXB + j1, nxb, x);
        for (int st = 0; st < nst; ++st) {
            if (st + C::NSW - 1 < nst) issue(st + C::NSW - 1);
            cp_async_commit();
            cp_async_wait<C::NSW - 1>();
            __syncwarp();
            if (q == 0) {   // a new slice: its activations and block count
                sl = g + k * p.ngroups;
                if (k > 0) load_x_global(p.xp, (int64_t)sl * kXB + j0, (int64_t)sl * kXB + j1, nxb, x);
                s0 = x.meta[0].x;
                s1 = x.meta[1].x;
                nblk = (int)min((int64_t)C::KB, nb - (int64_t)sl * C::KB);
                rel_pair = mis0 + (uint32_t)sl * C::SEG;
            }
            const bool lv = L.valid(nblk);
            const uint32_t seglen = (uint32_t)nblk * C::BB;
            float v[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                v[h] = 0.0f;
                if (2 * q + h < nr) {
                    const uint32_t rel = rel_pair + h * rstep;
                    uint8_t* slot = ring + ((st % C::NSW) * 2 + h) * C::SLOT;
                    if (rel + seglen > lim) {
                        // Bytes past the last full 16 bytes of W (the matrix's final row).
                        uint8_t* sbase = slot - (rel & ~15u);
                        for (uint32_t bb = max(rel, lim) + lane; bb < rel + seglen; bb += 32) sbase[bb] = base[bb];
                        __syncwarp();
                    }
                    if (lv) v[h] = row_dot<T>(L, F, slot + (rel & 15u), x, nblk, s0, s1);
                }
            }
            // Two-row butterfly: lanes 0-15 end with row 2q, lanes 16-31 with 2q+1.
            const bool upper = lane & 16;
            float keep = upper ? v[1] : v[0];
            keep += __shfl_xor_sync(0xffffffffu, upper ? v[0] : v[1], 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
            // Every lane of a half holds its row's sum; lane 0 / 16 stores it.
            const int i = 2 * q + (upper ? 1 : 0);
            float* r = &red[(sub + min(i, nr - 1) * wps) * kW4 + g];
            const float prev = (k == 0) ? 0.0f : *r;
            __syncwarp();
            if ((lane & 15) == 0 && i < nr) *r = prev + keep;
            __syncwarp();
            rel_pair += 2u * rstep;
            if (++q == np) { q = 0; ++k; }
        }
        cp_async_wait<0>();
        __syncthreads();
        for (int t = threadIdx.x; t < (int)(ce - cb); t += kW4 * 32) {
            float vv = 0.0f;
            for (int gg = 0; gg < p.ngroups; ++gg) vv += red[t * kW4 + gg];
            p.y[cb + t] = vv;
        }
        __syncthreads();
    }
}

}  // namespace gv
}  // namespace qk

namespace qk {

namespace {
int mt_for(int64_t M) { return M >= 4 ? 4 : (M >= 2 ? 2 : 1); }

int64_t nst_for(int type, int64_t cols) {
    switch (type) {
    case T_Q4_K: case T_Q6_K: return (cols / 256 + 7) / 8;
    case T_Q8_0: case T_Q5_0: return (cols / 32 + 63) / 64;
    }
    return 0;
}

int64_t align16(int64_t v) { return (v + 15) & ~(int64_t)15; }
}  // namespace

GemvPlan plan_gemv(int type, int64_t rows, int64_t cols, int64_t M, int sm_count) {
    GemvPlan pl;
    if (M == 1) {   // K-sliced decode kernel: prepped activations only
        pl.mt = 1;
        pl.splits = 1;
        pl.ws_bytes = align16((cols / 32) * gv::kXBytes);
        return pl;
    }
    pl.mt = mt_for(M);
    const int64_t tiles = ((rows + gv::kRows - 1) / gv::kRows) * ((M + pl.mt - 1) / pl.mt);
    const int64_t nst = nst_for(type, cols);
    const int64_t sms = std::max(sm_count, 1);
    int64_t splits = 1;
    if (tiles > 0 && tiles < sms && nst > 1) {
        splits = std::min<int64_t>({(2 * sms + tiles - 1) / tiles, nst, 32});
        const int64_t per = (nst + splits - 1) / splits;
        splits = (nst + per - 1) / per;   // every split owns at least one stage
    }
    pl.splits = (int)splits;
    const int64_t xp = M * (cols / 32) * gv::kXBytes;
    const int64_t part = splits > 1 ? align16(splits * M * rows * (int64_t)sizeof(float)) : 0;
    const int64_t cnt = splits > 1 ? align16(tiles * (int64_t)sizeof(unsigned)) : 0;
    pl.ws_bytes = align16(xp) + part + cnt;
    return pl;
}

template <int T, int MT>
static cudaError_t launch_t(const GemvPlan& pl, const gv::Args& a, cudaStream_t s) {
    using C = gv::Cfg<T, MT>;
    auto kern = gv::gemv_kernel<T, MT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.rows + gv::kRows - 1) / gv::kRows), (unsigned)((a.M + MT - 1) / MT),
                       (unsigned)pl.splits);
    cfg.blockDim = dim3(gv::kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int T>
static cudaError_t launch4(const gv::Args4& b, int64_t grid, cudaStream_t s) {
    using C = gv::Cfg4<T>;
    auto kern = gv::gemv4_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(gv::kW4 * 32);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, b);
}

template <int T>
static cudaError_t launch_mt(const GemvPlan& pl, const gv::Args& a, cudaStream_t s) {
    switch (pl.mt) {
    case 1: return launch_t<T, 1>(pl, a, s);
    case 2: return launch_t<T, 2>(pl, a, s);
    default: return launch_t<T, 4>(pl, a, s);
    }
}

cudaError_t launch_gemv(int type, const GemvPlan& pl, const uint8_t* W, int64_t rows, int64_t cols, const float* x,
                        int64_t M, float* y, float* ws, unsigned* status, cudaStream_t s) {
    gv::Args a = {};
    a.W = W;
    a.rows = rows;
    a.cols = cols;
    a.M = M;
    switch (type) {
    case T_Q4_K: a.row_bytes = cols / 256 * 144; break;
    case T_Q6_K: a.row_bytes = cols / 256 * 210; break;
    case T_Q8_0: a.row_bytes = cols / 32 * 34; break;
    case T_Q5_0: a.row_bytes = cols / 32 * 22; break;
    default: return cudaErrorInvalidValue;
    }
    a.total16 = (rows * a.row_bytes) & ~(int64_t)15;
    const int64_t nst = nst_for(type, cols);
    a.splits = pl.splits;
    a.stages_per_split = (int)((nst + pl.splits - 1) / pl.splits);
    a.y = y;
    a.status = status;
    uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
    const int64_t xp_bytes = align16(M * (cols / 32) * gv::kXBytes);
    a.xp = wsb;
    const int64_t tiles = ((rows + gv::kRows - 1) / gv::kRows) * ((M + pl.mt - 1) / pl.mt);
    int ncounters = 0;
    if (pl.splits > 1) {
        a.part = reinterpret_cast<float*>(wsb + xp_bytes);
        a.counters = reinterpret_cast<unsigned*>(wsb + xp_bytes + align16(pl.splits * M * rows * 4));
        ncounters = (int)tiles;
    }

    // 1) activation prep (also zeroes the split-K counters)
    {
        const int64_t warps = M * (cols / 32);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, (warps * 32 + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, gv::xprep_kernel, x, M, cols, wsb, a.counters, ncounters);
        if (e != cudaSuccess) return e;
    }
    // 2) the fused GEMV
    if (M == 1) {
        gv::Args4 b = {};
        b.W = W;
        b.rows = rows;
        b.cols = cols;
        b.row_bytes = a.row_bytes;
        b.total16 = a.total16;
        b.xp = wsb;
        b.y = y;
        b.nsl = (int)nst;
        int wps = 1;
        if (nst <= gv::kW4) {
            while (2 * wps * nst <= gv::kW4) wps *= 2;
            b.ngroups = (int)nst;
        } else {
            b.ngroups = gv::kW4;
        }
        b.wps_log2 = 0;
        while ((1 << b.wps_log2) < wps) ++b.wps_log2;
        b.nmine0 = (int)((nst + b.ngroups - 1) / b.ngroups);
        int sms = 0, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        // Two CTAs per SM, each with a contiguous range of rows.
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(2 * (int64_t)std::max(sms, 1), rows / 4));
        b.rows_q = rows / grid;
        b.rows_r = (int)(rows % grid);
        switch (type) {
        case T_Q4_K: return launch4<T_Q4_K>(b, grid, s);
        case T_Q6_K: return launch4<T_Q6_K>(b, grid, s);
        case T_Q8_0: return launch4<T_Q8_0>(b, grid, s);
        case T_Q5_0: return launch4<T_Q5_0>(b, grid, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (type) {
    case T_Q4_K: return launch_mt<T_Q4_K>(pl, a, s);
    case T_Q6_K: return launch_mt<T_Q6_K>(pl, a, s);
    case T_Q8_0: return launch_mt<T_Q8_0>(pl, a, s);
    case T_Q5_0: return launch_mt<T_Q5_0>(pl, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
