// qk_gemm.cu -- tensor-core dequant-GEMM for prefill: Y[m, n] = sum_k w[n, k] X[m, k].
//
// Prefill turns the per-token GEMV into a real dense contraction ("12 --
// llama.cpp / GGUF": prompt processing is big GEMMs of high arithmetic
// intensity; decode is bandwidth-bound).  A CTA owns 128 weight rows x 512
// tokens and walks K in blocks of 64:
//   * 16 dequant warps unpack the packed blocks of the 128 weight rows, round
//     the fp32 weights to bf16 and store them straight into shared memory in
//     the tensor core's K-major 128-byte-swizzled layout (operand A);
//   * one thread loads the two 256 x 64 bf16 activation tiles with TMA
//     (operand B);
//   * one thread issues tcgen05.mma (M = 128, N = 256, K = 16 per instruction)
//     into two fp32 accumulators in tensor memory (tokens 0-255 and 256-511:
//     all 512 columns) and releases each stage with tcgen05.commit;
//   * the dequant warps then read the accumulators back (tcgen05.ld) and
//     write Y.
// Dequantizing a weight tile is the costly part; covering 512 tokens per
// tile halves it per FLOP compared with one 256-column accumulator.
// Every mbarrier wait is bounded; tensor memory is always released.
#include <algorithm>
#include <cstring>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_ptx.cuh"
#include "qk_tc.cuh"

namespace qk {
namespace gv {
// (from qk_gemv.cu; shared-memory word loads at 2-byte alignment)
template <int N>
__device__ __forceinline__ void lds_words_a2(const uint8_t* p, uint32_t (&w)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8;   // 0 or 16
    uint32_t prev = *reinterpret_cast<const uint32_t*>(base);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t next = *reinterpret_cast<const uint32_t*>(base + 4 * (i + 1));
        w[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}
}  // namespace gv
namespace gm {

__device__ __forceinline__ uint4 lds128_g(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

constexpr int kBM = 128;          // weight rows per CTA (MMA M)
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int kA = kBM * kBK * 2; // 16 KB of bf16 weights per stage
constexpr int kDeqWarps = 16;
constexpr int kThreads = (2 + kDeqWarps) * 32;   // TMA warp, MMA warp, dequant warps

// Pipeline shape.  Three rings: NS weight stages (bf16 operand A, written by
// the dequant warps), an activation ring of run-time depth (operand B, one
// 64-wide k-block of every accumulator's tokens per stage, loaded by TMA)
// and NSP packed macro-block stages; NACC accumulators of BNM tokens each.
// The activation ring has its own barriers, so its loads run as far ahead of
// the tensor core as its depth allows instead of waiting for the weight
// stage they pair with.
//   Wide (prefill, M > 64): two 256-token accumulators fill tensor memory and
//   each k-block carries 8 MMAs of 128 x 256 x 16, so two weight stages keep
//   the tensor core fed.
//   Small batches (M <= 64) use gemm_skinny_kernel below instead.
template <int NS_, int NACC_, int BNM_, int NSP_> struct Cfg {
    static constexpr int NS = NS_, NACC = NACC_, BNM = BNM_, NSP = NSP_;
    static constexpr int BN = BNM * NACC;            // tokens per CTA
    static constexpr int TMEM = BN < 32 ? 32 : BN;   // power of two >= 32
    static_assert((TMEM & (TMEM - 1)) == 0, "tensor memory columns");
};
using Wide = Cfg<2, 2, 256, 2>;
constexpr int kSkinnyBN = 64;     // largest M the skinny pipeline takes
constexpr int kMaxXStages = 16;   // activation ring depth limit
constexpr int kSmemMax = 227 * 1024;

// Packed macro-block geometry: weights and bytes per row (one super-block,
// or four / eight 32-weight blocks), and the per-row slot: the aligned-down
// window starts up to 14 bytes early and the funnel-shifted word reads run up
// to 4 bytes past the end.
template <int T> struct PkGeo {
    static constexpr int MB = T == T_Q8_0 ? 128 : 256;
    static constexpr int KPM = MB / kBK;                         // k-blocks per macro-block
    static constexpr int BYTES = MB / Fmt<T>::BE * Fmt<T>::BB;   // 144, 210, 136, 176, 144
    // Row slots are 16-byte multiples (cp.async) and an odd number of 16-byte
    // units, so the 32 rows a warp reads spread over 8 bank groups.
    static constexpr int SLOT0 = (BYTES + 14 + 4 + 15) / 16 * 16;
    static constexpr int SLOT = (SLOT0 / 16) % 2 == 0 ? SLOT0 + 16 : SLOT0;
    static constexpr int STAGE = kBM * SLOT;
};

// Small-batch kernel (M <= 64): 256-weight macro-blocks for every type (four
// 64-wide k-blocks), a CTA-wide packed ring of NSP stages filled by bulk
// copies, NS bf16 weight stages.  20 warps: activation producer, two MMA
// issuers, packed producer, 16 dequant warps (4 row quarters x 4 k-block
// phases).
template <int T> struct SkGeo {
    static constexpr int BYTES = 256 / Fmt<T>::BE * Fmt<T>::BB;          // 144, 210, 272, 176, 144
    // 2D TMA box width, also the row stride of a packed stage: the
    // macro-block itself, or for Q6_K (whose starts are 2-byte aligned) 240
    // bytes from the 16-byte boundary below its start.  An odd number of
    // 16-byte units, so the 32 rows a warp reads spread over 8 bank groups.
    // The word reads of the 32-weight types run up to 4 bytes past a row's
    // box (into the next row, or past the ring into the barriers): read, never
    // used.
    // Q2_K (84 bytes, starts 4-byte aligned) needs 12 + 84 -> 112; Q3_K
    // (110 bytes, 2-byte aligned) 14 + 110 -> 144.
    static constexpr int BOXW = T == T_Q6_K ? 240 : (T == T_Q2_K ? 112 : (T == T_Q3_K ? 144 : BYTES));
    static_assert(BOXW % 16 == 0 && (BOXW / 16) % 2 == 1, "packed TMA box");
    static constexpr int STAGE = kBM * BOXW;
    static constexpr int NSP = 3;
    static constexpr int NS = T == T_Q8_0 ? 4 : 6;
    static constexpr int FIX = 1024 + NS * kA + NSP * STAGE;
    __host__ __device__ static constexpr int smem(int nsb, int xst) {
        return FIX + nsb * xst + (2 * NS + 2 * nsb + 2 * NSP + 1) * 8 + 16;
    }
};
constexpr int kSkMma = 2;                      // MMA warps, one accumulator each
constexpr int kSkThreads = (2 + kSkMma + 16) * 32;   // activation producer, MMA warps, packed producer, 16 dequant
constexpr int kSkTmem = 64 * kSkMma;

// Shared-memory map (from the 1024-byte aligned base): NS weight stages, the
// activation ring (nsb stages of xst bytes), the packed ring, the mbarriers
// and the tensor-memory address slot.  FIX is everything but the activation
// ring and the barriers; 1 KB of slack covers the base alignment.
template <int T, class C> struct Pk : PkGeo<T> {
    static constexpr int OFF_X = C::NS * kA;
    static constexpr int FIX = 1024 + C::NS * kA + C::NSP * PkGeo<T>::STAGE;
    __host__ __device__ static constexpr int smem(int nsb, int xst) {
        return FIX + nsb * xst + (2 * C::NS + 2 * nsb + 1) * 8 + 16;
    }
};

struct Args {
    const uint8_t* W;
    int64_t rows, cols, row_bytes, M, total16;
    float* Y;
    float* part;          // split-K partials [splits][M][rows] (nullptr: write Y)
    unsigned* status;
    int nkb;              // 64-wide k-blocks of K
    int kb_per_split;     // k-blocks per split (a multiple of the macro-block's)
    int nmma;             // MMA N (tokens per accumulator): 256, or M rounded up to 16 when M <= 256
    int nsb;              // activation ring depth
    int xst;              // bytes per activation stage (accumulators x nmma x 128)
};

// (unit, half) of the 16 weights that start `o` weights into a block.
template <int T>
__device__ __forceinline__ void locate(int o, int& u, int& h) {
    if constexpr (T == T_Q4_K || T == T_Q5_K) {   // koff = 64(u>>1) + 32h + 16(u&1)
        u = 2 * (o >> 6) + ((o >> 4) & 1);
        h = (o >> 5) & 1;
    } else if constexpr (T == T_Q2_K || T == T_Q3_K) {   // koff = 32u + 16h
        u = o >> 5;
        h = (o >> 4) & 1;
    } else if constexpr (T == T_Q6_K) {   // koff = 128(u>>2) + 32((u>>1&1) + 2h) + 16(u&1)
        const int t = o >> 7, g = (o >> 5) & 3;
        u = 4 * t + 2 * (g & 1) + ((o >> 4) & 1);
        h = g >> 1;
    } else {                              // 32-weight blocks: koff = 16h
        u = 0;
        h = (o >> 4) & 1;
    }
}

// ---------------------------------------------------------------------------
// Fast bf16 decoders (16 weights of one tile row: quarter qq of a 64-wide
// k-block).  A code byte is placed into an fp32 mantissa by one byte permute
// (exact: 128 + q with the code in bits 16-23 of 0x43000000, or 256 + u/128
// with the byte in bits 8-15 of 0x43800000), then one packed fp32 FMA per two
// weights applies scale and offset, and one convert packs two bf16.

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Four bytes of v (each < 128) -> 128 + byte as fp32, times a, plus c;
// packed as two bf16x2 words.
__device__ __forceinline__ void four_hi(uint32_t v, float2 a, float2 c, uint32_t& o0, uint32_t& o1) {
    const float f0 = __uint_as_float(__byte_perm(v, 0x43000000u, 0x7044));
    const float f1 = __uint_as_float(__byte_perm(v, 0x43000000u, 0x7144));
    const float f2 = __uint_as_float(__byte_perm(v, 0x43000000u, 0x7244));
    const float f3 = __uint_as_float(__byte_perm(v, 0x43000000u, 0x7344));
    const float2 w01 = __ffma2_rn(a, make_float2(f0, f1), c);
    const float2 w23 = __ffma2_rn(a, make_float2(f2, f3), c);
    o0 = pack_bf16(w01.x, w01.y);
    o1 = pack_bf16(w23.x, w23.y);
}

// Q4_K header of super-block `blk` (16-byte aligned) -> FMA operands for
// sub-blocks 2c + hh, c = 0..3 (the ones a thread with quarter qq, hh =
// qq / 2, decodes in the four k-blocks):  w = a*(128 + q) + o with a = d*sc,
// o = -(128 a + dmin*m).  The twelve scale bytes are unpacked four at a time:
// sub-blocks 0-3 take the low 6 bits of bytes 0-3 (scales) and 4-7 (mins);
// sub-blocks 4-7 take the low / high nibble of bytes 8-11 plus the top two
// bits of bytes 0-3 / 4-7.
__device__ __forceinline__ void q4k_operands(const uint8_t* blk, int hh, float2 (&a)[4], float2 (&o)[4]) {
    const uint4 h = lds128_g(blk);
    const uint32_t sh = 8u * (uint32_t)hh;
    const uint32_t sc_lo = (h.y & 0x3F3F3F3Fu) >> sh, m_lo = (h.z & 0x3F3F3F3Fu) >> sh;
    const uint32_t sc_hi = ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u)) >> sh;
    const uint32_t m_hi = (((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u)) >> sh;
    const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
    const uint32_t sc[4] = {sc_lo, sc_lo >> 16, sc_hi, sc_hi >> 16};
    const uint32_t mm[4] = {m_lo, m_lo >> 16, m_hi, m_hi >> 16};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float ds = d * (float)(sc[c] & 0xFFu), dm = dmin * (float)(mm[c] & 0xFFu);
        const float off = -(128.0f * ds + dm);
        a[c] = make_float2(ds, ds);
        o[c] = make_float2(off, off);
    }
}

// 16 Q4_K weights of k-block c, quarter qq (codes: nibble qq / 2 of bytes
// 16 (qq & 1) .. +15 of the k-block's 32 code bytes), operands from
// q4k_operands.
__device__ __forceinline__ void q4k16(const uint8_t* blk, int c, int qq, float2 a, float2 o, uint32_t (&pk)[8]) {
    const uint4 q = lds128_g(blk + 16 + 32 * c + 16 * (qq & 1));
    const uint32_t sh = 4u * (uint32_t)(qq >> 1);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) four_hi((w[i] >> sh) & 0x0F0F0F0Fu, a, o, pk[2 * i], pk[2 * i + 1]);
}

// 16 Q5_K weights of k-block c, quarter qq: the Q4_K codes (at byte 48 of
// the super-block) with bit 2c + qq/2 of qh[16 (qq & 1) + i] as the fifth bit
// of code i; operands from q4k_operands (the header is Q4_K's).
__device__ __forceinline__ void q5k16(const uint8_t* blk, int c, int qq, float2 a, float2 o, uint32_t (&pk)[8]) {
    const uint4 q = lds128_g(blk + 48 + 32 * c + 16 * (qq & 1));
    const uint4 e = lds128_g(blk + 16 + 16 * (qq & 1));
    const uint32_t sh = 4u * (uint32_t)(qq >> 1), hs = 2u * (uint32_t)c + (uint32_t)(qq >> 1);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w}, hb[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        four_hi(((w[i] >> sh) & 0x0F0F0F0Fu) | (((hb[i] >> hs) & 0x01010101u) << 4), a, o, pk[2 * i], pk[2 * i + 1]);
}

// Q8_0: 16 weights of one 34-byte block (2-byte aligned), half `half`:
// w = d*q = 128d*(256 + u/128) - 32896d with u = q + 128.
__device__ __forceinline__ void fast16_q80(const uint8_t* blk, int half, uint32_t (&pk)[8]) {
    uint32_t q[4];
    gv::lds_words_a2<4>(blk + 2 + 16 * half, q);
    const float d = h2f(ld_u16(blk));
    const float2 a = make_float2(128.0f * d, 128.0f * d), cc = make_float2(-32896.0f * d, -32896.0f * d);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = q[i] ^ 0x80808080u;
        const float f0 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7604));
        const float f1 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7614));
        const float f2 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7624));
        const float f3 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7634));
        const float2 w01 = __ffma2_rn(a, make_float2(f0, f1), cc);
        const float2 w23 = __ffma2_rn(a, make_float2(f2, f3), cc);
        pk[2 * i] = pack_bf16(w01.x, w01.y);
        pk[2 * i + 1] = pack_bf16(w23.x, w23.y);
    }
}

// Q6_K: 16 weights o = 64c + 16qq .. of super-block `blk` (2-byte aligned):
// half t = o / 128, group g = (o % 128) / 32; w = d*sc*(q - 32) = ds*(128 + q) - 160 ds.
__device__ __forceinline__ void fast16_q6k(const uint8_t* blk, int c, int qq, uint32_t (&pk)[8]) {
    const int o = 64 * c + 16 * qq, t = o >> 7, g = (o >> 5) & 3, l0 = o & 31;
    uint32_t ql[4], qh[4];
    gv::lds_words_a2<4>(blk + 64 * t + 32 * (g & 1) + l0, ql);
    gv::lds_words_a2<4>(blk + 128 + 32 * t + l0, qh);
    const float d = h2f(ld_u16(blk + 208));
    const float ds = d * (float)(int)(int8_t)blk[192 + 8 * t + 2 * g + (l0 >> 4)];
    const int nsh = 4 * (g >> 1), hsh = 2 * g;
    const float2 a = make_float2(ds, ds), cc = make_float2(-160.0f * ds, -160.0f * ds);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = ((ql[i] >> nsh) & 0x0F0F0F0Fu) | (((qh[i] >> hsh) & 0x03030303u) << 4);
        four_hi(v, a, cc, pk[2 * i], pk[2 * i + 1]);
    }
}

// ---------------------------------------------------------------------------
// 64-weight decoders (small-batch kernel): one thread decodes one tile row's
// 64-wide k-block kk (0..3) of a 256-weight macro-block at `blk` in shared
// memory into 32 bf16x2 words in k order.  Same arithmetic as above: a byte
// permute puts 128 + q (or 256 + u/128) in an fp32 mantissa, one packed FMA
// applies scale and offset, one convert packs two bf16.

// Q4_K (blk 16-byte aligned): k-block kk is sub-blocks 2kk (low nibbles of
// code bytes 32kk .. 32kk+31) and 2kk+1 (their high nibbles).
__device__ __forceinline__ void q4k64(const uint8_t* blk, int kk, uint32_t (&pk)[32]) {
    const uint4 h = lds128_g(blk);
    // Scale / min bytes of sub-blocks 0-3 (kk < 2) or 4-7; this pair is bytes
    // 2(kk & 1) and 2(kk & 1) + 1 of the word.
    const uint32_t scw = kk < 2 ? (h.y & 0x3F3F3F3Fu) : ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u));
    const uint32_t mw = kk < 2 ? (h.z & 0x3F3F3F3Fu) : (((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u));
    const uint32_t sh = 16u * (uint32_t)(kk & 1);
    const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
    const float ds0 = d * (float)((scw >> sh) & 0xFFu), ds1 = d * (float)((scw >> (sh + 8u)) & 0xFFu);
    const float dm0 = dmin * (float)((mw >> sh) & 0xFFu), dm1 = dmin * (float)((mw >> (sh + 8u)) & 0xFFu);
    const float o0 = -(128.0f * ds0 + dm0), o1 = -(128.0f * ds1 + dm1);
    const uint4 c0 = lds128_g(blk + 16 + 32 * kk), c1 = lds128_g(blk + 32 + 32 * kk);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        four_hi(w[i] & 0x0F0F0F0Fu, make_float2(ds0, ds0), make_float2(o0, o0), pk[2 * i], pk[2 * i + 1]);
        four_hi((w[i] >> 4) & 0x0F0F0F0Fu, make_float2(ds1, ds1), make_float2(o1, o1), pk[16 + 2 * i],
                pk[17 + 2 * i]);
    }
}

// Q5_K (blk 16-byte aligned): q4k64's header and codes (at byte 48) with the
// fifth bits of k-block kk: bit 2kk of qh[l] for the low-nibble code of byte
// 32kk + l, bit 2kk + 1 for its high-nibble code.
__device__ __forceinline__ void q5k64(const uint8_t* blk, int kk, uint32_t (&pk)[32]) {
    const uint4 h = lds128_g(blk);
    const uint32_t scw = kk < 2 ? (h.y & 0x3F3F3F3Fu) : ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u));
    const uint32_t mw = kk < 2 ? (h.z & 0x3F3F3F3Fu) : (((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u));
    const uint32_t sh = 16u * (uint32_t)(kk & 1);
    const float d = h2f(h.x & 0xFFFFu), dmin = h2f(h.x >> 16);
    const float ds0 = d * (float)((scw >> sh) & 0xFFu), ds1 = d * (float)((scw >> (sh + 8u)) & 0xFFu);
    const float dm0 = dmin * (float)((mw >> sh) & 0xFFu), dm1 = dmin * (float)((mw >> (sh + 8u)) & 0xFFu);
    const float o0 = -(128.0f * ds0 + dm0), o1 = -(128.0f * ds1 + dm1);
    const uint4 c0 = lds128_g(blk + 48 + 32 * kk), c1 = lds128_g(blk + 64 + 32 * kk);
    const uint4 e0 = lds128_g(blk + 16), e1 = lds128_g(blk + 32);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const uint32_t e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = e[i] >> (2 * kk);   // bit 0: low code's fifth bit, bit 1: high code's
        four_hi((w[i] & 0x0F0F0F0Fu) | ((b << 4) & 0x10101010u), make_float2(ds0, ds0), make_float2(o0, o0),
                pk[2 * i], pk[2 * i + 1]);
        four_hi(((w[i] >> 4) & 0x0F0F0F0Fu) | ((b << 3) & 0x10101010u), make_float2(ds1, ds1),
                make_float2(o1, o1), pk[16 + 2 * i], pk[17 + 2 * i]);
    }
}

// Q2_K (blk 2-byte aligned): k-block kk is weights 64kk .. 64kk+63 = plane
// half t = kk / 2, fields j0 = 2(kk & 1) (first 32) and j0 + 1 (next 32) of
// code bytes 32t .. 32t+31, groups 4kk .. 4kk+3 with their (scale, min)
// bytes 4kk .. 4kk+3 (scale low nibble).  w = ds*q - dm, as a*(128 + q) + o.
__device__ __forceinline__ void q2k64(const uint8_t* blk, int kk, uint32_t (&pk)[32]) {
    const int t = kk >> 1, j0 = 2 * (kk & 1);
    uint32_t qs[8];
    gv::lds_words_a2<8>(blk + 16 + 32 * t, qs);
    const uint32_t sm = ld_u32_a2(blk + 4 * kk);
    const float d = h2f(ld_u16(blk + 80)), dmin = h2f(ld_u16(blk + 82));
    float2 a[4], o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t b = (sm >> (8 * e)) & 0xFFu;
        const float ds = d * (float)(b & 15u), dm = dmin * (float)(b >> 4);
        const float off = -(128.0f * ds + dm);
        a[e] = make_float2(ds, ds);
        o[e] = make_float2(off, off);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {   // code bytes 4i .. 4i+3: weights 4i.. of each 32
        four_hi((qs[i] >> (2 * j0)) & 0x03030303u, a[i >> 2], o[i >> 2], pk[2 * i], pk[2 * i + 1]);
        four_hi((qs[i] >> (2 * j0 + 2)) & 0x03030303u, a[2 + (i >> 2)], o[2 + (i >> 2)], pk[16 + 2 * i],
                pk[17 + 2 * i]);
    }
}

// Q3_K (blk 2-byte aligned): the Q2_K plane at byte 32 with the third bit of
// weight (j, l) at bit 4t + j of hmask[l] (bytes 0-31), u = lo2 + 4 * bit in
// 0..7 and q = u - 4; groups 4kk + e take the signed scale (low four bits:
// nibble t of byte 96 + 4(kk & 1) + e; high two: bits 2kk.. of byte 104 + e;
// minus 32).  w = ds*(u - 4) = ds*(128 + u) - 132 ds.
__device__ __forceinline__ void q3k64(const uint8_t* blk, int kk, uint32_t (&pk)[32]) {
    const int t = kk >> 1, j0 = 2 * (kk & 1);
    uint32_t qs[8], hm[8];
    gv::lds_words_a2<8>(blk + 32 + 32 * t, qs);
    gv::lds_words_a2<8>(blk, hm);
    const uint32_t lo4 = (ld_u32_a2(blk + 96 + 4 * (kk & 1)) >> (4 * t)) & 0x0F0F0F0Fu;
    const uint32_t hi2 = (ld_u32_a2(blk + 104) >> (2 * kk)) & 0x03030303u;
    const uint32_t sw = lo4 | (hi2 << 4);   // byte e: scale of group 4kk + e, plus 32
    const float d = h2f(ld_u16(blk + 108));
    float2 a[4], o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float ds = d * ((float)((sw >> (8 * e)) & 0xFFu) - 32.0f);
        a[e] = make_float2(ds, ds);
        o[e] = make_float2(-132.0f * ds, -132.0f * ds);
    }
    const int hb = 4 * t + j0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t v0 = ((qs[i] >> (2 * j0)) & 0x03030303u) | (((hm[i] >> hb) & 0x01010101u) << 2);
        const uint32_t v1 = ((qs[i] >> (2 * j0 + 2)) & 0x03030303u) | (((hm[i] >> (hb + 1)) & 0x01010101u) << 2);
        four_hi(v0, a[i >> 2], o[i >> 2], pk[2 * i], pk[2 * i + 1]);
        four_hi(v1, a[2 + (i >> 2)], o[2 + (i >> 2)], pk[16 + 2 * i], pk[17 + 2 * i]);
    }
}

// Q6_K (blk 2-byte aligned): k-block kk is half t = kk / 2, groups g = 2(kk & 1)
// and g + 1: low 4 bits from ql[64t .. 64t + 63] (nibble kk & 1), high 2 bits
// from qh[32t + l] bits 2g (+ 2), sixteen-weight scales 8t + 2g .. + 3.
__device__ __forceinline__ void q6k64(const uint8_t* blk, int kk, uint32_t (&pk)[32]) {
    const int t = kk >> 1, hi = kk & 1;
    uint32_t ql[16], qh[8];
    gv::lds_words_a2<16>(blk + 64 * t, ql);
    gv::lds_words_a2<8>(blk + 128 + 32 * t, qh);
    const uint32_t sw = ld_u32_a2(blk + 192 + 8 * t + 4 * hi);
    const float d = h2f(ld_u16(blk + 208));
    float ds[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) ds[e] = d * (float)(int)(int8_t)((sw >> (8 * e)) & 0xFFu);
    const int nsh = 4 * hi, hsh = 4 * hi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = ds[i >> 2], b = ds[2 + (i >> 2)];
        const uint32_t v0 = ((ql[i] >> nsh) & 0x0F0F0F0Fu) | (((qh[i] >> hsh) & 0x03030303u) << 4);
        const uint32_t v1 = ((ql[8 + i] >> nsh) & 0x0F0F0F0Fu) | (((qh[i] >> (hsh + 2)) & 0x03030303u) << 4);
        four_hi(v0, make_float2(a, a), make_float2(-160.0f * a, -160.0f * a), pk[2 * i], pk[2 * i + 1]);
        four_hi(v1, make_float2(b, b), make_float2(-160.0f * b, -160.0f * b), pk[16 + 2 * i], pk[17 + 2 * i]);
    }
}

// Bits 0-3 of x to bit 0 of bytes 0-3.
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

// One 32-weight block (2-byte aligned) -> 16 words.  Q8_0: d, 32 signed codes,
// w = d*q.  Q5_0: d, a word of fifth bits, 16 nibble bytes, w = d*(q - 16).
// Q4_0: d, 16 nibble bytes, w = d*(q - 8).  Nibble bytes: element j low,
// element j + 16 high.
template <int T>
__device__ __forceinline__ void block32(const uint8_t* b, uint32_t* pk) {
    const float d = h2f(ld_u16(b));
    if constexpr (T == T_Q8_0) {
        uint32_t q[8];
        gv::lds_words_a2<8>(b + 2, q);
        const float2 a = make_float2(128.0f * d, 128.0f * d), c = make_float2(-32896.0f * d, -32896.0f * d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t u = q[i] ^ 0x80808080u;
            const float f0 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7604));
            const float f1 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7614));
            const float f2 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7624));
            const float f3 = __uint_as_float(__byte_perm(u, 0x43800000u, 0x7634));
            const float2 w01 = __ffma2_rn(a, make_float2(f0, f1), c);
            const float2 w23 = __ffma2_rn(a, make_float2(f2, f3), c);
            pk[2 * i] = pack_bf16(w01.x, w01.y);
            pk[2 * i + 1] = pack_bf16(w23.x, w23.y);
        }
    } else {
        constexpr bool k5 = T == T_Q5_0;
        uint32_t qs[4];
        gv::lds_words_a2<4>(b + (k5 ? 6 : 2), qs);
        const uint32_t qh = k5 ? ld_u32_a2(b + 2) : 0u;
        const float off = k5 ? -144.0f * d : -136.0f * d;
        const float2 a = make_float2(d, d), c = make_float2(off, off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = (qs[i] & 0x0F0F0F0Fu) | (k5 ? spread4((qh >> (4 * i)) & 15u) << 4 : 0u);
            const uint32_t hi = ((qs[i] >> 4) & 0x0F0F0F0Fu) | (k5 ? spread4((qh >> (16 + 4 * i)) & 15u) << 4 : 0u);
            four_hi(lo, a, c, pk[2 * i], pk[2 * i + 1]);
            four_hi(hi, a, c, pk[8 + 2 * i], pk[9 + 2 * i]);
        }
    }
}

// Generic (Q5_0, Q4_0) 16 weights via the shared decoders: k in [k0, k0 + 16).
template <int T>
__device__ __forceinline__ void generic16(const uint8_t* mb, int o, uint32_t (&pk)[8]) {
    using F = Fmt<T>;
    int u, h;
    locate<T>(o % F::BE, u, h);
    float w[16];
    dequant_half<T>(mb + (o / F::BE) * F::BB, u, h, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16(w[2 * i], w[2 * i + 1]);
}

// Copy macro-block `m` of one warp's 8 tile rows (8 dw .. 8 dw + 7) into
// packed slot `dst` with 16-byte cp.async (each row's aligned-down window).
// The (row, chunk) pairs are numbered row-major over SLOT / 16 chunk places
// per row and taken by consecutive lanes, so that one instruction's lanes
// read a few rows' contiguous windows (few cache lines) and write
// consecutive 16-byte units of shared memory (a slot is an odd number of
// them: no bank conflicts).  Bytes past the last full 16 bytes of W are
// loaded by the consumer of that row (tail_fix).
template <int T>
__device__ __forceinline__ void issue_packed(const Args& p, uint8_t* dst, int64_t row0, int64_t m, int dw, int lane) {
    using K = PkGeo<T>;
    constexpr int NCH = K::SLOT / 16;   // chunk places per row (at least the longest window)
    const int64_t kb0 = m * K::MB;
    const int64_t len = min((int64_t)K::MB, p.cols - kb0) / Fmt<T>::BE * Fmt<T>::BB;
#pragma unroll
    for (int k = 0; k < (8 * NCH + 31) / 32; ++k) {
        const int pr = lane + 32 * k, rl = pr / NCH, ch = pr - rl * NCH;
        const int r = 8 * dw + rl;
        const int64_t row = row0 + r;
        if (rl < 8 && row < p.rows) {
            const int64_t st = row * p.row_bytes + m * K::BYTES;
            const int64_t a = st & ~(int64_t)15;
            const int64_t e = min((st + len + 15) & ~(int64_t)15, p.total16);
            if (a + 16 * ch < e) cp_async16(dst + r * K::SLOT + 16 * ch, p.W + a + 16 * ch);
        }
    }
}

template <int T>
__device__ __forceinline__ void tail_fix(const Args& p, uint8_t* slot_row, int64_t row, int64_t m) {
    using K = PkGeo<T>;
    const int64_t kb0 = m * K::MB;
    const int64_t len = min((int64_t)K::MB, p.cols - kb0) / Fmt<T>::BE * Fmt<T>::BB;
    const int64_t st = row * p.row_bytes + m * K::BYTES;
    if (st + len <= p.total16) return;
    uint8_t* base = slot_row - (st & ~(int64_t)15);
    for (int64_t b = max(st, p.total16); b < st + len; ++b) base[b] = p.W[b];
}

template <int T, class C>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Args p) {
    using K = Pk<T, C>;
    constexpr int kNS = C::NS, kNSP = C::NSP, kBNM = C::BNM;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (the 128-byte swizzle atoms must be aligned).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* xring = smem + K::OFF_X;
    const int nsb = p.nsb;
    uint8_t* packed = smem + K::OFF_X + nsb * p.xst;
    uint64_t* full_w = reinterpret_cast<uint64_t*>(packed + kNSP * K::STAGE);   // weight stage written
    uint64_t* empty = full_w + kNS;                                             // weight stage consumed
    uint64_t* full_x = empty + kNS;                                             // activation stage landed
    uint64_t* empty_x = full_x + nsb;                                           // activation stage consumed
    uint64_t* accum = empty_x + nsb;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Token tiles vary fastest: the CTAs that share a weight tile run
    // together, so each packed weight byte comes from DRAM once.
    const int64_t row0 = (int64_t)blockIdx.y * kBM;
    const int64_t tok0 = (int64_t)blockIdx.x * C::BN;
    const int nacc = C::NACC > 1 && p.M - tok0 > kBNM ? 2 : 1;   // accumulators holding real tokens
    // This CTA's share of K: k-blocks [kb0, kb1) (blockIdx.z = split).
    const int kb0 = (int)blockIdx.z * p.kb_per_split;
    const int kb1 = min(p.nkb, kb0 + p.kb_per_split);
    const int nk = kb1 - kb0;
    // Macro-blocks m0 .. m0 + nmb - 1 cover these k-blocks (kb0 is a multiple
    // of the macro-block's k-blocks).
    const int m0 = kb0 / K::KPM;
    const int nmb = (kb1 + K::KPM - 1) / K::KPM - m0;
    const uint32_t bsub = (uint32_t)p.nmma * (kBK * 2);   // bytes of one accumulator's activation tile
    float* out = p.part ? p.part + (size_t)blockIdx.z * (size_t)p.M * (size_t)p.rows : p.Y;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&full_w[s], kDeqWarps);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < nsb; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&empty_x[s], 1);
        }
        mbar_init(accum, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::TMEM);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        // TMA producer for the activation tiles (they may come from the
        // previous kernel: wait for it first).
        if (lane == 0) {
            pdl_wait_prior();
            int issued = 0, s = 0;
            uint32_t par = 1;   // phase parity of empty_x[s] to wait for (from the second lap)
            for (int kb = kb0; kb < kb1; ++kb) {
                if (issued >= nsb && !mbar_wait_sleep_bounded(&empty_x[s], par, p.status)) break;
                mbar_arrive_expect_tx(&full_x[s], bsub * (uint32_t)nacc);
                for (int j = 0; j < nacc; ++j)
                    tc::tma_load_2d(xring + s * p.xst + j * bsub, &xmap, kb * kBK, (int)tok0 + kBNM * j, &full_x[s]);
                ++issued;
                if (++s == nsb) {
                    s = 0;
                    par ^= 1u;
                }
            }
            // Every load issued must land before the CTA may exit.
            for (int i = issued > nsb ? issued - nsb : 0; i < issued; ++i)
                mbar_wait_bounded(&full_x[i % nsb], (uint32_t)((i / nsb) & 1), p.status);
        }
    } else if (warp == 1) {
        // MMA issuer: lane 0 runs the loop.  Descriptor start addresses
        // advance in 16-byte units from the ring bases.
        const bool leader = lane == 0;
        const uint32_t idesc = tc::idesc_bf16_f32(kBM, p.nmma);
        const uint64_t da0 = tc::sdesc_k128(smem_u32(smem)), db0 = tc::sdesc_k128(smem_u32(xring));
        const uint64_t dbj = (uint64_t)(bsub >> 4);   // second accumulator's activation tile
        int s = 0, sx = 0;
        uint32_t par = 0, parx = 0;   // phase parities of full_w[s] and full_x[sx]
        for (int i = 0; i < nk && leader; ++i) {
            if (!mbar_wait_sleep_bounded(&full_x[sx], parx, p.status) ||
                !mbar_wait_sleep_bounded(&full_w[s], par, p.status))
                break;
            tc::fence_after_sync();
            const uint64_t da = da0 + (uint64_t)((s * kA) >> 4), db = db0 + (uint64_t)((sx * p.xst) >> 4);
            if (leader) {
                for (int j = 0; j < nacc; ++j) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16(tmem + kBNM * j, da + 2 * kk, db + dbj * j + 2 * kk, idesc,
                                     (i | kk) != 0 ? 1u : 0u);
                }
                tc::commit(&empty[s]);     // both stages free once these MMAs complete
                tc::commit(&empty_x[sx]);
            }
            if (++s == kNS) {
                s = 0;
                par ^= 1u;
            }
            if (++sx == nsb) {
                sx = 0;
                parx ^= 1u;
            }
        }
        if (leader) tc::commit(accum);   // fires once every MMA issued above has completed
        __syncwarp();
        // Tensor memory may only be released after the MMAs are done.
        if (lane == 0) mbar_wait_sleep_bounded(accum, 0, p.status);
        __syncwarp();
    } else {
        // Dequant warps.  Warp dw owns tile rows 8dw .. 8dw+7; lane -> (row
        // 8dw + lane/4, 16-weight quarter lane%4 of each 64-wide k-block).  The
        // warp streams its rows' packed macro-blocks into an NSP-deep ring with
        // cp.async and decodes them with no CTA barrier.
        const int dw = warp - 2;
        const int r = 8 * dw + (lane >> 2), qq = lane & 3;
        const int64_t row = row0 + r;
        const bool live = row < p.rows;
        // This thread's two swizzled 16-byte chunks inside an operand stage.
        const uint32_t rbase = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
        const uint32_t dst0 = rbase + ((((uint32_t)(2 * qq)) ^ (uint32_t)(r & 7)) << 4);
        const uint32_t dst1 = rbase + ((((uint32_t)(2 * qq + 1)) ^ (uint32_t)(r & 7)) << 4);
        // k-block kb holds this thread's 16 weights iff 64 kb < kq.
        const int64_t kq = p.cols - 16 * qq;
        bool ok = true;
        int s = 0;            // operand stage of the next local k-block
        uint32_t par = 1;     // phase parity of empty[s] to wait for (after the first NS k-blocks)
        int li = 0;           // local k-block
        int ps = 0;           // packed slot of the current macro-block
#pragma unroll 1
        for (int mi = 0; mi < kNSP - 1; ++mi) {
            if (mi < nmb) issue_packed<T>(p, packed + mi * K::STAGE, row0, (int64_t)(m0 + mi), dw, lane);
            cp_async_commit();
        }
#pragma unroll 1
        for (int mi = 0; mi < nmb; ++mi) {
            const int m = m0 + mi;
            const int pn = ps == 0 ? kNSP - 1 : ps - 1;   // slot of macro-block mi + NSP - 1
            if (mi + kNSP - 1 < nmb)
                issue_packed<T>(p, packed + pn * K::STAGE, row0, (int64_t)(m + kNSP - 1), dw, lane);
            cp_async_commit();
            cp_async_wait<kNSP - 1>();
            uint8_t* pk = packed + ps * K::STAGE;
            if (qq == 0 && live) tail_fix<T>(p, pk + r * K::SLOT, row, (int64_t)m);
            __syncwarp();   // this warp's rows of macro-block m are visible
            const int64_t st = row * p.row_bytes + (int64_t)m * K::BYTES;
            const uint8_t* mbp = pk + r * K::SLOT + (int)(st & 15);
            const int kbm = m * K::KPM;
            float2 qa[4], qo[4];
            if constexpr (T == T_Q4_K || T == T_Q5_K) {
                if (live) q4k_operands(mbp, qq >> 1, qa, qo);
            }
#pragma unroll
            for (int kk = 0; kk < K::KPM; ++kk) {
                const int kb = kbm + kk;
                if (kb >= kb1) break;
                if (ok && li >= kNS) {   // one lane polls, the warp follows
                    int good = 1;
                    if (lane == 0) good = mbar_wait_bounded(&empty[s], par, p.status);
                    ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                }
                if (ok) {
                    uint32_t pk8[8];
                    if (live && (int64_t)kb * kBK < kq) {
                        if constexpr (T == T_Q4_K) q4k16(mbp, kk, qq, qa[kk], qo[kk], pk8);
                        else if constexpr (T == T_Q5_K) q5k16(mbp, kk, qq, qa[kk], qo[kk], pk8);
                        else if constexpr (T == T_Q6_K) fast16_q6k(mbp, kk, qq, pk8);
                        else if constexpr (T == T_Q8_0) fast16_q80(mbp + (2 * kk + (qq >> 1)) * 34, qq & 1, pk8);
                        else generic16<T>(mbp, kk * kBK + 16 * qq, pk8);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) pk8[i] = 0u;
                    }
                    uint8_t* As = smem + s * kA;
                    *reinterpret_cast<uint4*>(As + dst0) = make_uint4(pk8[0], pk8[1], pk8[2], pk8[3]);
                    *reinterpret_cast<uint4*>(As + dst1) = make_uint4(pk8[4], pk8[5], pk8[6], pk8[7]);
                }
                fence_proxy_async_smem();   // generic stores -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_w[s]);
                ++li;
                if (++s == kNS) {
                    s = 0;
                    par ^= 1u;
                }
            }
            __syncwarp();   // this warp is done reading slot ps
            if (++ps == kNSP) ps = 0;
        }
        cp_async_wait<0>();
        // Epilogue: warp w may read tensor-memory lanes 32 (w % 4) .. +31 (its
        // quarter of the weight rows); the four warps of a quarter split the
        // accumulator columns (tokens) into four equal groups.
        {
            constexpr int kGrp = C::BN / 4;
            const int q = warp & 3, grp = dw >> 2;
            if (lane == 0) mbar_wait_sleep_bounded(accum, 0, p.status);
            __syncwarp();
            tc::fence_after_sync();
            const int64_t orow = row0 + 32 * q + lane;
#pragma unroll 1
            for (int j = 0; j < kGrp / 16; ++j) {
                const int col = kGrp * grp + 16 * j;
                if (tok0 + col >= p.M) break;   // warp-uniform
                uint32_t v[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + col, v);
                tc::tmem_wait_ld();
                if (orow < p.rows) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t tok = tok0 + col + i;
                        if (tok < p.M) out[tok * p.rows + orow] = __uint_as_float(v[i]);
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::TMEM);
    }
}

// ---------------------------------------------------------------------------
// Small-batch dequant-GEMM (M <= 64, one token tile): each dequant thread owns
// one weight row and decodes a whole 64-wide k-block of it, so scale decoding,
// synchronisation and stores are paid once per 64 weights.
//   warp 0  TMA producer of the activation tiles (its own ring);
//   warps 1-2  MMA issuers: warp 1 + w takes local k-blocks w, w + 2, ...
//           into accumulator w (issuing a k-block's MMAs and commits costs a
//           few hundred ns whatever N is, so two issuers halve that per
//           k-block); the epilogue adds the two accumulators in order.  Each
//           runs its loop on the whole warp, one elected lane issuing;
//   warp 3  packed producer: each 256-weight macro-block of the 128 rows into
//           a CTA-wide ring (full_p / empty_p barriers) as one 2D TMA box of
//           W seen as [rows, row_bytes] (row_bytes must be a multiple of 16:
//           the planner sends other shapes to gemm_kernel);
//   warps 4..19  dequant: row quarter q = warp % 4 (the TMEM lanes it may
//           read back), phase ph = (warp - 4) / 4: k-block ph of every
//           macro-block; the four warps of a phase fill one weight stage.
template <int T>
__global__ void __launch_bounds__(kSkThreads, 1) gemm_skinny_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                   const __grid_constant__ CUtensorMap wmap,
                                                                   const Args p) {
    using G = SkGeo<T>;
    using F = Fmt<T>;
    constexpr int kNS = G::NS, kNSP = G::NSP;
    static_assert(kNS % kSkMma == 0, "each MMA warp owns whole weight stages");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-aligned (swizzle atoms)
    const int nsb = p.nsb;
    uint8_t* xring = smem + kNS * kA;
    uint8_t* packed = xring + nsb * p.xst;
    uint64_t* full_w = reinterpret_cast<uint64_t*>(packed + kNSP * G::STAGE);
    uint64_t* empty = full_w + kNS;
    uint64_t* full_x = empty + kNS;
    uint64_t* empty_x = full_x + nsb;
    uint64_t* full_p = empty_x + nsb;
    uint64_t* empty_p = full_p + kNSP;
    uint64_t* accum = empty_p + kNSP;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)blockIdx.y * kBM;
    const int kb0 = (int)blockIdx.z * p.kb_per_split;   // a multiple of 4
    const int kb1 = min(p.nkb, kb0 + p.kb_per_split);
    const int nk = kb1 - kb0;
    const int m0 = kb0 / 4, nmb = (kb1 + 3) / 4 - m0;
    const uint32_t bsub = (uint32_t)p.nmma * (kBK * 2);
    float* out = p.part ? p.part + (size_t)blockIdx.z * (size_t)p.M * (size_t)p.rows : p.Y;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&full_w[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < nsb; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&empty_x[s], 1);
        }
        for (int s = 0; s < kNSP; ++s) {
            mbar_init(&full_p[s], 1);
            mbar_init(&empty_p[s], kDeqWarps);
        }
        mbar_init(accum, kSkMma);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kSkTmem);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        // Activation tiles (they may come from the previous kernel: wait for it).
        if (lane == 0) {
            pdl_wait_prior();
            int issued = 0, s = 0;
            uint32_t par = 1;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (issued >= nsb && !mbar_wait_sleep_bounded(&empty_x[s], par, p.status)) break;
                mbar_arrive_expect_tx(&full_x[s], bsub);
                tc::tma_load_2d(xring + s * p.xst, &xmap, kb * kBK, 0, &full_x[s]);
                ++issued;
                if (++s == nsb) {
                    s = 0;
                    par ^= 1u;
                }
            }
            for (int i = issued > nsb ? issued - nsb : 0; i < issued; ++i)
                mbar_wait_bounded(&full_x[i % nsb], (uint32_t)((i / nsb) & 1), p.status);
        }
    } else if (warp <= kSkMma) {
        // MMA issuer w: local k-blocks w, w + kSkMma, ... into accumulator w
        // (weight stage and activation stage both advance by kSkMma; NS and
        // the activation ring depth are multiples of kSkMma).
        const int mw = warp - 1;
        const bool leader = tc::elect_one();
        const uint32_t idesc = tc::idesc_bf16_f32(kBM, p.nmma);
        const uint64_t da0 = tc::sdesc_k128(smem_u32(smem)), db0 = tc::sdesc_k128(smem_u32(xring));
        const uint32_t acc = tmem + (uint32_t)(64 * mw);
        int s = mw, sx = mw;
        uint32_t par = 0, parx = 0;
        for (int i = mw; i < nk; i += kSkMma) {
            int good = 1;
            if (lane == 0)
                good = mbar_wait_sleep_bounded(&full_x[sx], parx, p.status) &&
                       mbar_wait_sleep_bounded(&full_w[s], par, p.status);
            if (__shfl_sync(0xffffffffu, good, 0) == 0) break;
            tc::fence_after_sync();
            const uint64_t da = da0 + (uint64_t)((s * kA) >> 4), db = db0 + (uint64_t)((sx * p.xst) >> 4);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc::mma_bf16(acc, da + 2 * kk, db + 2 * kk, idesc, (i != mw || kk != 0) ? 1u : 0u);
                tc::commit(&empty[s]);
                tc::commit(&empty_x[sx]);
            }
            __syncwarp();
            if ((s += kSkMma) >= kNS) {
                s -= kNS;
                par ^= 1u;
            }
            if ((sx += kSkMma) >= nsb) {
                sx -= nsb;
                parx ^= 1u;
            }
        }
        if (leader) tc::commit(accum);
        __syncwarp();
        if (lane == 0) mbar_wait_sleep_bounded(accum, 0, p.status);
        __syncwarp();
    } else if (warp == kSkMma + 1) {
        // Packed producer: each macro-block of the tile's 128 rows as one 2D
        // TMA box of W seen as [rows, row_bytes] (4-byte elements): rows past
        // the matrix and bytes past a row's end arrive as zeros.
        int ps = 0, issued = 0;
        uint32_t par = 1;
        if (lane == 0) {
            for (int mi = 0; mi < nmb; ++mi) {
                const int64_t m = m0 + mi;
                if (mi >= kNSP && !mbar_wait_sleep_bounded(&empty_p[ps], par, p.status)) break;
                mbar_arrive_expect_tx(&full_p[ps], (uint32_t)(kBM * G::BOXW));
                tc::tma_load_2d(packed + ps * G::STAGE, &wmap, (int)(((m * G::BYTES) & ~(int64_t)15) / 4), (int)row0,
                                &full_p[ps]);
                ++issued;
                if (++ps == kNSP) {
                    ps = 0;
                    par ^= 1u;
                }
            }
            // Every copy issued must land before the CTA may exit.
            for (int i = issued > kNSP ? issued - kNSP : 0; i < issued; ++i)
                mbar_wait_bounded(&full_p[i % kNSP], (uint32_t)((i / kNSP) & 1), p.status);
        }
    } else {
        const int q = warp & 3, ph = (warp - kSkMma - 2) >> 2;
        const int r = 32 * q + lane;
        const int64_t row = row0 + r;
        const bool live = row < p.rows;
        const uint32_t line = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);   // row r's line in a weight stage
        bool ok = true;
        int ps = 0;
        uint32_t ppar = 0;
#pragma unroll 1
        for (int mi = 0; mi < nmb; ++mi) {
            const int m = m0 + mi;
            if (ok) {
                int good = 1;
                if (lane == 0) good = mbar_wait_bounded(&full_p[ps], ppar, p.status);
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
            const int kb = 4 * m + ph;
            if (kb < kb1) {
                const int li = kb - kb0;
                const int s = li % kNS;
                if (ok && li >= kNS) {
                    int good = 1;
                    if (lane == 0) good = mbar_wait_bounded(&empty[s], (uint32_t)((li / kNS - 1) & 1), p.status);
                    ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                }
                if (ok) {
                    uint32_t pk[32];
                    if (live) {
                        const int64_t st = row * p.row_bytes + (int64_t)m * G::BYTES;
                        const uint8_t* blk = packed + ps * G::STAGE + r * G::BOXW + (int)(st & 15);
                        if constexpr (T == T_Q4_K) {
                            q4k64(blk, ph, pk);
                        } else if constexpr (T == T_Q5_K) {
                            q5k64(blk, ph, pk);
                        } else if constexpr (T == T_Q2_K) {
                            q2k64(blk, ph, pk);
                        } else if constexpr (T == T_Q3_K) {
                            q3k64(blk, ph, pk);
                        } else if constexpr (T == T_Q6_K) {
                            q6k64(blk, ph, pk);
                        } else {
                            // Two 32-weight blocks; the second may lie past cols.
                            block32<T>(blk + (2 * ph) * F::BB, pk);
                            if ((int64_t)kb * kBK + 32 < p.cols) {
                                block32<T>(blk + (2 * ph + 1) * F::BB, pk + 16);
                            } else {
#pragma unroll
                                for (int i = 16; i < 32; ++i) pk[i] = 0u;
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) pk[i] = 0u;
                    }
                    uint8_t* As = smem + s * kA + line;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(As + ((c ^ (r & 7)) << 4)) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                }
                fence_proxy_async_smem();   // generic stores -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_w[s]);
            }
            __syncwarp();   // every lane is done reading packed slot ps
            if (lane == 0) mbar_arrive(&empty_p[ps]);
            if (++ps == kNSP) {
                ps = 0;
                ppar ^= 1u;
            }
        }
        // Epilogue: warp reads TMEM lanes 32q .. 32q+31; the four phases of a
        // quarter split the 64 columns into groups of 16.
        if (lane == 0) mbar_wait_sleep_bounded(accum, 0, p.status);
        __syncwarp();
        tc::fence_after_sync();
        const int col = 16 * ph;
        if (col < p.M) {
            uint32_t v[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + col, v);
            tc::tmem_wait_ld();
#pragma unroll 1
            for (int w = 1; w < kSkMma && w < nk; ++w) {   // the other accumulators, in order
                uint32_t u[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * w) + col, u);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(u[e]));
            }
            if (live) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (col + i < p.M) out[(int64_t)(col + i) * p.rows + row] = __uint_as_float(v[i]);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kSkTmem);
    }
}

// Y = sum over splits of the partials, in split order (deterministic).
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ part, int splits, int64_t n,
                                                           float* __restrict__ Y) {
    pdl_wait_prior();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float a = part[i];
        for (int s = 1; s < splits; ++s) a += part[(int64_t)s * n + i];
        Y[i] = a;
    }
}

}  // namespace gm
}  // namespace qk

namespace qk {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int T, class C>
static cudaError_t gemm_tc(gm::Args a, const GemmPlan& pl, const CUtensorMap& map, cudaStream_t s) {
    using K = gm::Pk<T, C>;
    // Activation ring: stages of one 64-wide k-block for every accumulator a
    // token tile can fill; as many as fit (at most 16).
    a.xst = (C::NACC > 1 && a.M > C::BNM ? C::NACC : 1) * a.nmma * gm::kBK * 2;
    a.nsb = std::min(gm::kMaxXStages, (gm::kSmemMax - K::smem(0, 0)) / (a.xst + 16));
    if (a.nsb < 1) return cudaErrorInvalidValue;
    const int smem = K::smem(a.nsb, a.xst);
    auto kern = gm::gemm_kernel<T, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gm::kSmemMax);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.M + C::BN - 1) / C::BN), (unsigned)((a.rows + gm::kBM - 1) / gm::kBM),
                       (unsigned)pl.splits);
    cfg.blockDim = dim3(gm::kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

template <int T>
static cudaError_t gemm_sk(gm::Args a, const GemmPlan& pl, const CUtensorMap& map, cudaStream_t s) {
    using G = gm::SkGeo<T>;
    // Packed weights by 2D TMA: W (16-byte aligned, rows a multiple of 16
    // bytes: the planner checks) as 4-byte elements, box (BOXW / 4) x 128 rows.
    if (a.row_bytes % 16 != 0) return cudaErrorInvalidValue;
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap wmap;
    cuuint64_t gdim[2] = {(cuuint64_t)(a.row_bytes / 4), (cuuint64_t)a.rows};
    cuuint64_t gstride[1] = {(cuuint64_t)a.row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(G::BOXW / 4), (cuuint32_t)gm::kBM};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(a.W), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // Activation ring: one nmma x 64 tile per stage, as many as fit (at most 16).
    a.xst = a.nmma * gm::kBK * 2;
    a.nsb = std::min(gm::kMaxXStages, (gm::kSmemMax - G::smem(0, 0)) / (a.xst + 16)) / gm::kSkMma * gm::kSkMma;
    if (a.nsb < gm::kSkMma) return cudaErrorInvalidValue;
    const int smem = G::smem(a.nsb, a.xst);
    auto kern = gm::gemm_skinny_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gm::kSmemMax);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1u, (unsigned)((a.rows + gm::kBM - 1) / gm::kBM), (unsigned)pl.splits);
    cfg.blockDim = dim3(gm::kSkThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, wmap, a);
}

template <int T>
static cudaError_t gemm_t(const gm::Args& a, const GemmPlan& pl, const CUtensorMap& map, cudaStream_t s) {
    return pl.skinny ? gemm_sk<T>(a, pl, map, s) : gemm_tc<T, gm::Wide>(a, pl, map, s);
}

namespace {
int k_blocks_per_macro(int type) { return type == T_Q8_0 ? 2 : 4; }   // PkGeo<T>::KPM
}  // namespace

// Split K when the (token, row) tiles leave SMs idle: among 1..16 splits
// (on macro-block boundaries) take the fewest waves x k-blocks per CTA, with
// a fixed cost of ~6 k-blocks per CTA for its prologue and epilogue.  Only a
// single token tile is split (the partials, splits x M x rows floats, are
// small there), and only for a gain of at least 15 %.
GemmPlan plan_gemm(int type, int64_t rows, int64_t cols, int64_t M, int sms) {
    GemmPlan pl;
    if (rows <= 0 || cols <= 0 || M <= 0) return pl;
    const int64_t nkb = (cols + gm::kBK - 1) / gm::kBK;
    // Small batches take gemm_skinny_kernel when W's rows can be loaded as TMA
    // boxes (row bytes a multiple of 16), else gemm_kernel.
    int64_t rb = 0;
    switch (type) {
    case T_Q4_K: rb = cols / 256 * 144; break;
    case T_Q6_K: rb = cols / 256 * 210; break;
    case T_Q8_0: rb = cols / 32 * 34; break;
    case T_Q5_0: rb = cols / 32 * 22; break;
    case T_Q4_0: rb = cols / 32 * 18; break;
    case T_Q5_K: rb = cols / 256 * 176; break;
    case T_Q2_K: rb = cols / 256 * 84; break;
    case T_Q3_K: rb = cols / 256 * 110; break;
    }
    pl.skinny = M <= gm::kSkinnyBN && rb % 16 == 0;
    const int64_t kpm = pl.skinny ? 4 : k_blocks_per_macro(type);   // the small-batch kernel's macro-blocks are 256 wide
    const int64_t bn = M <= gm::kSkinnyBN ? gm::kSkinnyBN : gm::Wide::BN;
    pl.nmma = M > gm::Wide::BNM ? gm::Wide::BNM : (int)std::max<int64_t>(16, (M + 15) / 16 * 16);
    const int64_t tiles = ((M + bn - 1) / bn) * ((rows + gm::kBM - 1) / gm::kBM);
    const int64_t S = std::max(sms, 1);
    int64_t best_cost = -1;
    const int64_t max_split = M <= bn ? 16 : 1;
    for (int64_t sp = 1; sp <= max_split; ++sp) {
        const int64_t kps = ((nkb + sp - 1) / sp + kpm - 1) / kpm * kpm;
        const int64_t se = (nkb + kps - 1) / kps;
        if (se != sp && sp > 1) continue;
        const int64_t waves = (tiles * se + S - 1) / S;
        const int64_t cost = waves * (kps + 6) * (se > 1 ? 20 : 17);   // splitting must win by 15 %
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            pl.splits = (int)se;
            pl.kb_per_split = (int)kps;
        }
    }
    pl.ws_bytes = pl.splits > 1 ? (int64_t)pl.splits * M * rows * (int64_t)sizeof(float) : 0;
    return pl;
}

cudaError_t launch_gemm(int type, const GemmPlan& pl, const uint8_t* W, int64_t rows, int64_t cols, const void* X,
                        int64_t M, float* Y, float* ws, unsigned* status, cudaStream_t s) {
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    // X: bf16 [M, cols] row-major; tiles of 64 (k) x nmma (tokens), 128-byte swizzle.
    CUtensorMap map;
    cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)M};
    cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)gm::kBK, (cuuint32_t)pl.nmma};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    gm::Args a = {};
    a.W = W;
    a.rows = rows;
    a.cols = cols;
    a.M = M;
    a.Y = Y;
    a.part = pl.splits > 1 ? ws : nullptr;
    a.status = status;
    a.nkb = (int)((cols + gm::kBK - 1) / gm::kBK);
    a.kb_per_split = pl.kb_per_split > 0 ? pl.kb_per_split : a.nkb;
    a.nmma = pl.nmma;
    switch (type) {
    case T_Q4_K: a.row_bytes = cols / 256 * 144; break;
    case T_Q6_K: a.row_bytes = cols / 256 * 210; break;
    case T_Q8_0: a.row_bytes = cols / 32 * 34; break;
    case T_Q5_0: a.row_bytes = cols / 32 * 22; break;
    case T_Q4_0: a.row_bytes = cols / 32 * 18; break;
    case T_Q5_K: a.row_bytes = cols / 256 * 176; break;
    case T_Q2_K: a.row_bytes = cols / 256 * 84; break;
    case T_Q3_K: a.row_bytes = cols / 256 * 110; break;
    default: return cudaErrorInvalidValue;
    }
    a.total16 = (rows * a.row_bytes) & ~(int64_t)15;
    cudaError_t e = cudaErrorInvalidValue;
    switch (type) {
    case T_Q4_K: e = gemm_t<T_Q4_K>(a, pl, map, s); break;
    case T_Q6_K: e = gemm_t<T_Q6_K>(a, pl, map, s); break;
    case T_Q8_0: e = gemm_t<T_Q8_0>(a, pl, map, s); break;
    case T_Q5_0: e = gemm_t<T_Q5_0>(a, pl, map, s); break;
    case T_Q4_0: e = gemm_t<T_Q4_0>(a, pl, map, s); break;
    case T_Q5_K: e = gemm_t<T_Q5_K>(a, pl, map, s); break;
    case T_Q2_K: e = gemm_t<T_Q2_K>(a, pl, map, s); break;
    case T_Q3_K: e = gemm_t<T_Q3_K>(a, pl, map, s); break;
    }
    if (e != cudaSuccess || pl.splits <= 1) return e;
    // Add the partials in split order.
    const int64_t n = M * rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gm::reduce_splits_kernel, (const float*)ws, pl.splits, n, Y);
}

}  // namespace qk
