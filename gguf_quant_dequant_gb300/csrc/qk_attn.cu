// qk_attn.cu -- decode attention over a block-quantized KV cache.
//
// "Hitchhiker's Guide -- Lab 01", 13.2: the KV-cache is quantized at serve
// time (q8_0 the safe default, q4_0 at a quality cost) and read inside
// attention; the heads share K/V in groups (grouped-query attention).  One
// query token: for query head h and its kv head g = h / (n_heads / n_kv),
//   s_t = scale * q_h . K[t, g],  p = softmax(s),  out_h = sum_t p_t V[t, g].
// K and V are [T, n_kv, d]; each (t, g) row is d/32 blocks of a 32-weight
// type (Q8_0, Q5_0, Q4_0), decoded in the dot products.
//
// Split over positions (the cache is streamed once per token, so the work is
// HBM-bound): CTA c n_kv + g takes kv head g and positions [CH c, CH c + CH).
// The chunk CH is set per cache type: a smaller chunk lowers the shared
// memory per CTA, so more CTAs share an SM and hide each other's latency,
// but repeats the per-CTA work (query limbs, softmax, warp sums) more often.
// All its K rows and then all its V rows are requested at once with 16-byte
// cp.async copies into shared memory (each row's aligned-down window; the
// copy that reaches the end of the cache takes only the bytes that exist),
// so every byte of the chunk is in flight together; the scores start as
// soon as the K rows have landed, while V is still arriving.
// Pass 1 runs on the fp16 warp MMA (m16n8k16, fp32 accumulation), the
// arithmetic of the decode GEMV: A = 16 positions x 16 elements of K codes
// minus the type's code offset, exact in fp16; B = the group's queries, two
// fp16 terms (hi, lo) per element after a power-of-two scale per 32-block,
// one column per (head, term), 8 columns per n-tile; each block's two k16
// steps are drained into fp32 scores with the block's d and the query
// block's scale.  Every query element keeps about 22 significant bits
// whatever the largest element of its block is (massive activations in the
// query cost no accuracy elsewhere).  Warp w takes the 16-position tiles
// w, w + 8, ...  The chunk's softmax statistics (max, sum of exp) follow in
// shared memory.
// Pass 2: each warp takes every 8th position; lane l owns d/32 elements of
// V and accumulates sum_t e^(s_t - m) V[t, g]
// per head; the warps' sums are added in warp order.  A second kernel
// combines the chunks (log-sum-exp) in a fixed order: deterministic.
#include <algorithm>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_hunits.cuh"
#include "qk_ptx.cuh"
#include "qk_tc.cuh"

namespace qk {
namespace attn {

constexpr int kMinChunk = 128;   // positions per CTA, at least (the workspace is sized for it)
// Measured on 32k positions, 32 / 8 heads, d = 128: Q8_0 52.3 / 49.2 / 53.4 us
// at 128 / 192 / 256 positions, Q5_0 56.1 / 55.3 us and Q4_0 47.2 / 47.2 us at
// 192 / 256.
template <int T> constexpr int chunk_of() { return T == T_Q8_0 ? 192 : 256; }
constexpr int kWarps = 8;
constexpr int kMaxG = 8;       // query heads per kv head, at most

// Integer code (offset removed) of element e (0..31) of a 32-weight block
// (in shared memory).
template <int T>
__device__ __forceinline__ int code_at(const uint8_t* blk, int e) {
    if constexpr (T == T_Q8_0) {
        return (int)(int8_t)blk[2 + e];
    } else if constexpr (T == T_Q4_0) {
        return (int)((blk[2 + (e & 15)] >> (4 * (e >> 4))) & 15) - 8;
    } else {   // Q5_0: nibble plus bit e of the fifth-bit word
        const uint32_t lo = (blk[6 + (e & 15)] >> (4 * (e >> 4))) & 15;
        const uint32_t hb = (blk[2 + (e >> 3)] >> (e & 7)) & 1;
        return (int)(lo | (hb << 4)) - 16;
    }
}

// Bytes of one (t, g) row and its shared-memory slot: the aligned-down
// 16-byte window.  Rows start at multiples of ROWB from a 16-byte aligned
// cache, so a window starts at most 16 - gcd(ROWB, 16) bytes before its row.
// The 16 bytes past the last slot keep the word loads that read one word
// ahead inside the allocation.
template <int T, int NB, int CH> struct Rows {
    static constexpr int ROWB = NB * Fmt<T>::BB;
    static constexpr int ALIGN = (ROWB & 15) == 0 ? 16 : ((ROWB & 7) == 0 ? 8 : ((ROWB & 3) == 0 ? 4 : 2));
    static constexpr int SLOT = (ROWB + 16 - ALIGN + 15) / 16 * 16;
    static constexpr int NCH = SLOT / 16;   // 16-byte copies per row
    static constexpr int SMEM = 2 * CH * SLOT + 16;
};

// 16-byte cp.async that reads only the first n (1..16) bytes of src and
// zero-fills the rest of the destination.
__device__ __forceinline__ void cp_async_upto16(uint32_t sdst, const void* src, uint32_t n) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sdst), "l"(src), "r"(n) : "memory");
}

// Requests the chunk's rows of one cache (K or V) into `slots`.
template <int T, int NB, int CH>
__device__ __forceinline__ void stage_rows(uint8_t* slots, const uint8_t* C, int64_t t0, int nt, int n_kv, int g,
                                           int64_t total) {
    using R = Rows<T, NB, CH>;
    const uint32_t s0 = smem_u32(slots);
    for (int idx = threadIdx.x; idx < nt * R::NCH; idx += blockDim.x) {
        const int j = idx / R::NCH, k = idx - j * R::NCH;
        const int64_t a = (((t0 + j) * n_kv + g) * (int64_t)R::ROWB & ~(int64_t)15) + 16 * k;
        if (a < total) cp_async_upto16(s0 + (uint32_t)(j * R::SLOT + 16 * k), C + a, (uint32_t)min((int64_t)16, total - a));
    }
}

// A shared-memory word load at a 32-bit shared address (volatile: it stays
// after the copy waits and barriers that precede it).
__device__ __forceinline__ uint32_t sld32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// N words from a 2-byte aligned address in shared memory, for a lane whose
// address moves by multiples of 16 bytes from position to position: the
// aligned word address and the funnel shift are fixed once.  The word address
// is reached by pointer arithmetic, so plain loads stay shared-space loads;
// ASM issues them as explicit shared loads instead (measured faster for the
// nibble types, slower for Q8_0).
template <int N, bool ASM = false> struct Run {
    const uint8_t* a;
    uint32_t sh;
    __device__ __forceinline__ explicit Run(const uint8_t* p) {
        const uint32_t m = (uint32_t)reinterpret_cast<uintptr_t>(p) & 3u;
        a = p - m;
        sh = 8u * m;
    }
    __device__ __forceinline__ void load(uint32_t off, uint32_t (&w)[N]) const {
        if constexpr (ASM) {
            const uint32_t b = smem_u32(a) + off;
            uint32_t prev = sld32(b);
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const uint32_t next = sld32(b + 4u * (i + 1));
                w[i] = __funnelshift_r(prev, next, sh);
                prev = next;
            }
        } else {
            const uint32_t* q = reinterpret_cast<const uint32_t*>(a + off);
            uint32_t prev = q[0];
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const uint32_t next = q[i + 1];
                w[i] = __funnelshift_r(prev, next, sh);
                prev = next;
            }
        }
    }
};
__device__ __forceinline__ uint32_t lds16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// The codes of elements e0 .. e0 + 4W - 1 of a 32-weight block in shared
// memory at blk (+ the position's offset) as W words of bytes, the offset
// still in (Q4_0 and Q5_0 codes are 0..15 / 0..31).  The range never
// straddles element 16 unless it is the whole block.
template <int T, int W> struct Codes {
    static constexpr bool kWhole = T != T_Q8_0 && W == 8;   // the whole block of a nibble type
    static constexpr int QS = T == T_Q8_0 ? 2 : (T == T_Q5_0 ? 6 : 2);
    Run<kWhole ? 4 : W, T != T_Q8_0> run;
    Run<1, T != T_Q8_0> qh;
    uint32_t nsh;
    int e0;
    __device__ __forceinline__ Codes(const uint8_t* blk, int e0_)
        : run(kWhole || T == T_Q8_0 ? blk + QS + (kWhole ? 0 : e0_) : blk + QS + (e0_ & 15)),
          qh(blk + 2), nsh(e0_ >= 16 ? 4u : 0u), e0(e0_) {}
    __device__ __forceinline__ void load(uint32_t off, uint32_t (&cw)[W]) const {
        if constexpr (T == T_Q8_0) {
            run.load(off, cw);
        } else {
            if constexpr (kWhole) {
                uint32_t w[4];
                run.load(off, w);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cw[i] = w[i] & 0x0F0F0F0Fu;
                    cw[4 + i] = (w[i] >> 4) & 0x0F0F0F0Fu;
                }
            } else {
                uint32_t w[W];
                run.load(off, w);
#pragma unroll
                for (int i = 0; i < W; ++i) cw[i] = (w[i] >> nsh) & 0x0F0F0F0Fu;
            }
            if constexpr (T == T_Q5_0) {
                uint32_t h[1];
                qh.load(off, h);
#pragma unroll
                for (int i = 0; i < W; ++i) {
                    const uint32_t t = (h[0] >> (e0 + 4 * i)) & 15u;
                    cw[i] |= ((t * 0x00204081u) & 0x01010101u) << 4;
                }
            }
        }
    }
};

// The integer code held in the low byte of b, as Codes leaves it (offset
// still in for Q4_0 / Q5_0).
template <int T>
__device__ __forceinline__ int code_of_byte(uint32_t b) {
    if constexpr (T == T_Q8_0) return (int)(int8_t)(b & 255u);
    else return (int)(b & 255u) - (T == T_Q5_0 ? 16 : 8);
}

// A little-endian word at a 2-byte aligned shared address (the slot has
// slack past the row, so the second aligned word is always inside it).
__device__ __forceinline__ uint32_t ldw_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    return __funnelshift_r(w[0], w[1], (uint32_t)(a & 3) * 8u);
}

// Bits 0..3 of z moved to bit 4 of bytes 0..3 (the four products of the
// multiply land on distinct bits, so nothing carries).
__device__ __forceinline__ uint32_t bit4_spread(uint32_t z) { return ((z & 15u) * 0x02040810u) & 0x10101010u; }

// The score MMA's A fragments of one 32-weight block of one row (position):
// the codes minus the type's offset (Q8_0 none, Q5_0 16, Q4_0 8), exact in
// fp16.  Half s of the block (elements 16 s .. 16 s + 15) is one k16 step;
// thread tq takes elements 16 s + 4 tq + {0, 2} in a[2 s] (k slots 2 tq,
// 2 tq + 1) and 16 s + 4 tq + {1, 3} in a[2 s + 1] (slots 2 tq + 8, 2 tq + 9).
// A code sits in the mantissa of 1024 (or of 64 when it is a high nibble,
// one unit being 1/16 there) and one fp16 add removes that and the offset.
template <int T>
__device__ __forceinline__ void kcodes(const uint8_t* blk, int tq, uint32_t (&a)[4]) {
    using hm::and_or;
    using hm::and_xor;
    using hm::hadd2;
    if constexpr (T == T_Q8_0) {   // d, 32 signed bytes
        const uint32_t w0 = ldw_a2(blk + 2 + 4 * tq), w1 = ldw_a2(blk + 18 + 4 * tq);
        // 0x6480 ^ b = 1024 + 128 + (signed b); minus 1152.
        a[0] = hadd2(and_xor(w0, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[1] = hadd2(and_xor(w0 >> 8, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[2] = hadd2(and_xor(w1, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[3] = hadd2(and_xor(w1 >> 8, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
    } else if constexpr (T == T_Q4_0) {   // d, 16 bytes: low nibbles elements 0..15, high 16..31
        const uint32_t w = ldw_a2(blk + 2 + 4 * tq);
        a[0] = hadd2(and_or(w, 0x000F000Fu, 0x64006400u), 0xE408E408u);        // 1024 + q - 1032
        a[1] = hadd2(and_or(w >> 8, 0x000F000Fu, 0x64006400u), 0xE408E408u);
        a[2] = hadd2(and_or(w, 0x00F000F0u, 0x54005400u), 0xD480D480u);        // 64 + q - 72
        a[3] = hadd2(and_or(w >> 8, 0x00F000F0u, 0x54005400u), 0xD480D480u);
    } else {   // Q5_0: d, 32 fifth bits, 16 bytes of nibbles
        const uint32_t qh = ldw_a2(blk + 2), w = ldw_a2(blk + 6 + 4 * tq);
        const uint32_t v0 = (w & 0x0F0F0F0Fu) | bit4_spread(qh >> (4 * tq));
        const uint32_t v1 = ((w >> 4) & 0x0F0F0F0Fu) | bit4_spread(qh >> (16 + 4 * tq));
        a[0] = hadd2(and_or(v0, 0x00FF00FFu, 0x64006400u), 0xE410E410u);       // 1024 + q - 1040
        a[1] = hadd2(and_or(v0 >> 8, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
        a[2] = hadd2(and_or(v1, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
        a[3] = hadd2(and_or(v1 >> 8, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
    }
}

// kcodes for the streaming kernel, with the row's word addressing set up
// once.  The three block sizes (34, 18, 22 bytes) are 2 mod 4, so the words a
// thread reads (element 4 tq of block b, and its second half at + 16 for
// Q8_0) sit at one misalignment m in the even blocks and m ^ 2 in the odd
// ones, the same in every row of the CTA (slots are 16-byte multiples).
// KAddr holds, per parity, the aligned address of block 0's word and the
// funnel shift; block b adds b * BB (an immediate once b is unrolled).
struct KAddr {
    const uint8_t* base[2];   // aligned word address of the element-4tq word of block 0 (even) / block 1 less BB (odd)
    uint32_t sh[2];           // funnel shifts, bits
    int qh;                   // Q5_0: offset of the fifth-bit word from the same aligned base
    int tq;                   // the thread's group of the MMA layout
};
template <int T>
__device__ __forceinline__ KAddr kaddr(const uint8_t* row, int tq) {
    constexpr int BB = Fmt<T>::BB;
    const int hdr = T == T_Q5_0 ? 6 : 2;   // first code byte
    const uint8_t* p = row + hdr + 4 * tq;
    const int m = (int)(reinterpret_cast<uintptr_t>(p) & 3);   // 0 or 2
    KAddr k;
    k.base[0] = p - m;
    k.base[1] = p + BB - (m ^ 2) - BB;   // block 1's word, less BB
    k.sh[0] = 8u * (uint32_t)m;
    k.sh[1] = 8u * (uint32_t)(m ^ 2);
    k.qh = -4 - 4 * tq;                   // Q5_0: the word at byte 2 has the same misalignment
    k.tq = tq;
    return k;
}
__device__ __forceinline__ uint32_t kword(const KAddr& k, int par, int off) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(k.base[par] + off);
    return __funnelshift_r(w[0], w[1], k.sh[par]);
}
template <int T>
__device__ __forceinline__ void kcodes_at(const KAddr& k, int b, uint32_t (&a)[4]) {
    using hm::and_or;
    using hm::and_xor;
    using hm::hadd2;
    constexpr int BB = Fmt<T>::BB;
    const int par = b & 1, o = BB * b;
    if constexpr (T == T_Q8_0) {
        const uint32_t w0 = kword(k, par, o), w1 = kword(k, par, o + 16);
        a[0] = hadd2(and_xor(w0, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[1] = hadd2(and_xor(w0 >> 8, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[2] = hadd2(and_xor(w1, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
        a[3] = hadd2(and_xor(w1 >> 8, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
    } else if constexpr (T == T_Q4_0) {
        const uint32_t w = kword(k, par, o);
        a[0] = hadd2(and_or(w, 0x000F000Fu, 0x64006400u), 0xE408E408u);
        a[1] = hadd2(and_or(w >> 8, 0x000F000Fu, 0x64006400u), 0xE408E408u);
        a[2] = hadd2(and_or(w, 0x00F000F0u, 0x54005400u), 0xD480D480u);
        a[3] = hadd2(and_or(w >> 8, 0x00F000F0u, 0x54005400u), 0xD480D480u);
    } else {
        const uint32_t qh = kword(k, par, o + k.qh), w = kword(k, par, o);
        const uint32_t v0 = (w & 0x0F0F0F0Fu) | bit4_spread(qh >> (4 * k.tq));
        const uint32_t v1 = ((w >> 4) & 0x0F0F0F0Fu) | bit4_spread(qh >> (16 + 4 * k.tq));
        a[0] = hadd2(and_or(v0, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
        a[1] = hadd2(and_or(v0 >> 8, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
        a[2] = hadd2(and_or(v1, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
        a[3] = hadd2(and_or(v1 >> 8, 0x00FF00FFu, 0x64006400u), 0xE410E410u);
    }
}

// B fragments of the group's queries (sq: [heads][D] fp32) and the scale of
// each (head, 32-block).  Per block, x' = q 2^-e with e = max(0,
// floor(log2 max|q|) - 14), so |x'| < 2^15 fits fp16; hi = fp16(x'), lo =
// fp16(x' - hi) keep about 22 significant bits of every element, whatever
// the block's largest element is.  Column gq of n-tile n is head
// 4 n + gq / 2, term gq % 2 (hi, lo); zero for heads >= G.  Thread (gq, tq)
// holds elements 32 b + 16 s + 4 tq + {0, 2} / {1, 3} of half s, the order
// of kcodes.  The four threads of a quad hold the whole block, so its
// maximum is two shuffles.  sup[h][b] = 2^e (1 for h >= G).
template <int NB, int NT>
__device__ __forceinline__ void prep_query(const float* sq, int D, int G, int gq, int tq,
                                           uint32_t (&bq)[NB][2][NT][2], float* sup) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int h = 4 * n + (gq >> 1);
        const bool live = h < G;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float v[2][4];
            float amax = 0.0f;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                float4 u = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (live) u = *reinterpret_cast<const float4*>(sq + h * D + 32 * b + 16 * s + 4 * tq);
                v[s][0] = u.x; v[s][1] = u.y; v[s][2] = u.z; v[s][3] = u.w;
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(v[s][k]));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int e = max(0, (int)((__float_as_uint(amax) >> 23) & 255u) - 127 - 14);
            const float down = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                uint32_t hv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float x = v[s][k] * down;
                    const __half hi = __float2half_rn(x);
                    hv[k] = (gq & 1) ? __half_as_ushort(__float2half_rn(x - __half2float(hi))) : __half_as_ushort(hi);
                }
                bq[b][s][n][0] = hv[0] | (hv[2] << 16);
                bq[b][s][n][1] = hv[1] | (hv[3] << 16);
            }
            if (tq == 0 && (gq & 1) == 0) sup[h * NB + b] = live ? __uint_as_float((uint32_t)(127 + e) << 23) : 1.0f;
        }
    }
}

template <int T, int NB, int GT, int CH>   // NB = d / 32; GT = heads per kv head when fixed, 0 when not; CH = chunk
__global__ void __launch_bounds__(kWarps * 32) attn_chunk_kernel(const float* __restrict__ q, const uint8_t* __restrict__ K,
                                                                const uint8_t* __restrict__ V, int64_t T_len, int n_heads,
                                                                int n_kv, float scale, float* __restrict__ ws) {
    using R = Rows<T, NB, CH>;
    constexpr int D = 32 * NB, BB = Fmt<T>::BB;
    constexpr int GG = GT > 0 ? GT : kMaxG;      // heads per kv head, at most
    constexpr int64_t ROWB = R::ROWB;            // bytes of one (t, g) row: d / 32 blocks
    extern __shared__ __align__(16) uint8_t dyn[];
    uint8_t* sK = dyn;                           // [CH][SLOT] row windows
    uint8_t* sV = dyn + CH * R::SLOT;
    __shared__ __align__(16) float sq[GG][D];    // the group's queries
    __shared__ __align__(16) float ss[CH][GG];   // scores, then e^(s - m), per position
    __shared__ float sred[2][GG];
    __shared__ float sup[4 * ((2 * GG + 7) / 8)][NB];   // 2^e of each head's query blocks
    const int g = (int)(blockIdx.x % (unsigned)n_kv), c = (int)(blockIdx.x / (unsigned)n_kv), G = n_heads / n_kv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)c * CH;
    const int nt = (int)min((int64_t)CH, T_len - t0);
    const int64_t total = T_len * n_kv * ROWB;   // bytes of each cache
    // Where a row starts in its slot: the same for all of a warp's positions
    // (they are 8 apart and rows are an even number of bytes, so 8 rows span
    // a multiple of 16 bytes).
    const int mis = (int)((((t0 + warp) * n_kv + g) * ROWB) & 15);
    constexpr int STEP = kWarps * R::SLOT;       // slot bytes between a warp's positions
    pdl_wait_prior();
    stage_rows<T, NB, CH>(sK, K, t0, nt, n_kv, g, total);
    cp_async_commit();
    stage_rows<T, NB, CH>(sV, V, t0, nt, n_kv, g, total);
    cp_async_commit();
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) sq[i / D][i % D] = q[(int64_t)(g * G + i / D) * D + i % D];
    __syncthreads();
    // Lane l: elements e0 .. e0 + NB - 1 of block eb (pass 2).
    const int e0 = (lane * NB) & 31, eb = (lane * NB) >> 5;
    // Pass 1 on the fp16 warp MMA.  A tile is 16 positions; thread (gq, tq)
    // of the MMA layout (gq = lane / 4, tq = lane % 4) decodes rows gq and
    // gq + 8 (positions) and holds the B column gq: head 4 nt + gq / 2, term
    // gq % 2 of the query (hi, lo) in n-tile nt.
    constexpr int NT = (2 * GG + 7) / 8;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t bq[NB][2][NT][2];
    prep_query<NB, NT>(&sq[0][0], D, G, gq, tq, bq, &sup[0][0]);
    cp_async_wait<1>();   // this thread's K copies
    __syncthreads();      // ... and everyone's (and the query scales)
    float upr[NT][NB];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int b = 0; b < NB; ++b) upr[n][b] = sup[4 * n + tq][b];
    {
        // Where row gq starts in its slot: the same in every tile (16 rows
        // span 16 n_kv ROWB bytes, a multiple of 16) and for row gq + 8.
        const int misq = (int)((((t0 + gq) * n_kv + g) * ROWB) & 15);
        const int ntiles = (nt + 15) >> 4;
        for (int tile = warp; tile < ntiles; tile += kWarps) {
            const int j0 = 16 * tile + gq;
            const uint8_t* r0 = sK + j0 * R::SLOT + misq;
            const uint8_t* r1 = r0 + 8 * R::SLOT;
            float s0[NT], s1[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) s0[n] = s1[n] = 0.0f;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                uint32_t a0[4], a1[4];
                kcodes<T>(r0 + b * BB, tq, a0);
                kcodes<T>(r1 + b * BB, tq, a1);
                const float d0 = h2f(lds16(r0 + b * BB)), d1 = h2f(lds16(r1 + b * BB));
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    hm::mma16816(c, a0[0], a1[0], a0[1], a1[1], bq[b][0][n][0], bq[b][0][n][1]);
                    hm::mma16816(c, a0[2], a1[2], a0[3], a1[3], bq[b][1][n][0], bq[b][1][n][1]);
                    s0[n] = fmaf(d0 * upr[n][b], c[0] + c[1], s0[n]);
                    s1[n] = fmaf(d1 * upr[n][b], c[2] + c[3], s1[n]);
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int h = 4 * n + tq;
                if (h < G) {
                    if (j0 < nt) ss[j0][h] = scale * s0[n];
                    if (j0 + 8 < nt) ss[j0 + 8][h] = scale * s1[n];
                }
            }
        }
    }
    __syncthreads();
    // Chunk statistics per head: m = max s, then e^(s - m) and their sum.
    for (int h = warp; h < G; h += kWarps) {
        float m = -__int_as_float(0x7f800000);
        for (int j = lane; j < nt; j += 32) m = fmaxf(m, ss[j][h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
        for (int j = lane; j < nt; j += 32) {
            const float e = expf(ss[j][h] - m);
            ss[j][h] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sred[0][h] = m;
            sred[1][h] = l;
        }
    }
    __syncthreads();
    cp_async_wait<0>();
    __syncthreads();
    // Pass 2: sum_t e^(s_t - m) V[t, g], this warp's positions.
    float acc[GG][NB];
#pragma unroll
    for (int h = 0; h < GG; ++h)
#pragma unroll
        for (int k = 0; k < NB; ++k) acc[h][k] = 0.0f;
    const uint8_t* vblk = sV + warp * R::SLOT + mis + eb * BB;
    const Codes<T, (NB >= 4 ? NB / 4 : 1)> vc(vblk, e0);
    uint32_t voff = 0;
    for (int j = warp; j < nt; j += kWarps, vblk += STEP, voff += STEP) {
        const float dv = h2f(lds16(vblk));
        float vv[NB];
        if constexpr (NB >= 4) {   // the lane's codes as words (they lie in one half of the block)
            uint32_t cw[NB / 4];
            vc.load(voff, cw);
#pragma unroll
            for (int k = 0; k < NB; ++k) vv[k] = dv * (float)code_of_byte<T>(cw[k >> 2] >> (8 * (k & 3)));
        } else {
#pragma unroll
            for (int k = 0; k < NB; ++k) vv[k] = dv * (float)code_at<T>(vblk, e0 + k);
        }
        float p[GG];
        if constexpr (GT > 0 && GT % 4 == 0) {
#pragma unroll
            for (int h = 0; h < GG; h += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(&ss[j][h]);
                p[h] = q4.x; p[h + 1] = q4.y; p[h + 2] = q4.z; p[h + 3] = q4.w;
            }
        } else {
#pragma unroll
            for (int h = 0; h < GG; ++h) p[h] = (GT > 0 || h < G) ? ss[j][h] : 0.0f;
        }
#pragma unroll
        for (int h = 0; h < GG; ++h) {
            if (GT == 0 && h >= G) break;
#pragma unroll
            for (int k = 0; k < NB; ++k) acc[h][k] = fmaf(p[h], vv[k], acc[h][k]);
        }
    }
    // The warps' partial sums go to the row slots (no longer needed), then
    // every output element adds them in warp order.
    static_assert(kWarps * GG * D * 4 <= 2 * CH * R::SLOT, "the partial sums fit in the row slots");
    float* part = reinterpret_cast<float*>(dyn);   // [kWarps][GG][D]
    __syncthreads();   // every warp is done with the slots
#pragma unroll
    for (int h = 0; h < GG; ++h)
#pragma unroll
        for (int k = 0; k < NB; ++k)
            if (h < G) part[(warp * GG + h) * D + lane * NB + k] = acc[h][k];
    __syncthreads();
    // Chunk partial (m, l, o[d]) per head.
    const int nchunks = (int)(gridDim.x / (unsigned)n_kv);
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D, e = i % D;
        float o = part[h * D + e];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) o += part[(w * GG + h) * D + e];
        float* dst = ws + ((int64_t)(g * G + h) * nchunks + c) * (D + 2);
        dst[2 + e] = o;
        if (e == 0) {
            dst[0] = sred[0][h];
            dst[1] = sred[1][h];
        }
    }
}

// ---------------------------------------------------------------------------
// Streaming kernel.  CTA (g, c) takes kv head g and positions [c P, c P + P)
// (P a multiple of the stage), so the query preparation, the final merge
// and the partial written per CTA are paid once per ~P positions.  A
// producer thread streams each stage (128 positions) of the K and of the V
// rows into a ring as one 2D TMA box each: the cache seen as [T, n_kv ROWB]
// bytes, the box the 16-byte aligned window of head g's rows (the same
// offset in every position) x 128 positions; positions past T arrive as
// zeros.  One copy request per stage instead of one per row keeps the copy
// engine off the critical path (a bulk copy costs a fixed few tens of
// cycles, more than a 144-byte row takes to stream).  Consumer warp w takes
// positions 16 w .. 16 w + 15 of every stage and keeps its own running
// softmax (max and sum per head, flash-attention style): scores of its tile
// on the MMA as in the chunk kernel, then p = e^(s - m) rescales and feeds
// its fp32 sums of p V (lane l owns d/32 elements of V for every head).  At
// the end the eight warps' (m, l, o) are merged in warp order: the result
// does not depend on timing.  For Q8_0 and Q4_0 with d = 128 and up to four
// query heads per kv head, p V runs on the MMA too (the kMmaV form below): the
// warps share each stage's softmax reference, and warp w sums one V block
// over half the stage's positions.
constexpr int kSW = 8;                      // consumer warps
constexpr int kSThreads = (kSW + 1) * 32;   // + the producer warp
constexpr int kSPos = 16 * kSW;             // positions per stage
constexpr int kSMaxStages = 6;
constexpr int kSBudget = 112 * 1024;        // shared memory per CTA (two CTAs per SM)

template <int T, int NB> struct SGeo {
    static constexpr int ROWB = NB * Fmt<T>::BB;
    // Head g's rows start g ROWB bytes into a position's n_kv ROWB bytes, at
    // most 16 - gcd(ROWB, 16) bytes past a 16-byte boundary; the box (SLOT
    // bytes wide, at most 256) covers that window, rounded up to 16 bytes.
    static constexpr int ALIGN = (ROWB & 15) == 0 ? 16 : ((ROWB & 7) == 0 ? 8 : ((ROWB & 3) == 0 ? 4 : 2));
    static constexpr int SLOT = (ROWB + 16 - ALIGN + 15) / 16 * 16;
    static constexpr int HALF = kSPos * SLOT;   // the K (or V) rows of a stage
    static constexpr int STAGE = 2 * HALF;
    static_assert(HALF % 128 == 0, "stages and halves start 128-byte aligned");
};

// Shared-memory map of the streaming kernel: ring (+16 bytes for word reads
// past the last row), queries [G][D], p [warp][16][G], rescale factors
// [warp][G], mbarriers and the abort word.  With the p V pass on the MMA
// (kMmaV: Q8_0 or Q4_0, d = 128, up to four query heads per kv head) the query area
// is reused, once the queries are in registers, for a stage's B fragments
// [4 blocks][8 position tiles][36 lane slots][2 words] (lanes 16..31 four
// slots on, so that a warp's 16-bit fragment stores meet distinct banks)
// and the warps' tile maxima
// [kSW][8] (four heads' scores, the V scales' magnitude), and there is no p
// or rescale area.
template <int T, int NB, int G> struct SMap {
    static constexpr int D = 32 * NB;
    static constexpr bool kMmaV = (T == T_Q8_0 || T == T_Q4_0) && NB == 4 && G <= 4;
    static constexpr int kBFrag = 4 * kSW * 36 * 2 * 4;   // B fragment bytes of a stage
    static constexpr int QB = kMmaV ? kBFrag + kSW * 8 * 4 : G * D * 4;
    static_assert(!kMmaV || QB >= G * D * 4, "the query area holds the queries first");
    __host__ __device__ static constexpr int off_q(int nstg) { return nstg * SGeo<T, NB>::STAGE + 16; }
    __host__ __device__ static constexpr int off_p(int nstg) { return off_q(nstg) + QB; }
    __host__ __device__ static constexpr int off_a(int nstg) { return off_p(nstg) + (kMmaV ? 0 : kSW * 16 * G * 4); }
    __host__ __device__ static constexpr int off_bar(int nstg) { return (off_a(nstg) + (kMmaV ? 0 : kSW * G * 4) + 7) / 8 * 8; }
    // + 128 bytes to align the ring.
    __host__ __device__ static constexpr int bytes(int nstg) { return off_bar(nstg) + 2 * kSMaxStages * 8 + 16 + 128; }
};

__device__ __forceinline__ void named_sync_stream_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSW * 32) : "memory");
}

template <int T, int NB, int G>   // NB = d / 32; G = query heads per kv head
__global__ void __launch_bounds__(kSThreads, 2) attn_stream_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                  const __grid_constant__ CUtensorMap vmap,
                                                                  const float* __restrict__ q, int64_t T_len, int n_kv,
                                                                  float scale, float* __restrict__ ws, int P,
                                                                  int nsplit, int nstg, unsigned* status) {
    using Gm = SGeo<T, NB>;
    using Mp = SMap<T, NB, G>;
    constexpr int D = 32 * NB, BB = Fmt<T>::BB;
    constexpr int NT = (2 * G + 7) / 8;
    constexpr int64_t ROWB = Gm::ROWB;
    extern __shared__ __align__(16) uint8_t dyn[];
    // The TMA boxes land at 128-byte aligned addresses (stages and halves
    // are multiples of 128 bytes; the launch adds 128 bytes of room).
    uint8_t* base = dyn + ((128u - (smem_u32(dyn) & 127u)) & 127u);
    uint8_t* ring = base;
    float* sq = reinterpret_cast<float*>(base + Mp::off_q(nstg));
    float* sp = reinterpret_cast<float*>(base + Mp::off_p(nstg));
    float* sa = reinterpret_cast<float*>(base + Mp::off_a(nstg));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + Mp::off_bar(nstg));
    uint64_t* empty = full + kSMaxStages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + kSMaxStages);
    __shared__ float sup[4 * NT][NB];   // 2^e of each head's query blocks

    const int g = (int)(blockIdx.x % (unsigned)n_kv), c = (int)(blockIdx.x / (unsigned)n_kv);
    const int64_t p0 = (int64_t)c * P, p1 = min(T_len, p0 + P);
    const int nst = (int)((p1 - p0 + kSPos - 1) / kSPos);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int xg = (int)(((int64_t)g * ROWB) & ~(int64_t)15);   // box start in a position's bytes
    const int misg = (int)(((int64_t)g * ROWB) & 15);             // where head g's row starts in the box
    if (threadIdx.x == 0) {
        for (int i = 0; i < nstg; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kSW);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait_prior();   // the cache and the query may come from the previous kernel

    if (warp == kSW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int slot = 0, issued = 0;
            uint32_t ph = 0;
            for (int st = 0; st < nst; ++st) {
                if (st >= nstg && !mbar_wait_abortable(&empty[slot], ph ^ 1u, status, abort)) break;
                uint8_t* dst = ring + slot * Gm::STAGE;
                const int y = (int)(p0 + (int64_t)st * kSPos);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)Gm::STAGE);
                tc::tma_load_2d(dst, &kmap, xg, y, &full[slot]);
                tc::tma_load_2d(dst + Gm::HALF, &vmap, xg, y, &full[slot]);
                ++issued;
                if (++slot == nstg) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            // Every copy requested lands before the CTA may exit.
            for (int k = max(0, issued - nstg); k < issued; ++k)
                mbar_wait_bounded(&full[k % nstg], (uint32_t)(k / nstg) & 1u, status);
        }
        return;
    }

    // ---------------- consumers ----------------
    const int tid = threadIdx.x;
    for (int i = tid; i < G * D; i += kSW * 32) sq[i] = q[(int64_t)g * G * D + i];
    named_sync_stream_consumers();
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t bq[NB][2][NT][2];
    prep_query<NB, NT>(sq, D, G, gq, tq, bq, &sup[0][0]);
    named_sync_stream_consumers();
    float upr[NT][NB];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int b = 0; b < NB; ++b) upr[n][b] = sup[4 * n + tq][b];
    if constexpr (Mp::kMmaV) {
        // p V on the fp16 MMA.  Per stage:
        //  1. warp w scores its positions 16 w .. 16 w + 15 (as below);
        //  2. the warps' tile maxima give the stage's maximum per head, the
        //     same in every warp, so all warps' p share one reference;
        //  3. thread (gq, tq) writes x = p d 2^E (d: the position's V block
        //     scale) of its positions gq, gq + 8 and head tq for each V block,
        //     as two fp16 terms hi = fp16(x), lo = fp16(x - hi), into the
        //     stage's B fragments (k = position in the tile, column 2 h + term).
        //     2^E brings the stage's largest |d| into [2^14, 2^15), so x stays
        //     below the fp16 maximum and out of its subnormal range, where
        //     hi + lo would keep fewer than 22 bits; the sums are rescaled when
        //     E changes and divided by 2^E at the end;
        //  4. warp w takes V block b = w & 3 as two 16-element MMA tiles
        //     (rows g and g + 8 of tile j: elements 32 b + 4 g + 2 j and
        //     32 b + 4 g + 2 j + 1) over position tiles 4 (w >> 2) .. + 3,
        //     A = the codes transposed by byte permutes (exact in fp16; a
        //     Q4_0 lane takes the low nibbles of bytes 4 g .. 4 g + 3 for
        //     g < 4, the high nibbles of the same bytes for g >= 4),
        //     accumulating in the MMA; an element's output is the sum of its
        //     hi and lo columns.
        // Warps w and w + 4 hold the same elements over different positions
        // and are added at the end, as are the threads' softmax sums.
        const float kNegInf = -__int_as_float(0x7f800000);
        uint32_t* bfr = reinterpret_cast<uint32_t*>(base + Mp::off_q(nstg));
        uint16_t* bfh = reinterpret_cast<uint16_t*>(bfr);
        float* tmx = reinterpret_cast<float*>(base + Mp::off_q(nstg) + Mp::kBFrag);   // [kSW][8]
        const int vb = warp & 3, pt0 = 4 * (warp >> 2);
        // This thread's four codes of a V row (Q4_0: lanes gq and gq + 4 read
        // the same bytes, low and high nibbles).
        const int voff = misg + vb * BB + 2 + 4 * (T == T_Q4_0 ? (gq & 3) : gq);
        // Code pairs to exact fp16 integers: (bytes & mask) | magic, then
        // minus the magic and the type's offset.
        const bool hin = T == T_Q4_0 && gq >= 4;
        const uint32_t cmask = T == T_Q8_0 ? 0x00FF00FFu : (hin ? 0x00F000F0u : 0x000F000Fu);
        const uint32_t cmag = T == T_Q8_0 ? 0x64806480u : (hin ? 0x54005400u : 0x64006400u);
        const uint32_t cneg = T == T_Q8_0 ? 0xE480E480u : (hin ? 0xD480D480u : 0xE408E408u);
        const bool hv = tq < G;
        float m_run = kNegInf, l_part = 0.0f;
        float cv[2][4] = {};
        int e_run = 0;   // the sums cv are in units of 2^-e_run
        int slot = 0;
        uint32_t ph = 0;
        bool dead = false;
        for (int st = 0; st < nst; ++st) {
            if (!dead && !mbar_wait_abortable(&full[slot], ph, status, abort)) dead = true;
            const int jt = 16 * warp;
            const int64_t sp0 = p0 + (int64_t)st * kSPos;
            const int nvalid = (int)max((int64_t)0, min((int64_t)16, p1 - sp0 - jt));
            const int svalid = (int)min((int64_t)kSPos, p1 - sp0);   // valid positions of the stage
            const uint8_t* kst = ring + slot * Gm::STAGE;
            const uint8_t* vst = kst + Gm::HALF;
            const bool v0 = gq < nvalid, v1 = gq + 8 < nvalid;
            float s0 = kNegInf, s1 = kNegInf;
            if (!dead && nvalid > 0) {
                const uint8_t* r0 = kst + (jt + gq) * Gm::SLOT + misg;
                const uint8_t* r1 = r0 + 8 * Gm::SLOT;
                const KAddr k0 = kaddr<T>(r0, tq), k1 = kaddr<T>(r1, tq);
                float a0s = 0.0f, a1s = 0.0f;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    uint32_t a0[4], a1[4];
                    kcodes_at<T>(k0, b, a0);
                    kcodes_at<T>(k1, b, a1);
                    const float d0 = h2f(lds16(r0 + b * BB)), d1 = h2f(lds16(r1 + b * BB));
                    float cc[4];
                    hm::mma16816_z(cc, a0[0], a1[0], a0[1], a1[1], bq[b][0][0][0], bq[b][0][0][1]);
                    hm::mma16816(cc, a0[2], a1[2], a0[3], a1[3], bq[b][1][0][0], bq[b][1][0][1]);
                    a0s = fmaf(d0 * upr[0][b], cc[0] + cc[1], a0s);
                    a1s = fmaf(d1 * upr[0][b], cc[2] + cc[3], a1s);
                }
                if (v0) s0 = scale * a0s;
                if (v1) s1 = scale * a1s;
            }
            float mt = fmaxf(s0, s1);
            // The largest |d| of V among the tile's rows (thread tq: block tq).
            float dmx = fmaxf(fabsf(h2f(lds16(vst + (jt + gq) * Gm::SLOT + misg + tq * BB))),
                              fabsf(h2f(lds16(vst + (jt + gq + 8) * Gm::SLOT + misg + tq * BB))));
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) dmx = fmaxf(dmx, __shfl_xor_sync(0xffffffffu, dmx, o));
            if (gq == 0) tmx[warp * 8 + tq] = mt;
            if (lane == 0) tmx[warp * 8 + 4] = dmx;
            named_sync_stream_consumers();
            float ms = tmx[tq], dm = tmx[4];
#pragma unroll
            for (int w = 1; w < kSW; ++w) {
                ms = fmaxf(ms, tmx[w * 8 + tq]);
                dm = fmaxf(dm, tmx[w * 8 + 4]);
            }
            const float mnew = fmaxf(m_run, ms);   // finite: the stage has a valid position
            // 2^E with 2^14 <= dm 2^E < 2^15 (an all-zero stage keeps E).
            const int e_st = dm > 0.0f ? 141 - (int)((__float_as_uint(dm) >> 23) & 255u) : e_run;
            const float dsc = __uint_as_float((uint32_t)(127 + e_st) << 23);
            const float alpha = expf(m_run - mnew);
            const float calpha = alpha * __uint_as_float((uint32_t)(127 + e_st - e_run) << 23);   // x 2^(E - E_old)
            m_run = mnew;
            e_run = e_st;
            const float pa = v0 ? expf(s0 - mnew) : 0.0f, pb = v1 ? expf(s1 - mnew) : 0.0f;
            l_part = fmaf(l_part, alpha, pa + pb);
            {
                // (k = gq, column n) is half gq & 1 of word 0 of lane 4 n + gq / 2,
                // k = gq + 8 the same half of word 1; columns 2 tq (hi) and
                // 2 tq + 1 (lo) are lanes 8 tq + gq / 2 and 8 tq + 4 + gq / 2
                // (lane l in slot l + 4 (l >> 4)).
                const uint8_t* rv0 = vst + (jt + gq) * Gm::SLOT + misg;
                const uint8_t* rv1 = rv0 + 8 * Gm::SLOT;
                const bool w0 = hv && v0 && !dead, w1 = hv && v1 && !dead;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float x0 = w0 ? pa * (h2f(lds16(rv0 + b * BB)) * dsc) : 0.0f;
                    const float x1 = w1 ? pb * (h2f(lds16(rv1 + b * BB)) * dsc) : 0.0f;
                    const __half2 hi = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(hi);
                    const __half2 lo = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
                    uint16_t* q0 = bfh + (((b * kSW + warp) * 36 + 8 * tq + 4 * (tq >> 1) + (gq >> 1)) * 2) * 2 + (gq & 1);
                    q0[0] = __half_as_ushort(__low2half(hi));    // hi, k = gq
                    q0[2] = __half_as_ushort(__high2half(hi));   // hi, k = gq + 8
                    q0[16] = __half_as_ushort(__low2half(lo));   // lo (4 lanes on), k = gq
                    q0[18] = __half_as_ushort(__high2half(lo));  // lo, k = gq + 8
                }
            }
            named_sync_stream_consumers();
            if (!dead) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) cv[j][k] *= calpha;   // columns 2 tq, 2 tq + 1: head tq
                const uint8_t* vr = vst + (pt0 * 16 + 2 * tq) * Gm::SLOT + voff;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (16 * (pt0 + i) >= svalid) break;
                    const uint8_t* vi = vr + i * 16 * Gm::SLOT;
                    // Elements 4 gq .. 4 gq + 3 at positions 2 tq, 2 tq + 1, 2 tq + 8,
                    // 2 tq + 9 of the tile (odd blocks' codes are 4-byte aligned).
                    uint32_t cw4[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint8_t* a = vi + ((r & 1) + 8 * (r >> 1)) * Gm::SLOT;
                        cw4[r] = (vb & 1) ? *reinterpret_cast<const uint32_t*>(a) : (lds16(a) | (lds16(a + 2) << 16));
                    }
                    const uint2 bf = *reinterpret_cast<const uint2*>(bfr + ((vb * kSW + pt0 + i) * 36 + lane + 4 * (lane >> 4)) * 2);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        // Elements 2 j, 2 j + 1 of positions k, k + 1 as bytes [e@k, e'@k, e@k+1, e'@k+1].
                        const uint32_t sel = j ? 0x7632u : 0x5410u;
                        const uint32_t zl = __byte_perm(cw4[0], cw4[1], sel), zh = __byte_perm(cw4[2], cw4[3], sel);
                        // Q8_0: 0x6480 ^ b = 1024 + 128 + (signed b), minus 1152.  Q4_0:
                        // 1024 + q (low nibble) or 64 + q (high nibble, unit 1/16
                        // there), minus that and 8.
                        uint32_t a0, a1, a2, a3;
                        if constexpr (T == T_Q8_0) {
                            a0 = hm::hadd2(hm::and_xor(zl, cmask, cmag), cneg);
                            a1 = hm::hadd2(hm::and_xor(zl >> 8, cmask, cmag), cneg);
                            a2 = hm::hadd2(hm::and_xor(zh, cmask, cmag), cneg);
                            a3 = hm::hadd2(hm::and_xor(zh >> 8, cmask, cmag), cneg);
                        } else {
                            a0 = hm::hadd2(hm::and_or(zl, cmask, cmag), cneg);
                            a1 = hm::hadd2(hm::and_or(zl >> 8, cmask, cmag), cneg);
                            a2 = hm::hadd2(hm::and_or(zh, cmask, cmag), cneg);
                            a3 = hm::hadd2(hm::and_or(zh >> 8, cmask, cmag), cneg);
                        }
                        hm::mma16816(cv[j], a0, a1, a2, a3, bf.x, bf.y);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == nstg) {
                slot = 0;
                ph ^= 1u;
            }
        }
        // Softmax sums: the lanes of a head, then the warps in order; o: warps
        // w and w + 4 in that order.
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, o);
        named_sync_stream_consumers();   // the ring is free
        float* og = reinterpret_cast<float*>(ring);   // [G][D] o, [kSW][4] l, [4] m
        float* lw = og + G * D;
        float* mw = lw + kSW * 4;
        if (gq == 0) {
            lw[warp * 4 + tq] = l_part;
            if (warp == 0) mw[tq] = m_run;
        }
        float* oh = og + tq * D + 32 * vb + 4 * gq;
        const float unscale = __uint_as_float((uint32_t)(127 - e_run) << 23);   // 2^-E
        if (warp < 4 && hv) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                oh[2 * j] = (cv[j][0] + cv[j][1]) * unscale;
                oh[2 * j + 1] = (cv[j][2] + cv[j][3]) * unscale;
            }
        }
        named_sync_stream_consumers();
        if (warp >= 4 && hv) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                oh[2 * j] += (cv[j][0] + cv[j][1]) * unscale;
                oh[2 * j + 1] += (cv[j][2] + cv[j][3]) * unscale;
            }
        }
        named_sync_stream_consumers();
        if (*abort) return;
        for (int i = tid; i < G * D; i += kSW * 32) {
            const int h = i / D, e = i - h * D;
            float* dst = ws + ((int64_t)(g * G + h) * nsplit + c) * (D + 2);
            dst[2 + e] = og[i];
            if (e == 0) {
                float L = 0.0f;
#pragma unroll
                for (int w = 0; w < kSW; ++w) L += lw[w * 4 + h];
                dst[0] = mw[h];
                dst[1] = L;
            }
        }
    } else {
        const int e0 = (lane * NB) & 31, eb = (lane * NB) >> 5;   // this lane's elements of V
        const float kNegInf = -__int_as_float(0x7f800000);
        float m_run[NT], l_part[NT];
    #pragma unroll
        for (int n = 0; n < NT; ++n) {
            m_run[n] = kNegInf;
            l_part[n] = 0.0f;
        }
        // Sums of p V: heads in pairs (packed fp32 FMAs), this lane's elements.
        constexpr int GP = (G + 1) / 2;
        float2 acc[GP][NB];
    #pragma unroll
        for (int h = 0; h < GP; ++h)
    #pragma unroll
            for (int k = 0; k < NB; ++k) acc[h][k] = make_float2(0.0f, 0.0f);
        float* spw = sp + warp * 16 * G;
        float* saw = sa + warp * G;
        int slot = 0;
        uint32_t ph = 0;
        bool dead = false;
        for (int st = 0; st < nst; ++st) {
            if (!dead && !mbar_wait_abortable(&full[slot], ph, status, abort)) dead = true;
            const int jt = 16 * warp;
            const int64_t tp0 = p0 + (int64_t)st * kSPos + jt;
            const int nvalid = (int)max((int64_t)0, min((int64_t)16, p1 - tp0));
            if (!dead && nvalid > 0) {
                const uint8_t* kst = ring + slot * Gm::STAGE;
                const uint8_t* vst = kst + Gm::HALF;
                // Scores of positions gq and gq + 8 of the tile.
                const uint8_t* r0 = kst + (jt + gq) * Gm::SLOT + misg;
                const uint8_t* r1 = r0 + 8 * Gm::SLOT;
                const KAddr k0 = kaddr<T>(r0, tq), k1 = kaddr<T>(r1, tq);
                float s0[NT], s1[NT];
    #pragma unroll
                for (int n = 0; n < NT; ++n) s0[n] = s1[n] = 0.0f;
    #pragma unroll
                for (int b = 0; b < NB; ++b) {
                    uint32_t a0[4], a1[4];
                    kcodes_at<T>(k0, b, a0);
                    kcodes_at<T>(k1, b, a1);
                    const float d0 = h2f(lds16(r0 + b * BB)), d1 = h2f(lds16(r1 + b * BB));
    #pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        float cc[4];
                        hm::mma16816_z(cc, a0[0], a1[0], a0[1], a1[1], bq[b][0][n][0], bq[b][0][n][1]);
                        hm::mma16816(cc, a0[2], a1[2], a0[3], a1[3], bq[b][1][n][0], bq[b][1][n][1]);
                        s0[n] = fmaf(d0 * upr[n][b], cc[0] + cc[1], s0[n]);
                        s1[n] = fmaf(d1 * upr[n][b], cc[2] + cc[3], s1[n]);
                    }
                }
                // Running softmax of head 4 n + tq over this warp's positions.
                const bool v0 = gq < nvalid, v1 = gq + 8 < nvalid;
    #pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float a0 = v0 ? scale * s0[n] : kNegInf, a1 = v1 ? scale * s1[n] : kNegInf;
                    float mt = fmaxf(a0, a1);
    #pragma unroll
                    for (int o = 4; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    const float mnew = fmaxf(m_run[n], mt);   // finite: position 0 of the tile is valid
                    const float alpha = expf(m_run[n] - mnew);
                    const float pa = v0 ? expf(a0 - mnew) : 0.0f, pb = v1 ? expf(a1 - mnew) : 0.0f;
                    l_part[n] = fmaf(l_part[n], alpha, pa + pb);
                    m_run[n] = mnew;
                    const int h = 4 * n + tq;
                    if (h < G) {
                        spw[gq * G + h] = pa;
                        spw[(gq + 8) * G + h] = pb;
                        if (gq == 0) saw[h] = alpha;
                    }
                }
                __syncwarp();
    #pragma unroll
                for (int h = 0; h < GP; ++h) {
                    const float2 al = make_float2(saw[2 * h], 2 * h + 1 < G ? saw[2 * h + 1] : 0.0f);
    #pragma unroll
                    for (int k = 0; k < NB; ++k) acc[h][k] = __fmul2_rn(acc[h][k], al);
                }
                // sum_j p_j d_j q_j: this lane's elements, every head (a full tile
                // unrolled, so the loads of several positions are in flight).  The
                // rows' alignment is the same in every position (misg; slots are
                // 16-byte multiples), so the code reader is set up once.
                const uint8_t* vt = vst + jt * Gm::SLOT + misg + eb * BB;
                const Codes<T, (NB >= 4 ? NB / 4 : 1)> vc(vt, e0);
                auto vrow = [&](int j) {
                    const uint8_t* vb = vt + j * Gm::SLOT;
                    const float dv = h2f(lds16(vb));
                    float vv[NB];
                    if constexpr (NB >= 4) {
                        uint32_t cw[NB / 4];
                        vc.load((uint32_t)(j * Gm::SLOT), cw);
                        // Byte b as the fp32 2^23 + b (one byte permute), less
                        // 2^23 and the code offset (Q8_0: bytes flipped to q + 128).
                        constexpr float kOff = 8388608.0f + (T == T_Q8_0 ? 128.0f : (T == T_Q5_0 ? 16.0f : 8.0f));
    #pragma unroll
                        for (int w = 0; w < NB / 4; ++w) {
                            const uint32_t u = T == T_Q8_0 ? cw[w] ^ 0x80808080u : cw[w];
                            const float2 f01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)),
                                                                      __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651))),
                                                          make_float2(-kOff, -kOff));
                            const float2 f23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)),
                                                                      __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653))),
                                                          make_float2(-kOff, -kOff));
                            vv[4 * w] = f01.x; vv[4 * w + 1] = f01.y; vv[4 * w + 2] = f23.x; vv[4 * w + 3] = f23.y;
                        }
                    } else {
    #pragma unroll
                        for (int k = 0; k < NB; ++k) vv[k] = (float)code_at<T>(vb, e0 + k);
                    }
                    float pj[2 * GP];
                    if constexpr (G % 4 == 0) {
    #pragma unroll
                        for (int h = 0; h < G; h += 4) {
                            const float4 p4 = *reinterpret_cast<const float4*>(spw + j * G + h);
                            pj[h] = p4.x; pj[h + 1] = p4.y; pj[h + 2] = p4.z; pj[h + 3] = p4.w;
                        }
                    } else {
    #pragma unroll
                        for (int h = 0; h < G; ++h) pj[h] = spw[j * G + h];
                        if constexpr (G % 2) pj[G] = 0.0f;
                    }
    #pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        const float2 pd = __fmul2_rn(make_float2(pj[2 * h], pj[2 * h + 1]), make_float2(dv, dv));
    #pragma unroll
                        for (int k = 0; k < NB; ++k) acc[h][k] = __ffma2_rn(pd, make_float2(vv[k], vv[k]), acc[h][k]);
                    }
                };
                if (nvalid == 16) {
    #pragma unroll
                    for (int j = 0; j < 16; ++j) vrow(j);
                } else {
                    for (int j = 0; j < nvalid; ++j) vrow(j);
                }
                __syncwarp();   // spw and saw are rewritten by the next tile
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == nstg) {
                slot = 0;
                ph ^= 1u;
            }
        }
        // The softmax sums of the warp's positions: the lanes of a head.
    #pragma unroll
        for (int n = 0; n < NT; ++n)
    #pragma unroll
            for (int o = 4; o < 32; o <<= 1) l_part[n] += __shfl_xor_sync(0xffffffffu, l_part[n], o);
        // Merge the warps in order (the ring is free now): per warp and head,
        // (m, l, o[D]) in shared memory, then per output element.
        named_sync_stream_consumers();
        float* mg = reinterpret_cast<float*>(ring);   // [kSW][G][D + 2]
    #pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int h = 4 * n + tq;
            if (h < G && gq == 0) {
                mg[(warp * G + h) * (D + 2)] = m_run[n];
                mg[(warp * G + h) * (D + 2) + 1] = l_part[n];
            }
        }
    #pragma unroll
        for (int h = 0; h < G; ++h)
    #pragma unroll
            for (int k = 0; k < NB; ++k)
                mg[(warp * G + h) * (D + 2) + 2 + lane * NB + k] = (h & 1) ? acc[h >> 1][k].y : acc[h >> 1][k].x;
        named_sync_stream_consumers();
        if (*abort) return;
        for (int i = tid; i < G * D; i += kSW * 32) {
            const int h = i / D, e = i - h * D;
            float M = kNegInf;
    #pragma unroll
            for (int w = 0; w < kSW; ++w) M = fmaxf(M, mg[(w * G + h) * (D + 2)]);
            float o = 0.0f, L = 0.0f;
    #pragma unroll
            for (int w = 0; w < kSW; ++w) {
                const float* r = mg + (w * G + h) * (D + 2);
                const float f = expf(r[0] - M);   // 0 for a warp with no position
                o = fmaf(f, r[2 + e], o);
                L = fmaf(f, r[1], L);
            }
            float* dst = ws + ((int64_t)(g * G + h) * nsplit + c) * (D + 2);
            dst[2 + e] = o;
            if (e == 0) {
                dst[0] = M;
                dst[1] = L;
            }
        }
    }
}

// (m, l) of two sets of scores merged: m = max, l = sum of l_i e^(m_i - m).
__device__ __forceinline__ void ml_merge(float& m, float& l, float m2, float l2) {
    const float mm = fmaxf(m, m2);
    if (mm == -__int_as_float(0x7f800000)) return;   // both empty
    l = l * expf(m - mm) + l2 * expf(m2 - mm);
    m = mm;
}

// out[h, e] = sum_c e^(m_c - M) o_c[e] / sum_c e^(m_c - M) l_c.  CTA (h, e0)
// takes head h and elements e0 .. e0 + 31: (M, L) by merging the chunks'
// (m_c, l_c) in a fixed order (each thread its chunks c = tid mod 256 in
// turn, then a shuffle tree per warp, then the warps in order), and each
// element's o-sum split over 8 chunk groups (chunks c = k mod 8) that are
// added in group order: deterministic.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ ws, int nchunks, int D,
                                                          float* __restrict__ out) {
    __shared__ float wm[8], wl[8], ML[2];
    __shared__ float part[8][32];
    pdl_wait_prior();
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t stride = D + 2;
    const float* base = ws + (int64_t)h * nchunks * stride;
    float m = -__int_as_float(0x7f800000), l = 0.0f;
    for (int c = tid; c < nchunks; c += 256) ml_merge(m, l, base[(int64_t)c * stride], base[(int64_t)c * stride + 1]);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
        // Lanes that meet merge in lane order, so both ends of a pair hold the same bits.
        if (lane & o) {
            float mb = m2, lb = l2;
            ml_merge(mb, lb, m, l);
            m = mb;
            l = lb;
        } else {
            ml_merge(m, l, m2, l2);
        }
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
    __syncthreads();
    if (tid == 0) {
        float M = wm[0], L = wl[0];
        for (int w = 1; w < 8; ++w) ml_merge(M, L, wm[w], wl[w]);
        ML[0] = M;
        ML[1] = L;
    }
    __syncthreads();
    const float M = ML[0], L = ML[1];
    const int el = tid & 31, cg = tid >> 5, e = blockIdx.y * 32 + el;
    float acc = 0.0f;
    if (e < D) {
#pragma unroll 4
        for (int c = cg; c < nchunks; c += 8) {
            const float* p = base + (int64_t)c * stride;
            acc = fmaf(expf(p[0] - M), p[2 + e], acc);
        }
    }
    part[cg][el] = acc;
    __syncthreads();
    if (cg == 0 && e < D) {
        float o = part[0][el];
        for (int k = 1; k < 8; ++k) o += part[k][el];
        out[(int64_t)h * D + e] = o / L;
    }
}

template <int T, int NB, int GT>
cudaError_t launch_tn(const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads, int n_kv,
                      float scale, float* out, float* ws, cudaStream_t s) {
    constexpr int CH = chunk_of<T>();
    using R = Rows<T, NB, CH>;
    const int64_t nch = (T_len + CH - 1) / CH;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)(n_kv * nch));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = R::SMEM;
    cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<T, NB, GT, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         R::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, attn_chunk_kernel<T, NB, GT, CH>, q, K, V, T_len, n_heads, n_kv, scale, ws);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)n_heads, (unsigned)((32 * NB + 31) / 32));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel, (const float*)ws, (int)nch, 32 * NB, out);
}

// The streaming kernel with CTAs ~ two per SM: P positions each (a multiple
// of the stage, at least one stage, so the partials fit the workspace sized
// for 128-position chunks).  It needs the TMA boxes: a position's n_kv ROWB
// bytes a multiple of 16 (the tensor map's row pitch) and the box at most
// 256 bytes wide; and two ring stages in its shared memory.
template <int T, int NB, int G>
bool stream_fits(int n_kv) {
    using Gm = SGeo<T, NB>;
    using Mp = SMap<T, NB, G>;
    const int nstg = std::min(kSMaxStages, (kSBudget - Mp::bytes(0)) / Gm::STAGE);
    return ((int64_t)n_kv * Gm::ROWB) % 16 == 0 && Gm::SLOT <= 256 && nstg >= 2 &&
           kSW * G * (32 * NB + 2) * 4 <= nstg * Gm::STAGE;
}

// The cache [T, n_kv ROWB] as 8-bit elements, box SLOT x kSPos.
template <int T, int NB>
bool encode_cache_map(CUtensorMap* map, const uint8_t* C, int64_t T_len, int n_kv) {
    using Gm = SGeo<T, NB>;
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t pitch = (cuuint64_t)n_kv * Gm::ROWB;
    cuuint64_t gdim[2] = {pitch, (cuuint64_t)T_len};
    cuuint64_t gstride[1] = {pitch};
    cuuint32_t box[2] = {(cuuint32_t)Gm::SLOT, (cuuint32_t)kSPos};
    cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(C), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int T, int NB, int G>
cudaError_t launch_sn(const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_kv, float scale,
                      float* out, float* ws, unsigned* status, int sms, cudaStream_t s) {
    using Gm = SGeo<T, NB>;
    using Mp = SMap<T, NB, G>;
    CUtensorMap kmap, vmap;
    if (!encode_cache_map<T, NB>(&kmap, K, T_len, n_kv) || !encode_cache_map<T, NB>(&vmap, V, T_len, n_kv))
        return cudaErrorInvalidValue;
    const int nstg = std::min(kSMaxStages, (kSBudget - Mp::bytes(0)) / Gm::STAGE);
    const int smem = Mp::bytes(nstg);
    const int64_t s0 = std::max<int64_t>(1, 2 * (int64_t)std::max(sms, 1) / n_kv);
    const int64_t per = (T_len + s0 - 1) / s0;
    const int P = (int)std::max<int64_t>(kSPos, (per + kSPos - 1) / kSPos * kSPos);
    const int nsplit = (int)((T_len + P - 1) / P);
    auto kern = attn_stream_kernel<T, NB, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)(n_kv * nsplit));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, q, T_len, n_kv, scale, ws, P, nsplit, nstg, status);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(n_kv * G), (unsigned)NB);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel, (const float*)ws, nsplit, 32 * NB, out);
}

// The streaming kernel for the fixed groups whose per-lane state fits the
// registers (G heads x d/32 sums, the query fragments), else the chunk
// kernels: fixed-group where a lane's G d/32 elements make whole words
// inside one block, the runtime-group one otherwise.
template <int T, int NB, int G>
constexpr bool stream_regs_ok() {
    return G * NB + 4 * NB * ((2 * G + 7) / 8) <= 48;
}

template <int T, int NB>
cudaError_t launch_g(const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads, int n_kv,
                     float scale, float* out, float* ws, unsigned* status, int sms, cudaStream_t s) {
    const int G = n_heads / n_kv;
    if constexpr (stream_regs_ok<T, NB, 1>())
        if (G == 1 && stream_fits<T, NB, 1>(n_kv)) return launch_sn<T, NB, 1>(q, K, V, T_len, n_kv, scale, out, ws, status, sms, s);
    if constexpr (stream_regs_ok<T, NB, 2>())
        if (G == 2 && stream_fits<T, NB, 2>(n_kv)) return launch_sn<T, NB, 2>(q, K, V, T_len, n_kv, scale, out, ws, status, sms, s);
    if constexpr (stream_regs_ok<T, NB, 4>())
        if (G == 4 && stream_fits<T, NB, 4>(n_kv)) return launch_sn<T, NB, 4>(q, K, V, T_len, n_kv, scale, out, ws, status, sms, s);
    if constexpr (stream_regs_ok<T, NB, 8>())
        if (G == 8 && stream_fits<T, NB, 8>(n_kv)) return launch_sn<T, NB, 8>(q, K, V, T_len, n_kv, scale, out, ws, status, sms, s);
    if constexpr (NB <= 4) {
        if (G == 8 && 8 * NB <= 32) return launch_tn<T, NB, 8>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    }
    if constexpr (NB >= 1 && NB <= 8) {
        if (G == 4 && 4 * NB >= 4 && 4 * NB <= 32) return launch_tn<T, NB, 4>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    }
    if constexpr (NB >= 2) {
        if (G == 2 && 2 * NB <= 32) return launch_tn<T, NB, 2>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    }
    if constexpr (NB >= 4) {
        if (G == 1) return launch_tn<T, NB, 1>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    }
    return launch_tn<T, NB, 0>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
}

template <int T>
cudaError_t launch_t(const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads, int n_kv, int d,
                     float scale, float* out, float* ws, unsigned* status, int sms, cudaStream_t s) {
    switch (d) {
    case 32: return launch_g<T, 1>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, status, sms, s);
    case 64: return launch_g<T, 2>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, status, sms, s);
    case 128: return launch_g<T, 4>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, status, sms, s);
    case 256: return launch_g<T, 8>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, status, sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace attn

int64_t attn_decode_ws_bytes(int64_t T_len, int n_heads, int d) {
    const int64_t nch = (T_len + attn::kMinChunk - 1) / attn::kMinChunk;
    return nch * n_heads * (int64_t)(d + 2) * (int64_t)sizeof(float);
}

bool attn_decode_shape_ok(int n_heads, int n_kv, int d) {
    return n_kv > 0 && n_heads % n_kv == 0 && n_heads / n_kv <= attn::kMaxG && (d == 32 || d == 64 || d == 128 || d == 256);
}

cudaError_t launch_attn_decode(int type, const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads,
                               int n_kv, int d, float scale, float* out, float* ws, unsigned* status, int sms,
                               cudaStream_t s) {
    switch (type) {
    case T_Q8_0: return attn::launch_t<T_Q8_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, status, sms, s);
    case T_Q5_0: return attn::launch_t<T_Q5_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, status, sms, s);
    case T_Q4_0: return attn::launch_t<T_Q4_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, status, sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
