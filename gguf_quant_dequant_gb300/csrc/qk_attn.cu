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
// Pass 1: each warp takes every 8th position.  With the group size G known
// at compile time (and 4 <= G d/32 <= 32), lane l works for head l / (32/G)
// on G d/32 consecutive elements (inside one block): the group's queries are
// first turned into three-limb fixed point (as the decode GEMV's activations:
// x = s (65536 a + 256 b + c) per 32-block, signed 8-bit limbs), so each
// score is an exact integer dp4a sum over the cache's codes, added over the
// head's lanes by shuffles.  Otherwise lane l owns d/32 elements and forms its
// share of q_h . K[t, g] for every head in fp32.  The chunk's softmax
// statistics (max, sum of exp) follow in shared memory.
// Pass 2: the same row mapping over V accumulates sum_t e^(s_t - m) V[t, g]
// per head; the warps' sums are added in warp order.  A second kernel
// combines the chunks (log-sum-exp) in a fixed order: deterministic.
#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_lanes.cuh"
#include "qk_ptx.cuh"

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
    __shared__ float sq[GG][D];                  // the group's queries
    __shared__ __align__(16) float ss[CH][GG];   // scores, then e^(s - m), per position
    __shared__ float sred[2][GG];
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
    // Lane l: elements e0 .. e0 + NB - 1 of block eb (pass 2, and pass 1 without a fixed group).
    const int e0 = (lane * NB) & 31, eb = (lane * NB) >> 5;
    if constexpr (GT > 0) {
        constexpr int LPH = 32 / GT, EPL = D / LPH, W = EPL / 4;   // lanes per head, elements per lane
        static_assert(EPL % 4 == 0 && EPL <= 32, "one lane's elements lie in one block");
        const int h = lane / LPH, ea = (lane % LPH) * EPL;          // head, first element
        const int kb = ea >> 5, k0 = ea & 31;
        // The lane's limbs: block maximum over the 32 / EPL lanes that share the block.
        float qv[EPL], amax = 0.0f;
#pragma unroll
        for (int k = 0; k < EPL; ++k) {
            qv[k] = sq[h][ea + k];
            amax = fmaxf(amax, fabsf(qv[k]));
        }
#pragma unroll
        for (int o = 1; o < 32 / EPL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sx = amax * (1.0f / gv::kXMax);
        const float inv = amax > 0.0f ? __fdividef(gv::kXMax, amax) : 0.0f;
        uint32_t la[W], lb[W], lc[W];
        int xsum = 0;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            uint32_t Y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int X = __float2int_rn(qv[4 * i + k] * inv);
                xsum += X;
                Y[k] = (uint32_t)(X + 0x808080);
            }
            la[i] = (((Y[0] >> 16) & 255u) | (((Y[1] >> 16) & 255u) << 8) | (((Y[2] >> 16) & 255u) << 16) |
                     (((Y[3] >> 16) & 255u) << 24)) ^ 0x80808080u;
            lb[i] = (((Y[0] >> 8) & 255u) | (((Y[1] >> 8) & 255u) << 8) | (((Y[2] >> 8) & 255u) << 16) |
                     (((Y[3] >> 8) & 255u) << 24)) ^ 0x80808080u;
            lc[i] = ((Y[0] & 255u) | ((Y[1] & 255u) << 8) | ((Y[2] & 255u) << 16) | ((Y[3] & 255u) << 24)) ^
                    0x80808080u;
        }
        constexpr float kOff = T == T_Q8_0 ? 0.0f : (T == T_Q5_0 ? 16.0f : 8.0f);
        const float offx = kOff * (float)xsum;
        cp_async_wait<1>();   // this thread's K copies
        __syncthreads();      // ... and everyone's
        const uint8_t* kblk = sK + warp * R::SLOT + mis + kb * BB;
        const Codes<T, W> kc(kblk, k0);
        uint32_t off = 0;
        for (int j = warp; j < nt; j += kWarps, off += STEP) {
            uint32_t cw[W];
            kc.load(off, cw);
            int A = 0, B = 0, C = 0;
#pragma unroll
            for (int i = 0; i < W; ++i) {
                A = gv::dp4a_ss(cw[i], la[i], A);
                B = gv::dp4a_ss(cw[i], lb[i], B);
                C = gv::dp4a_ss(cw[i], lc[i], C);
            }
            float v = h2f(lds16(kblk + off)) * (sx * (gv::limbs3_to_f(A, B, C) - offx));
#pragma unroll
            for (int o = LPH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane % LPH == 0) ss[j][h] = scale * v;
        }
    } else {
    float qr[kMaxG][NB];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h)
#pragma unroll
        for (int k = 0; k < NB; ++k) qr[h][k] = h < G ? sq[h][lane * NB + k] : 0.0f;

    cp_async_wait<1>();   // this thread's K copies
    __syncthreads();      // ... and everyone's
    // Pass 1: scores.
    const uint8_t* blk = sK + warp * R::SLOT + mis + eb * BB;
    for (int j = warp; j < nt; j += kWarps, blk += STEP) {
        const float dk = h2f(ld_u16(blk));
        int cv[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) cv[k] = code_at<T>(blk, e0 + k);
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
            if (h >= G) break;
            float a = 0.0f;
#pragma unroll
            for (int k = 0; k < NB; ++k) a = fmaf(qr[h][k], (float)cv[k], a);
            a *= dk;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) ss[j][h] = scale * a;
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

// The fixed-group kernel where a lane's G d/32 elements make whole words
// inside one block, the runtime-group one otherwise.
template <int T, int NB>
cudaError_t launch_g(const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads, int n_kv,
                     float scale, float* out, float* ws, cudaStream_t s) {
    const int G = n_heads / n_kv;
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
                     float scale, float* out, float* ws, cudaStream_t s) {
    switch (d) {
    case 32: return launch_g<T, 1>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    case 64: return launch_g<T, 2>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    case 128: return launch_g<T, 4>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
    case 256: return launch_g<T, 8>(q, K, V, T_len, n_heads, n_kv, scale, out, ws, s);
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
                               int n_kv, int d, float scale, float* out, float* ws, cudaStream_t s) {
    switch (type) {
    case T_Q8_0: return attn::launch_t<T_Q8_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, s);
    case T_Q5_0: return attn::launch_t<T_Q5_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, s);
    case T_Q4_0: return attn::launch_t<T_Q4_0>(q, K, V, T_len, n_heads, n_kv, d, scale, out, ws, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
