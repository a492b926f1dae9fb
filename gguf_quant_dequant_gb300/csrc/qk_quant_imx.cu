// qk_quant_imx.cu -- importance-weighted quantization (the imatrix objective
// of "Hitchhiker's Guide -- Lab 01", 11.3: minimise sum_i E[x_i^2] (w_i -
// w^_i)^2 instead of the plain weight-space error).  Per block, in this
// order (all fp32, every sum in index order, explicit round-to-nearest
// operations so that nothing is contracted):
//   1. per group (32-weight block of Q8_0 / Q5_0 / Q4_0, 32-weight sub-block
//      of Q4_K / Q5_K, 16-weight group of Q6_K / Q3_K / Q2_K): the plain
//      scheme's scale s0 (and min m0); 21 candidate scales s0 (90 + k) / 100;
//      codes rounded with (s, m0); a weighted least-squares refit of the
//      scale (or of scale and min together, kept only with a positive
//      determinant, a positive scale and a non-negative min); the candidate
//      of least weighted error wins, the first on ties;
//   2. the block assembled as the plain quantizer does, with the winners in
//      place of (s0, m0);
//   3. that block and the plain one decoded, their weighted errors summed per
//      group and then over groups; the plain block is kept unless the
//      weighted one is no worse.
// Layout of the work: the plain quantizer's (qk_qlanes.cuh): a warp takes 32
// consecutive 32-weight groups, each lane the 32 weights of one (its one or
// two groups of step 1), so every lane searches its own groups with its
// weights and importances in registers; both blocks are assembled by the
// shared lane code into shared memory, each lane decodes its own weights of
// both, and the lanes of a block add the group errors in group order.
#include "qk_internal.h"
#include "qk_qlanes.cuh"

namespace qk {
namespace imx {

constexpr int kWarps = 8;                    // per CTA
constexpr int kBufWords = 32 * 34 / 4;      // largest warp output: 32 Q8_0 blocks = 1088 bytes

template <int T> struct Geo;   // symmetric?, code range of step 1
template <> struct Geo<T_Q8_0> { static constexpr bool SYM = true; static constexpr int LO = -128, HI = 127; };
template <> struct Geo<T_Q5_0> { static constexpr bool SYM = true; static constexpr int LO = -16, HI = 15; };
template <> struct Geo<T_Q4_0> { static constexpr bool SYM = true; static constexpr int LO = -8, HI = 7; };
template <> struct Geo<T_Q6_K> { static constexpr bool SYM = true; static constexpr int LO = -32, HI = 31; };
template <> struct Geo<T_Q3_K> { static constexpr bool SYM = true; static constexpr int LO = -4, HI = 3; };
template <> struct Geo<T_Q4_K> { static constexpr bool SYM = false; static constexpr int LO = 0, HI = 15; };
template <> struct Geo<T_Q5_K> { static constexpr bool SYM = false; static constexpr int LO = 0, HI = 31; };
template <> struct Geo<T_Q2_K> { static constexpr bool SYM = false; static constexpr int LO = 0, HI = 3; };

// Step 1 for one group of G weights x with importances a, from the plain
// (s0, m0).  The codes of a candidate come from one reciprocal of its scale
// (group rounding of qk_codes.cuh: the division's codes exactly).
template <int T, int G>
__device__ __forceinline__ void search(const float* x, const float* a, float s0, float m0, float& s_out,
                                       float& m_out) {
    using P = Geo<T>;
    s_out = s0;
    m_out = m0;
    if (!(s0 > 0.0f)) return;
    // Candidate-independent sums of the refit (index order).
    float Sa = 0.0f, Sw = 0.0f;
    if constexpr (!P::SYM) {
#pragma unroll
        for (int l = 0; l < G; ++l) {
            Sa = __fadd_rn(Sa, a[l]);
            Sw = __fadd_rn(Sw, __fmul_rn(a[l], x[l]));
        }
    }
    const float flo = (float)P::LO, fhi = (float)P::HI, magic = 12582912.0f;
    // The rounding test of group_codes (qk_codes.cuh): per value for wide
    // code ranges, the group's largest distance for ranges within +-16.
    constexpr int kM = (-P::LO > P::HI) ? -P::LO : P::HI;
    constexpr bool kWide = kM > 16;
    const float limit = kWide ? 0.5f : 0.5f - (float)kM * 0x1p-20f;
    float best = __int_as_float(0x7f800000);
#pragma unroll 1
    for (int k = 0; k <= 20; ++k) {
        const float s = __fmul_rn(s0, __fdiv_rn((float)(90 + k), 100.0f));
        const float rd = approx_rcp(s);
        float q[G];
        float worst = 0.0f;
#pragma unroll
        for (int l = 0; l < G; ++l) {
            const float u = P::SYM ? x[l] : __fadd_rn(x[l], m0);
            const float y = fminf(fmaxf(__fmul_rn(u, rd), flo), fhi);
            q[l] = __fsub_rn(__fadd_rn(y, magic), magic);
            const float dist = fabsf(__fsub_rn(y, q[l]));
            worst = fmaxf(worst, kWide ? __fmaf_rn(fabsf(y), 0x1p-20f, dist) : dist);
        }
        if (!(rcp_usable(s) && worst < limit)) {   // rare: a code the approximate quotient cannot decide
#pragma unroll
            for (int l = 0; l < G; ++l)
                q[l] = (float)cr(__fdiv_rn(P::SYM ? x[l] : __fadd_rn(x[l], m0), s), P::LO, P::HI);
        }
        float ss, mm = 0.0f;
        if constexpr (P::SYM) {
            float num = 0.0f, den = 0.0f;
#pragma unroll
            for (int l = 0; l < G; ++l) {
                const float aq = __fmul_rn(a[l], q[l]);
                num = __fadd_rn(num, __fmul_rn(aq, x[l]));
                den = __fadd_rn(den, __fmul_rn(aq, q[l]));
            }
            if (!(den > 0.0f)) continue;
            ss = __fdiv_rn(num, den);
        } else {
            float Sq = 0.0f, Sqq = 0.0f, Swq = 0.0f;
#pragma unroll
            for (int l = 0; l < G; ++l) {
                const float aq = __fmul_rn(a[l], q[l]);
                Sq = __fadd_rn(Sq, aq);
                Sqq = __fadd_rn(Sqq, __fmul_rn(aq, q[l]));
                Swq = __fadd_rn(Swq, __fmul_rn(aq, x[l]));
            }
            const float det = __fsub_rn(__fmul_rn(Sqq, Sa), __fmul_rn(Sq, Sq));
            if (!(det > 0.0f)) continue;
            ss = __fdiv_rn(__fsub_rn(__fmul_rn(Swq, Sa), __fmul_rn(Sq, Sw)), det);
            mm = __fdiv_rn(__fsub_rn(__fmul_rn(Swq, Sq), __fmul_rn(Sqq, Sw)), det);
            if (!(ss > 0.0f) || !(mm >= 0.0f)) continue;
        }
        // Weighted error of this candidate (the same codes).
        float e = 0.0f;
#pragma unroll
        for (int l = 0; l < G; ++l) {
            const float r = __fsub_rn(x[l], __fsub_rn(__fmul_rn(ss, q[l]), mm));
            e = __fadd_rn(e, __fmul_rn(a[l], __fmul_rn(r, r)));
        }
        if (e < best) {
            best = e;
            s_out = ss;
            m_out = mm;
        }
    }
}

// Step 3 for the lane's weights: the weighted error of each of its groups,
// from the block's bytes (`blk`: the super-block for the K types, the
// lane's block otherwise) decoded by the shared half decoders.  The lane's
// 32 weights are two halves of 16: (u0, h0) then (u1, h1).
template <int T>
__device__ __forceinline__ void lane_errors(const uint8_t* blk, const float (&x)[32], const float (&a)[32], int lane,
                                            float (&e)[2]) {
    const int j = lane & 7;
    int u0 = 0, h0 = 0, u1 = 0, h1 = 1;
    if constexpr (T == T_Q4_K || T == T_Q5_K) {   // sub-block j: halves j % 2 of units 2(j/2), 2(j/2) + 1
        u0 = 2 * (j >> 1);
        u1 = u0 + 1;
        h0 = h1 = j & 1;
    } else if constexpr (T == T_Q2_K || T == T_Q3_K) {   // unit j
        u0 = u1 = j;
    } else if constexpr (T == T_Q6_K) {   // weights 32j..: units 4(j/4) + 2(j%2) + {0, 1}, half (j/2) % 2
        u0 = 4 * (j >> 2) + 2 * (j & 1);
        u1 = u0 + 1;
        h0 = h1 = (j >> 1) & 1;
    }
    float w0[16], w1[16];
    dequant_half<T>(blk, u0, h0, w0);
    dequant_half<T>(blk, u1, h1, w1);
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        const float r = __fsub_rn(x[l], w0[l]);
        s0 = __fadd_rn(s0, __fmul_rn(a[l], __fmul_rn(r, r)));
    }
    float& t = ql::LaneGeo<T>::G == 32 ? s0 : s1;   // a 32-weight group continues the same sum
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        const float r = __fsub_rn(x[16 + l], w1[l]);
        t = __fadd_rn(t, __fmul_rn(a[16 + l], __fmul_rn(r, r)));
    }
    e[0] = s0;
    e[1] = s1;
}

template <int T>
__global__ void __launch_bounds__(kWarps * 32) quantize_imatrix_kernel(const float* __restrict__ w,
                                                                       const float* __restrict__ imp, int64_t ngroups,
                                                                       int64_t groups_per_row,
                                                                       uint8_t* __restrict__ out) {
    using LG = ql::LaneGeo<T>;
    constexpr int kBB = Fmt<T>::BB;
    __shared__ __align__(16) uint32_t buf[2][kWarps][kBufWords];   // plain, weighted
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g0 = ((int64_t)blockIdx.x * kWarps + warp) * 32;
    if (g0 >= ngroups) return;   // whole warp
    const int64_t left = ngroups - g0;
    const int ng = left < 32 ? (int)left : 32;   // a multiple of 8 for the K types
    const bool live = lane < ng;
    float v[32], a[32];
    if (live) {
        const float4* src = reinterpret_cast<const float4*>(w + (g0 + lane) * 32);
        const float* isrc = imp + ((g0 + lane) % groups_per_row) * 32;   // 4-byte aligned
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = __ldcs(src + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
        if ((reinterpret_cast<uintptr_t>(imp) & 15) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 m = __ldg(reinterpret_cast<const float4*>(isrc) + i);
                a[4 * i] = m.x;
                a[4 * i + 1] = m.y;
                a[4 * i + 2] = m.z;
                a[4 * i + 3] = m.w;
            }
        } else {
#pragma unroll
            for (int l = 0; l < 32; ++l) a[l] = __ldg(isrc + l);
        }
    } else {
#pragma unroll
        for (int l = 0; l < 32; ++l) v[l] = a[l] = 0.0f;
    }
    const int bo = (LG::K ? (lane >> 3) : lane) * kBB;
    uint8_t* bp = reinterpret_cast<uint8_t*>(buf[0][warp]);
    uint8_t* bw = reinterpret_cast<uint8_t*>(buf[1][warp]);
    float sp[2], mp[2], sw[2], mw[2];
    ql::plain_params<T>(v, sp, mp);
    ql::assemble<T>(v, sp, mp, lane, live, bp + bo);
    sw[1] = mw[1] = 0.0f;
#pragma unroll
    for (int e = 0; e < LG::NG; ++e) search<T, LG::G>(v + LG::G * e, a + LG::G * e, sp[e], mp[e], sw[e], mw[e]);
    ql::assemble<T>(v, sw, mw, lane, live, bw + bo);
    __syncwarp();
    float ep[2], ew[2];
    lane_errors<T>(bp + bo, v, a, lane, ep);
    lane_errors<T>(bw + bo, v, a, lane, ew);
    // Block totals over its groups in order (a K type's groups sit in the
    // eight lanes of its super-block, in lane order).
    float tp = 0.0f, tw = 0.0f;
    if constexpr (LG::K) {
#pragma unroll
        for (int jp = 0; jp < 8; ++jp) {
#pragma unroll
            for (int e = 0; e < LG::NG; ++e) {
                tp = __fadd_rn(tp, __shfl_sync(ql::kFull, ep[e], (lane & ~7) + jp));
                tw = __fadd_rn(tw, __shfl_sync(ql::kFull, ew[e], (lane & ~7) + jp));
            }
        }
    } else {
        tp = __fadd_rn(tp, ep[0]);
        tw = __fadd_rn(tw, ew[0]);
    }
    // The weighted block replaces the plain one where it is no worse; the
    // lanes of a block copy its bytes.
    if (live && tw <= tp) {
        const int nl = LG::K ? 8 : 1, me = LG::K ? (lane & 7) : 0;
        for (int i = me; i < kBB; i += nl) bp[bo + i] = bw[bo + i];
    }
    __syncwarp();
    const int64_t ob = (LG::K ? g0 / 8 : g0) * kBB;
    const int nb = (LG::K ? ng / 8 : ng) * kBB;
    uint8_t* dst = out + ob;
    for (int i = lane; i < nb / 4; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = buf[0][warp][i];
    if (lane < (nb & 3)) dst[(nb & ~3) + lane] = bp[(nb & ~3) + lane];
}

template <int T>
cudaError_t launch_t(const float* w, const float* imp, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t s) {
    const int64_t gpr = cols / 32, ngroups = rows * gpr;
    if (ngroups == 0) return cudaSuccess;
    const int64_t warps = (ngroups + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quantize_imatrix_kernel<T><<<(unsigned)blocks, kWarps * 32, 0, s>>>(w, imp, ngroups, gpr, out);
    return cudaGetLastError();
}

}  // namespace imx

cudaError_t launch_quantize_imatrix(int type, const float* w, const float* imp, int64_t rows, int64_t cols,
                                   uint8_t* out, cudaStream_t s) {
    switch (type) {
    case T_Q4_K: return imx::launch_t<T_Q4_K>(w, imp, rows, cols, out, s);
    case T_Q6_K: return imx::launch_t<T_Q6_K>(w, imp, rows, cols, out, s);
    case T_Q8_0: return imx::launch_t<T_Q8_0>(w, imp, rows, cols, out, s);
    case T_Q5_0: return imx::launch_t<T_Q5_0>(w, imp, rows, cols, out, s);
    case T_Q4_0: return imx::launch_t<T_Q4_0>(w, imp, rows, cols, out, s);
    case T_Q5_K: return imx::launch_t<T_Q5_K>(w, imp, rows, cols, out, s);
    case T_Q2_K: return imx::launch_t<T_Q2_K>(w, imp, rows, cols, out, s);
    case T_Q3_K: return imx::launch_t<T_Q3_K>(w, imp, rows, cols, out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
