// qk_quant_imx.cu -- importance-weighted quantization (the imatrix objective
// of "Hitchhiker's Guide -- Lab 01", 11.3: minimise sum_i E[x_i^2] (w_i -
// w^_i)^2 instead of the plain weight-space error).  Offline work, so one
// thread encodes one block, in this order (all fp32, every sum in index
// order, explicit round-to-nearest operations so that nothing is contracted):
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
#include <cuda_fp16.h>

#include "qk_formats.cuh"
#include "qk_internal.h"

namespace qk {
namespace imx {

__device__ __forceinline__ int cr(float v, int lo, int hi) {
    float r = roundf(v);
    if (!(r >= (float)lo)) r = (float)lo;
    if (r > (float)hi) r = (float)hi;
    return (int)r;
}
__device__ __forceinline__ uint32_t h16(float v) { return (uint32_t)__half_as_ushort(__float2half_rn(v)); }
__device__ __forceinline__ float f16(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }

template <int T> struct Geo;   // group size, symmetric?, plain divisor / steps, code range
template <> struct Geo<T_Q8_0> { static constexpr int G = 32; static constexpr bool SYM = true; static constexpr int DIV = 127, LO = -128, HI = 127; };
template <> struct Geo<T_Q5_0> { static constexpr int G = 32; static constexpr bool SYM = true; static constexpr int DIV = 15, LO = -16, HI = 15; };
template <> struct Geo<T_Q4_0> { static constexpr int G = 32; static constexpr bool SYM = true; static constexpr int DIV = 7, LO = -8, HI = 7; };
template <> struct Geo<T_Q6_K> { static constexpr int G = 16; static constexpr bool SYM = true; static constexpr int DIV = 32, LO = -32, HI = 31; };
template <> struct Geo<T_Q3_K> { static constexpr int G = 16; static constexpr bool SYM = true; static constexpr int DIV = 4, LO = -4, HI = 3; };
template <> struct Geo<T_Q4_K> { static constexpr int G = 32; static constexpr bool SYM = false; static constexpr int DIV = 15, LO = 0, HI = 15; };
template <> struct Geo<T_Q5_K> { static constexpr int G = 32; static constexpr bool SYM = false; static constexpr int DIV = 31, LO = 0, HI = 31; };
template <> struct Geo<T_Q2_K> { static constexpr int G = 16; static constexpr bool SYM = false; static constexpr int DIV = 3, LO = 0, HI = 3; };

// Step 1 for one group at x (weights) and a (importances); plain == true
// returns the plain (s0, m0) without searching.
template <int T>
__device__ void group_params(const float* x, const float* a, bool plain, float& s_out, float& m_out) {
    using P = Geo<T>;
    float s0, m0 = 0.0f;
    if constexpr (P::SYM) {
        float amax = 0.0f;
        for (int l = 0; l < P::G; ++l) {
            const float v = fabsf(x[l]);
            if (v > amax) amax = v;
        }
        s0 = __fdiv_rn(amax, (float)P::DIV);
    } else {
        float lo = 0.0f, hi = x[0];
        for (int l = 0; l < P::G; ++l) {
            if (x[l] < lo) lo = x[l];
            if (x[l] > hi) hi = x[l];
        }
        s0 = __fdiv_rn(__fsub_rn(hi, lo), (float)P::DIV);
        m0 = -lo;
    }
    s_out = s0;
    m_out = m0;
    if (plain || !(s0 > 0.0f)) return;
    float best = __int_as_float(0x7f800000);
    for (int k = 0; k <= 20; ++k) {
        const float s = __fmul_rn(s0, __fdiv_rn((float)(90 + k), 100.0f));
        float ss, mm = 0.0f;
        if constexpr (P::SYM) {
            float num = 0.0f, den = 0.0f;
            for (int l = 0; l < P::G; ++l) {
                const float q = (float)cr(__fdiv_rn(x[l], s), P::LO, P::HI);
                const float aq = __fmul_rn(a[l], q);
                num = __fadd_rn(num, __fmul_rn(aq, x[l]));
                den = __fadd_rn(den, __fmul_rn(aq, q));
            }
            if (!(den > 0.0f)) continue;
            ss = __fdiv_rn(num, den);
        } else {
            float Sa = 0.0f, Sq = 0.0f, Sqq = 0.0f, Sw = 0.0f, Swq = 0.0f;
            for (int l = 0; l < P::G; ++l) {
                const float q = (float)cr(__fdiv_rn(__fadd_rn(x[l], m0), s), P::LO, P::HI);
                const float aq = __fmul_rn(a[l], q);
                Sa = __fadd_rn(Sa, a[l]);
                Sq = __fadd_rn(Sq, aq);
                Sqq = __fadd_rn(Sqq, __fmul_rn(aq, q));
                Sw = __fadd_rn(Sw, __fmul_rn(a[l], x[l]));
                Swq = __fadd_rn(Swq, __fmul_rn(aq, x[l]));
            }
            const float det = __fsub_rn(__fmul_rn(Sqq, Sa), __fmul_rn(Sq, Sq));
            if (!(det > 0.0f)) continue;
            ss = __fdiv_rn(__fsub_rn(__fmul_rn(Swq, Sa), __fmul_rn(Sq, Sw)), det);
            mm = __fdiv_rn(__fsub_rn(__fmul_rn(Swq, Sq), __fmul_rn(Sqq, Sw)), det);
            if (!(ss > 0.0f) || !(mm >= 0.0f)) continue;
        }
        // Weighted error of this candidate (codes rounded again with s, m0).
        float e = 0.0f;
        for (int l = 0; l < P::G; ++l) {
            const float q = P::SYM ? (float)cr(__fdiv_rn(x[l], s), P::LO, P::HI)
                                   : (float)cr(__fdiv_rn(__fadd_rn(x[l], m0), s), P::LO, P::HI);
            const float r = __fsub_rn(x[l], __fsub_rn(__fmul_rn(ss, q), mm));
            e = __fadd_rn(e, __fmul_rn(a[l], __fmul_rn(r, r)));
        }
        if (e < best) {
            best = e;
            s_out = ss;
            m_out = mm;
        }
    }
}

// Step 2: the block bytes from per-group (s, m), the plain assembly.
template <int T>
__device__ void assemble(const float* x, const float* sg, const float* mg, uint8_t* b) {
    using F = Fmt<T>;
    for (int i = 0; i < F::BB; ++i) b[i] = 0;
    if constexpr (T == T_Q8_0 || T == T_Q5_0 || T == T_Q4_0) {
        constexpr int off = T == T_Q8_0 ? 0 : (T == T_Q5_0 ? 16 : 8);
        constexpr int lo = T == T_Q8_0 ? -128 : 0, hi = T == T_Q8_0 ? 127 : (T == T_Q5_0 ? 31 : 15);
        const uint32_t db = h16(sg[0]);
        const float d = f16(db);
        b[0] = (uint8_t)db;
        b[1] = (uint8_t)(db >> 8);
        uint32_t qh = 0;
        for (int l = 0; l < 32; ++l) {
            const int q = d > 0.0f ? cr(__fdiv_rn(x[l], d), lo - off, hi - off) + off : off;
            if constexpr (T == T_Q8_0) {
                b[2 + l] = (uint8_t)(int8_t)q;
            } else {
                const int base = T == T_Q5_0 ? 6 : 2;
                b[base + (l & 15)] |= (uint8_t)((q & 15) << (4 * (l >> 4)));
                if (T == T_Q5_0) qh |= (uint32_t)(q >> 4) << l;
            }
        }
        if constexpr (T == T_Q5_0)
            for (int k = 0; k < 4; ++k) b[2 + k] = (uint8_t)(qh >> (8 * k));
    } else if constexpr (T == T_Q6_K || T == T_Q3_K) {
        constexpr bool six = T == T_Q6_K;
        float maxs = 0.0f;
        for (int g = 0; g < 16; ++g)
            if (sg[g] > maxs) maxs = sg[g];
        const uint32_t db = h16(__fdiv_rn(maxs, six ? 127.0f : 31.0f));
        const float d = f16(db);
        for (int g = 0; g < 16; ++g) {
            const int sc = d > 0.0f ? cr(__fdiv_rn(sg[g], d), six ? -128 : -32, six ? 127 : 31) : 0;
            const float ds = __fmul_rn(d, (float)sc);
            if constexpr (six) {
                b[192 + g] = (uint8_t)(int8_t)sc;
            } else {
                const int v = sc + 32;
                b[96 + (g & 7)] |= (uint8_t)((v & 15) << (4 * (g >> 3)));
                b[104 + (g & 3)] |= (uint8_t)((v >> 4) << (2 * (g >> 2)));
            }
            for (int l = 0; l < 16; ++l) {
                const int n = 16 * g + l, t = n >> 7, r = n & 127, j = r >> 5, li = n & 31;
                if constexpr (six) {
                    const int q = ds != 0.0f ? cr(__fdiv_rn(x[n], ds), -32, 31) + 32 : 32;
                    b[64 * t + li + 32 * (j & 1)] |= (uint8_t)(j < 2 ? (q & 15) : (q & 15) << 4);
                    b[128 + 32 * t + li] |= (uint8_t)((q >> 4) << (2 * j));
                } else {
                    const int q = ds != 0.0f ? cr(__fdiv_rn(x[n], ds), -4, 3) : 0;
                    const int hb = q >= 0, lo2 = hb ? q : q + 4;
                    b[32 + 32 * t + li] |= (uint8_t)(lo2 << (2 * j));
                    b[li] |= (uint8_t)(hb << (4 * t + j));
                }
            }
        }
        const int dpos = six ? 208 : 108;
        b[dpos] = (uint8_t)db;
        b[dpos + 1] = (uint8_t)(db >> 8);
    } else {   // Q4_K, Q5_K (32-weight sub-blocks), Q2_K (16-weight groups)
        constexpr bool two = T == T_Q2_K;
        constexpr int G = two ? 16 : 32, NG = two ? 16 : 8, top = T == T_Q5_K ? 31 : (two ? 3 : 15);
        constexpr int smax = two ? 15 : 63;
        float maxsc = 0.0f, maxm = 0.0f;
        for (int g = 0; g < NG; ++g) {
            if (sg[g] > maxsc) maxsc = sg[g];
            if (mg[g] > maxm) maxm = mg[g];
        }
        const uint32_t db = h16(__fdiv_rn(maxsc, (float)smax)), dmb = h16(__fdiv_rn(maxm, (float)smax));
        const float d = f16(db), dmin = f16(dmb);
        int sc[16], mn[16];
        for (int g = 0; g < NG; ++g) {
            sc[g] = d > 0.0f ? cr(__fdiv_rn(sg[g], d), 0, smax) : 0;
            mn[g] = dmin > 0.0f ? cr(__fdiv_rn(mg[g], dmin), 0, smax) : 0;
            const float ds = __fmul_rn(d, (float)sc[g]), dm = __fmul_rn(dmin, (float)mn[g]);
            for (int l = 0; l < G; ++l) {
                const int n = G * g + l;
                const int q = ds > 0.0f ? cr(__fdiv_rn(__fadd_rn(x[n], dm), ds), 0, top) : 0;
                if constexpr (two) {
                    const int t = n >> 7, j = (n & 127) >> 5;
                    b[16 + 32 * t + (n & 31)] |= (uint8_t)(q << (2 * j));
                } else {
                    const int c = n >> 6, h = (n >> 5) & 1, li = n & 31;
                    const int qs = T == T_Q5_K ? 48 : 16;
                    b[qs + 32 * c + li] |= (uint8_t)((q & 15) << (4 * h));
                    if (T == T_Q5_K) b[16 + li] |= (uint8_t)((q >> 4) << (2 * c + h));
                }
            }
        }
        if constexpr (two) {
            for (int g = 0; g < 16; ++g) b[g] = (uint8_t)(sc[g] | (mn[g] << 4));
            b[80] = (uint8_t)db;
            b[81] = (uint8_t)(db >> 8);
            b[82] = (uint8_t)dmb;
            b[83] = (uint8_t)(dmb >> 8);
        } else {
            for (int j = 0; j < 4; ++j) {
                b[4 + j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
                b[8 + j] = (uint8_t)(mn[j] | ((mn[j + 4] >> 4) << 6));
                b[12 + j] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
            }
            b[0] = (uint8_t)db;
            b[1] = (uint8_t)(db >> 8);
            b[2] = (uint8_t)dmb;
            b[3] = (uint8_t)(dmb >> 8);
        }
    }
}

// Step 3: weighted error of an encoded block (its weights through the
// shared half decoders), per group then over groups.
template <int T>
__device__ float weighted_error(const uint8_t* b, const float* x, const float* a) {
    using F = Fmt<T>;
    constexpr int G = Geo<T>::G;
    float w[256];
    for (int u = 0; u < F::UPB; ++u)
        for (int h = 0; h < 2; ++h) {
            float v[16];
            dequant_half<T>(b, u, h, v);
            for (int i = 0; i < 16; ++i) w[F::koff(u, h) + i] = v[i];
        }
    float total = 0.0f;
    for (int g = 0; g < F::BE / G; ++g) {
        float e = 0.0f;
        for (int l = 0; l < G; ++l) {
            const float r = __fsub_rn(x[G * g + l], w[G * g + l]);
            e = __fadd_rn(e, __fmul_rn(a[G * g + l], __fmul_rn(r, r)));
        }
        total = __fadd_rn(total, e);
    }
    return total;
}

template <int T>
__global__ void __launch_bounds__(128) quantize_imatrix_kernel(const float* __restrict__ w, const float* __restrict__ imp,
                                                               int64_t nblocks, int64_t nb_row, uint8_t* __restrict__ out) {
    using F = Fmt<T>;
    constexpr int G = Geo<T>::G, NG = F::BE / G;
    const int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (blk >= nblocks) return;
    const int64_t bi = blk % nb_row;
    const float* x = w + blk * F::BE;      // rows are consecutive blocks
    const float* a = imp + bi * F::BE;
    float sg[16], mg[16];
    alignas(16) uint8_t plain[F::BB + 16], mine[F::BB + 16];
    for (int g = 0; g < NG; ++g) group_params<T>(x + G * g, a + G * g, true, sg[g], mg[g]);
    assemble<T>(x, sg, mg, plain);
    for (int g = 0; g < NG; ++g) group_params<T>(x + G * g, a + G * g, false, sg[g], mg[g]);
    assemble<T>(x, sg, mg, mine);
    const float ep = weighted_error<T>(plain, x, a), em = weighted_error<T>(mine, x, a);
    const uint8_t* src = em <= ep ? mine : plain;
    uint8_t* o = out + blk * F::BB;
    for (int i = 0; i < F::BB; ++i) o[i] = src[i];
}

template <int T>
cudaError_t launch_t(const float* w, const float* imp, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t s) {
    const int64_t nb_row = cols / Fmt<T>::BE, nblocks = rows * nb_row;
    if (nblocks == 0) return cudaSuccess;
    const int64_t grid = (nblocks + 127) / 128;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quantize_imatrix_kernel<T><<<(unsigned)grid, 128, 0, s>>>(w, imp, nblocks, nb_row, out);
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
