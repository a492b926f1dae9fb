// qk_gemv5.cu -- the decode GEMV (one activation row): y[n] = sum_k w[n, k] x[k].
//
// Token generation streams every packed weight once per token and is bound
// by memory bandwidth ("12 -- llama.cpp / GGUF", performance model; "Local
// LLM inference": dequantize inside the dot product).  Layout of the work:
//   * Two CTAs per SM (8 warps each, at most 112 KB of shared memory each):
//     sixteen warps per SM hide the latency of the copies and of the integer
//     dot products.  (One CTA per SM, leaving room for the next GEMV's CTAs
//     to start early, measured slower: 8 warps do not keep up.)
//   * A CTA owns a contiguous range of rows and all of K.  It converts the
//     activation vector into the three-limb fixed-point form (qk_lanes.cuh)
//     in its own shared memory, after the weights of its first rows have
//     already been requested, so no separate prep kernel sits between two
//     GEMVs.
//   * The CTA's work is the list of (K slice, row) units, slice-major; warp w
//     takes the w-th eighth of the list.  A warp streams its units' row
//     segments (the aligned-down 16-byte window of each) with 16-byte
//     cp.async copies into its own ring of row slots and parses them there;
//     a lane keeps the limbs of its 64 weights of the current slice in
//     registers and reloads them from shared memory only when the slice
//     changes.  Rows are taken in pairs (two independent dot products, one
//     shuffle reduction).
//   * The ring's copies mark the weight lines evict-first in L2 (each byte
//     is read once).
//   * Each unit's dot goes to a shared array of partials [slice][row]; after
//     a CTA barrier the partials of a row are added in slice order, so the
//     result does not depend on timing.
// Nothing here waits on a flag or an mbarrier: cp.async groups and CTA
// barriers only.
#include <algorithm>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_lanes.cuh"
#include "qk_ptx.cuh"

namespace qk {
namespace gv5 {
using namespace gv;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSmemBudget = 112 * 1024;   // two CTAs per SM
constexpr int kCtasPerSm = 2;
constexpr int kRedFloats = 2048;          // partial sums per reduction chunk, at most
constexpr int kMaxPairs = 4;              // ring depth per warp in row pairs, at most
constexpr int kMinPairs = 2;

template <int T> struct Cfg {
    static constexpr int BB = Fmt<T>::BB, BE = Fmt<T>::BE;
    static constexpr int KB = kKR / BE;                      // blocks per row segment
    static constexpr int SEG = KB * BB;                      // bytes per row segment
    static constexpr int SLOT = (SEG + 32 + 15) / 16 * 16;   // alignment remainder + read slack
};

constexpr int kMaxGroup = QK_GEMV_BATCH_MAX;

// One launch serves up to kMaxGroup matrices that share x (and type and
// K): matrix i owns CTAs [cta0[i], cta0[i+1]).
struct Args {
    const float* x;
    int64_t cols;
    uint32_t row_bytes;
    int n;               // matrices
    int nsl;             // K slices
    int chunk;           // rows per reduction chunk (chunk * nsl <= kRedFloats)
    uint32_t off_ring, off_red;
    const uint8_t* W[kMaxGroup];
    float* y[kMaxGroup];
    int64_t rows[kMaxGroup];
    int64_t rows_q[kMaxGroup];   // rows / CTAs of the matrix
    int rows_r[kMaxGroup];       // its first rows_r CTAs take one row more
    int cta0[kMaxGroup + 1];
};

// Byte k of each of y0..y3, as one word.
template <int k>
__device__ __forceinline__ uint32_t gather_byte(uint32_t y0, uint32_t y1, uint32_t y2, uint32_t y3) {
    constexpr uint32_t sel = (uint32_t)k | ((uint32_t)(k + 4) << 4);
    return __byte_perm(__byte_perm(y0, y1, sel), __byte_perm(y2, y3, sel), 0x5410);
}

// The activation vector as limbs in shared memory, in the per-32-block
// layout the lane decoders read: a[32] b[32] c[32], then {s, sum of x[0..15],
// sum of x[16..31], sum of x}.  Two threads per block, sixteen elements each.
// s = max|x| / (127 * 65536) and X = round(x * (1/s)), with the reciprocal
// from the fast divide (relative error ~2^-22, far inside the GEMV
// tolerance; s * X reproduces x to that error).  |X| stays within a few
// units of 127 * 65536, so X + 0x808080 lies in [0, 2^24) and its bytes
// minus 128 are the balanced base-256 digits c (byte 0), b (byte 1),
// a (byte 2) of X, each in [-128, 127].
__device__ __forceinline__ void prep_x(const float* __restrict__ x, int64_t nxb, uint8_t* xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, hh = lane & 1;
    const int ntask = (int)nxb * 2;
    // Whole warps iterate together (the shuffles need every lane).
    for (int qb = warp * 32; qb < ntask; qb += kThreads) {
        const int q = qb + lane;
        const bool ok = q < ntask;
        const int jb = q >> 1;
        float v[16];
        if (ok) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 u = __ldg(reinterpret_cast<const float4*>(x) + 4 * q + k);
                v[4 * k] = u.x; v[4 * k + 1] = u.y; v[4 * k + 2] = u.z; v[4 * k + 3] = u.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float s = amax * (1.0f / kXMax);
        const float inv = amax > 0.0f ? __fdividef(kXMax, amax) : 0.0f;
        uint32_t Y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) Y[i] = (uint32_t)(__float2int_rn(v[i] * inv) + 0x808080);
        float half = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i += 4) half += (v[i] + v[i + 1]) + (v[i + 2] + v[i + 3]);
        const float other = __shfl_xor_sync(0xffffffffu, half, 1);   // the block's other half
        if (ok) {
            uint8_t* o = xs + jb * kXBytes + 16 * hh;
            uint4 w[3];
            uint32_t* wv = reinterpret_cast<uint32_t*>(w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wv[i] = gather_byte<2>(Y[4 * i], Y[4 * i + 1], Y[4 * i + 2], Y[4 * i + 3]) ^ 0x80808080u;
                wv[4 + i] = gather_byte<1>(Y[4 * i], Y[4 * i + 1], Y[4 * i + 2], Y[4 * i + 3]) ^ 0x80808080u;
                wv[8 + i] = gather_byte<0>(Y[4 * i], Y[4 * i + 1], Y[4 * i + 2], Y[4 * i + 3]) ^ 0x80808080u;
            }
            *reinterpret_cast<uint4*>(o) = w[0];
            *reinterpret_cast<uint4*>(o + 32) = w[1];
            *reinterpret_cast<uint4*>(o + 64) = w[2];
            if (hh == 0)
                *reinterpret_cast<float4*>(xs + jb * kXBytes + 96) = make_float4(s, half, other, half + other);
        }
    }
}

// The lane's two x-blocks of slice `sl` from the shared limbs (zero past the
// end of x: such lanes own no weights of the slice).
__device__ __forceinline__ void load_x_slice(const uint8_t* xs, int sl, int j0, int j1, int64_t nxb, XL& x) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t xb = (int64_t)sl * kXB + (j == 0 ? j0 : j1);
        uint4 v[7];
        if (xb < nxb) {
#pragma unroll
            for (int q = 0; q < 7; ++q) v[q] = lds128(xs + xb * kXBytes + 16 * q);
        } else {
#pragma unroll
            for (int q = 0; q < 7; ++q) v[q] = make_uint4(0u, 0u, 0u, 0u);
        }
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

// Copies a row's bytes that lie past the last full 16 bytes of W (the
// matrix's final row) into its slot; `rel` is the row segment's offset from
// `base`, `slot` its slot.
__device__ __forceinline__ void tail_fill(uint8_t* slot, const uint8_t* base, uint32_t rel, uint32_t seglen,
                                          uint32_t lim, int lane) {
    uint8_t* sbase = slot - (rel & ~15u);
    for (uint32_t bb = max(rel, lim) + lane; bb < rel + seglen; bb += 32) sbase[bb] = base[bb];
    __syncwarp();
}

// NP = ring depth in row pairs (one cp.async group per pair).
// SWI: one matrix pair, W[0] = gate and W[1] = up of the same shape, y[0] = h
// = SiLU(gate x) * (up x).
template <int T, int NP, bool SWI>
__global__ void __launch_bounds__(kThreads, 2) gemv5_kernel(const Args p) {
    using C = Cfg<T>;
    constexpr int NIT = ((C::SEG + 30) / 16 + 31) / 32;   // 16-byte copies per lane per row segment, at most
    constexpr uint32_t PAIR = 2u * C::SLOT;
    constexpr uint32_t RING = NP * PAIR;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + p.off_ring + (uint32_t)warp * RING;
    const uint32_t ring_lane_s = smem_u32(ring) + 16u * lane;   // this lane's copy destination, slot 0
    float* red = reinterpret_cast<float*>(smem + p.off_red);
    // My matrix (constant indices only: no local copy of the parameters).
    const uint8_t* Wm = p.W[0];
    float* ym = p.y[0];
    int64_t rows = p.rows[0], rq = p.rows_q[0];
    int rr = p.rows_r[0], bx = (int)blockIdx.x;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (i < p.n && (int)blockIdx.x >= p.cta0[i]) {
            Wm = p.W[i];
            ym = p.y[i];
            rows = p.rows[i];
            rq = p.rows_q[i];
            rr = p.rows_r[i];
            bx = (int)blockIdx.x - p.cta0[i];
        }
    const int64_t total16 = (rows * (int64_t)p.row_bytes) & ~(int64_t)15;
    const int64_t r_begin = bx * rq + min(bx, rr);
    const int64_t r_end = r_begin + rq + (bx < rr ? 1 : 0);
    const int64_t nb = p.cols / C::BE, nxb = p.cols / 32;
    const uint32_t rb = p.row_bytes;
    const Lane<T> L(lane);
    const Q4KFast F(lane);
    int j0, j1;
    L.xblocks(lane, j0, j1);
    const uint64_t pol = policy_evict_first();
    pdl_launch_dependents();
    auto seg_len = [&](int s) -> uint32_t {   // bytes of one row's segment of slice s
        return (uint32_t)(min((int64_t)C::KB, nb - (int64_t)s * C::KB) * C::BB);
    };

    bool prepped = false;
    // SwiGLU: each chunk of rows is walked twice, through the gate matrix and
    // then the up matrix; the gate results wait in h (written and read back
    // by the same thread) until the up pass finishes the row.
    constexpr int npass = SWI ? 2 : 1;
    for (int64_t cb = r_begin; cb < r_end; cb += p.chunk)
    for (int pass = 0; pass < npass; ++pass) {
        const int nrc = (int)min((int64_t)p.chunk, r_end - cb);
        const int npr = (nrc + 1) >> 1;                 // row pairs per slice (the last may be single)
        const int U = npr * p.nsl;
        const int u0 = (int)((int64_t)warp * U / kWarps);
        const int nu = (int)((int64_t)(warp + 1) * U / kWarps) - u0;
        // 32-bit byte offsets relative to an aligned base at the chunk's first row.
        const int64_t cboff = cb * (int64_t)rb;
        const uint8_t* base = (SWI && pass ? p.W[1] : Wm) + (cboff & ~(int64_t)15);
        const uint8_t* gl = base + 16 * lane;
        const uint32_t mis = (uint32_t)(cboff & 15);
        const int64_t lim64 = total16 - (cboff & ~(int64_t)15);
        const uint32_t lim = lim64 > 0xFFFFFFF0ll ? 0xFFFFFFF0u : (uint32_t)lim64;   // copy limit

        // Issue cursor: my pair ni is (slice is, pair ip) at byte offset rel_i
        // (its first row); one cp.async group per pair (an empty one past my
        // last pair).
        int ni = 0, is = u0 / npr, ip = u0 - is * npr;
        uint32_t rel_i = mis + 2u * ip * rb + (uint32_t)is * C::SEG;
        uint32_t len_i = seg_len(is), ioff = 0;
        auto copy_row = [&](uint32_t rel, uint32_t sd) {
            const uint32_t a = rel & ~15u;
            const uint32_t e = min((rel + len_i + 15u) & ~15u, lim);
            const uint32_t n = e > a ? e - a : 0u;   // bytes to copy
            const uint8_t* g = gl + a;
#pragma unroll
            for (int k = 0; k < NIT; ++k) cp_async16_if_lt(sd + 512u * k, g + 512 * k, pol, 16u * lane + 512u * k, n);
        };
        auto issue_next = [&]() {
            if (ni < nu) {
                copy_row(rel_i, ring_lane_s + ioff);
                if (2 * ip + 1 < nrc) copy_row(rel_i + rb, ring_lane_s + ioff + C::SLOT);
                rel_i += 2u * rb;
                if (++ip == npr) {
                    ip = 0;
                    ++is;
                    rel_i = mis + (uint32_t)is * C::SEG;
                    len_i = seg_len(is);
                }
            }
            cp_async_commit();
            ++ni;
            ioff += PAIR;
            if (ioff == RING) ioff = 0;
        };
        // One pair's copies overlap the previous kernel; the rest wait until
        // x (which may be that kernel's output) is in shared memory, so that
        // x's loads do not queue behind them.
        issue_next();
        if (!prepped) {
            pdl_wait_prior();
            prep_x(p.x, nxb, smem);
            prepped = true;
        }
        __syncthreads();   // limbs visible to every warp
#pragma unroll
        for (int i = 1; i < NP - 1; ++i) issue_next();

        // Consume cursor: my pair j is (slice cs, pair cp) at offset rel_c, slot coff.
        int cs = u0 / npr, cp = u0 - cs * npr, xsl = -1, nblk = 0;
        uint32_t rel_c = mis + 2u * cp * rb + (uint32_t)cs * C::SEG, coff = 0, seglen = 0;
        bool lv = false;
        XL xr;
        float s0 = 0.0f, s1 = 0.0f;
        for (int j = 0; j < nu; ++j) {
            issue_next();                 // pair j + NP - 1
            cp_async_wait<NP - 1>();      // pair j has landed (my copies)
            __syncwarp();                 // ... and every lane's
            if (cs != xsl) {
                load_x_slice(smem, cs, j0, j1, nxb, xr);
                xsl = cs;
                s0 = xr.meta[0].x;
                s1 = xr.meta[1].x;
                nblk = (int)min((int64_t)C::KB, nb - (int64_t)cs * C::KB);
                seglen = (uint32_t)nblk * C::BB;
                lv = L.valid(nblk);
            }
            // A single last row is paired with itself (its second result is dropped).
            const bool two = 2 * cp + 1 < nrc;
            uint8_t* slot0 = ring + coff;
            uint8_t* slot1 = two ? slot0 + C::SLOT : slot0;
            const uint32_t rel1 = two ? rel_c + rb : rel_c;
            if (rel1 + seglen > lim) {   // only the matrix's final rows
                tail_fill(slot0, base, rel_c, seglen, lim, lane);
                if (two) tail_fill(slot1, base, rel1, seglen, lim, lane);
            }
            float v0 = 0.0f, v1 = 0.0f;
            if (lv) {
                v0 = row_dot<T>(L, F, slot0 + (rel_c & 15u), xr, nblk, s0, s1);
                v1 = row_dot<T>(L, F, slot1 + (rel1 & 15u), xr, nblk, s0, s1);
            }
            // Two-row butterfly: lanes 0-15 end with row 2cp, lanes 16-31 with 2cp + 1.
            const bool upper = lane & 16;
            float keep = upper ? v1 : v0;
            keep += __shfl_xor_sync(0xffffffffu, upper ? v0 : v1, 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
            if ((lane & 15) == 0 && (!upper || two)) red[cs * nrc + 2 * cp + (upper ? 1 : 0)] = keep;
            __syncwarp();   // the slots are read before they are refilled
            coff += PAIR;
            if (coff == RING) coff = 0;
            rel_c += 2u * rb;
            if (++cp == npr) {
                cp = 0;
                ++cs;
                rel_c = mis + (uint32_t)cs * C::SEG;
            }
        }
        cp_async_wait<0>();
        __syncthreads();
        for (int t = threadIdx.x; t < nrc; t += kThreads) {
            float acc = 0.0f;
            for (int s = 0; s < p.nsl; ++s) acc += red[s * nrc + t];
            if (!SWI || pass == 0) {
                ym[cb + t] = acc;
            } else {   // h = SiLU(g) * u, SiLU(g) = g / (1 + e^-g)
                const float g = ym[cb + t];
                ym[cb + t] = g / (1.0f + expf(-g)) * acc;
            }
        }
        __syncthreads();   // partials consumed before the next chunk writes them
    }
}

}  // namespace gv5

namespace {
template <int T>
constexpr int slot_bytes() { return gv5::Cfg<T>::SLOT; }

int slot_of(int type) {
    switch (type) {
    case T_Q4_K: return slot_bytes<T_Q4_K>();
    case T_Q6_K: return slot_bytes<T_Q6_K>();
    case T_Q8_0: return slot_bytes<T_Q8_0>();
    case T_Q5_0: return slot_bytes<T_Q5_0>();
    case T_Q4_0: return slot_bytes<T_Q4_0>();
    case T_Q5_K: return slot_bytes<T_Q5_K>();
    case T_Q2_K: return slot_bytes<T_Q2_K>();
    case T_Q3_K: return slot_bytes<T_Q3_K>();
    }
    return 0;
}

int64_t nsl_of(int type, int64_t cols) {
    const int be = (type == T_Q8_0 || type == T_Q5_0 || type == T_Q4_0) ? 32 : 256;
    const int64_t nb = cols / be, kb = gv::kKR / be;
    return (nb + kb - 1) / kb;
}

struct Plan5 {
    int grid = 0, np = 0, chunk = 0, nsl = 0;
    int64_t rows_q[gv5::kMaxGroup] = {}, rows_r[gv5::kMaxGroup] = {};
    int cta0[gv5::kMaxGroup + 1] = {};
    uint32_t off_ring = 0, off_red = 0, smem = 0;
};

// CTAs in proportion to each matrix's rows (at least one per non-empty
// matrix, at most one per row), ring depth from what shared memory is left.
Plan5 plan5(int type, int n, const int64_t* rows, int64_t cols, int sms) {
    Plan5 p;
    const int slot = slot_of(type);
    if (slot == 0 || n < 1 || n > gv5::kMaxGroup || cols <= 0) return p;
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += std::max<int64_t>(rows[i], 0);
    if (total == 0) return p;
    p.nsl = (int)nsl_of(type, cols);
    if (p.nsl > gv5::kRedFloats) return Plan5{};
    const int64_t G = (int64_t)gv5::kCtasPerSm * std::max(sms, 1);
    int64_t per_cta = 0, g0 = 0;
    for (int i = 0; i < n; ++i) {
        p.cta0[i] = (int)g0;
        if (rows[i] <= 0) continue;
        const int64_t g = std::max<int64_t>(1, std::min<int64_t>(rows[i], (G * rows[i] + total / 2) / total));
        p.rows_q[i] = rows[i] / g;
        p.rows_r[i] = rows[i] % g;
        per_cta = std::max<int64_t>(per_cta, p.rows_q[i] + (p.rows_r[i] > 0 ? 1 : 0));
        g0 += g;
    }
    for (int i = n; i <= gv5::kMaxGroup; ++i) p.cta0[i] = (int)g0;
    p.grid = (int)g0;
    p.chunk = (int)std::min<int64_t>(per_cta, gv5::kRedFloats / p.nsl);
    const int64_t xbytes = (cols / 32) * gv::kXBytes;          // 16-byte multiple
    const int64_t red = ((int64_t)p.chunk * p.nsl * 4 + 15) & ~(int64_t)15;
    const int64_t ring0 = (xbytes + red + 127) & ~(int64_t)127;   // the ring starts on a 128-byte line
    const int64_t room = gv5::kSmemBudget - ring0;
    const int64_t np = room / ((int64_t)gv5::kWarps * 2 * slot);
    if (np < gv5::kMinPairs) return Plan5{};
    p.np = (int)std::min<int64_t>(np, gv5::kMaxPairs);
    p.off_red = (uint32_t)xbytes;
    p.off_ring = (uint32_t)ring0;
    p.smem = (uint32_t)(ring0 + (int64_t)gv5::kWarps * p.np * 2 * slot);
    return p;
}

template <int T, int NP, bool SWI>
cudaError_t launch5_np(const gv5::Args& a, const Plan5& pl, cudaStream_t s) {
    auto kern = gv5::gemv5_kernel<T, NP, SWI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gv5::kSmemBudget);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(gv5::kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int T, bool SWI>
cudaError_t launch5_t(const gv5::Args& a, const Plan5& pl, cudaStream_t s) {
    switch (pl.np) {
    case 2: return launch5_np<T, 2, SWI>(a, pl, s);
    case 3: return launch5_np<T, 3, SWI>(a, pl, s);
    default: return launch5_np<T, 4, SWI>(a, pl, s);
    }
}

template <bool SWI>
cudaError_t launch5_type(int type, const gv5::Args& a, const Plan5& pl, cudaStream_t s) {
    switch (type) {
    case T_Q4_K: return launch5_t<T_Q4_K, SWI>(a, pl, s);
    case T_Q6_K: return launch5_t<T_Q6_K, SWI>(a, pl, s);
    case T_Q8_0: return launch5_t<T_Q8_0, SWI>(a, pl, s);
    case T_Q5_0: return launch5_t<T_Q5_0, SWI>(a, pl, s);
    case T_Q4_0: return launch5_t<T_Q4_0, SWI>(a, pl, s);
    case T_Q5_K: return launch5_t<T_Q5_K, SWI>(a, pl, s);
    case T_Q2_K: return launch5_t<T_Q2_K, SWI>(a, pl, s);
    case T_Q3_K: return launch5_t<T_Q3_K, SWI>(a, pl, s);
    }
    return cudaErrorInvalidValue;
}

int64_t row_bytes_of(int type, int64_t cols) {
    switch (type) {
    case T_Q4_K: return cols / 256 * 144;
    case T_Q6_K: return cols / 256 * 210;
    case T_Q8_0: return cols / 32 * 34;
    case T_Q5_0: return cols / 32 * 22;
    case T_Q4_0: return cols / 32 * 18;
    case T_Q5_K: return cols / 256 * 176;
    case T_Q2_K: return cols / 256 * 84;
    case T_Q3_K: return cols / 256 * 110;
    }
    return 0;
}
}  // namespace

int gemv5_ring_pairs(int type, int n, const int64_t* rows, int64_t cols, int sms) {
    return plan5(type, n, rows, cols, sms).np;
}

cudaError_t launch_gemv5(int type, int n, const uint8_t* const* W, const int64_t* rows, int64_t cols, const float* x,
                         float* const* y, int sms, cudaStream_t s) {
    const Plan5 pl = plan5(type, n, rows, cols, sms);
    if (pl.np == 0) return cudaErrorInvalidValue;
    if (pl.grid == 0) return cudaSuccess;
    gv5::Args a = {};
    a.x = x;
    a.cols = cols;
    a.row_bytes = (uint32_t)row_bytes_of(type, cols);
    a.n = n;
    a.nsl = pl.nsl;
    a.chunk = pl.chunk;
    a.off_ring = pl.off_ring;
    a.off_red = pl.off_red;
    for (int i = 0; i < n; ++i) {
        a.W[i] = W[i];
        a.y[i] = y[i];
        a.rows[i] = rows[i];
        a.rows_q[i] = pl.rows_q[i];
        a.rows_r[i] = (int)pl.rows_r[i];
    }
    for (int i = 0; i <= gv5::kMaxGroup; ++i) a.cta0[i] = pl.cta0[i];
    return launch5_type<false>(type, a, pl, s);
}

cudaError_t launch_gemv5_swiglu(int type, const uint8_t* Wg, const uint8_t* Wu, int64_t rows, int64_t cols,
                                const float* x, float* h, int sms, cudaStream_t s) {
    const Plan5 pl = plan5(type, 1, &rows, cols, sms);
    if (pl.np == 0) return cudaErrorInvalidValue;
    if (pl.grid == 0) return cudaSuccess;
    gv5::Args a = {};
    a.x = x;
    a.cols = cols;
    a.row_bytes = (uint32_t)row_bytes_of(type, cols);
    a.n = 1;
    a.nsl = pl.nsl;
    a.chunk = pl.chunk;
    a.off_ring = pl.off_ring;
    a.off_red = pl.off_red;
    a.W[0] = Wg;
    a.W[1] = Wu;
    a.y[0] = h;
    a.rows[0] = rows;
    a.rows_q[0] = pl.rows_q[0];
    a.rows_r[0] = (int)pl.rows_r[0];
    for (int i = 0; i <= gv5::kMaxGroup; ++i) a.cta0[i] = pl.cta0[i];
    return launch5_type<true>(type, a, pl, s);
}


}  // namespace qk
