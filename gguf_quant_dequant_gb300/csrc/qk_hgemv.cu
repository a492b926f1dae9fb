// qk_hgemv.cu -- the decode GEMV on the tensor cores: y[n] = sum_k w[n, k] x[k]
// for one activation row, the batched form over matrices that share x
// (q/k/v, gate/up) and the fused SwiGLU gate.
//
// Token generation streams every packed weight once per token and is bound
// by memory bandwidth ("12 -- llama.cpp / GGUF", performance model; "Local
// LLM inference": dequantize inside the dot product).  The work per weight
// is kept small enough for the SMs to keep pace with HBM:
//   * the dot products run on the fp16 warp MMA (qk_hunits.cuh): 16 rows x
//     16 weights per instruction, codes converted to fp16 with one mask and
//     one exact add per two weights, x held as two fp16 terms (hi + lo);
//   * two CTAs per SM, each of eight consumer warps and one producer warp
//     (more warps would not help: the decode is bound by the SM's integer,
//     tensor and shared-memory pipes, not by latency);  A CTA owns
//     a contiguous range of rows (of one matrix) and all of K.  The producer
//     streams "stages" of 16 rows x 2048 weights into a shared-memory ring:
//     one bulk async copy per row segment (its aligned-down 16-byte window;
//     Q6_K rows of 11008 weights are 9030 bytes apart), completion counted on
//     the stage's full mbarrier, release on its empty mbarrier.  Every wait
//     is bounded in time.
//   * consumer warp w decodes unit w (256 weights) of each stage for the 16
//     rows, so the stage's K range is spread over the warps; stages go K
//     chunk by K chunk over the CTA's row tiles, so that a warp keeps its
//     unit of x in registers for all its tiles; partial sums of each row
//     collect in shared memory and are added in a fixed order
//     (deterministic);
//   * x is converted in each CTA's shared memory after the grid-dependency
//     wait (the previous kernel may produce it), while the producer already
//     streams weights: no separate prep kernel runs between two GEMVs.
#include <algorithm>
#include <type_traits>

#include "qk_formats.cuh"
#include "qk_hunits.cuh"
#include "qk_internal.h"
#include "qk_ptx.cuh"

namespace qk {
namespace hg {
using namespace hm;

constexpr int kCW = 8;                      // consumer warps
constexpr int kThreads = (kCW + 1) * 32;    // + one producer warp
constexpr int kTileRows = 16;               // rows per MMA tile
constexpr int kPartW = 4 * kTileRows;       // partial sums per (tile pass, token, warp): a row's four threads each
constexpr int kUnitW = 256;                 // weights per unit (16 rows x 256 weights: one warp's work item)
constexpr int kXBB = 128;                   // prepared bytes per x-block: 2 planes x 8 words x 8 bytes
constexpr int kMaxGroup = QK_GEMV_BATCH_MAX;
constexpr int kMinStages = 2, kMaxStages = 8;

struct Args {
    const float* x;
    int64_t cols;
    uint32_t row_bytes;
    int n;               // matrices (SwiGLU: 1, with W[1] the up matrix)
    int64_t ystride;     // elements between the outputs of consecutive tokens (MT > 1)
    int nxb;             // x-blocks of x (cols / 32)
    int nunits;          // units per row
    int nchunks;         // stages per row (per tile)
    int stages;          // ring depth
    uint32_t slot;       // bytes per row slot of a stage
    uint32_t off_xb, off_xm, off_xs, off_ring, off_bar, off_red;
    unsigned* status;
    const uint8_t* W[kMaxGroup];
    float* y[kMaxGroup];
    int64_t rows[kMaxGroup];
    int64_t rows_q[kMaxGroup];   // rows / CTAs of the matrix
    int rows_r[kMaxGroup];       // its first rows_r CTAs take one row more
    int cta0[kMaxGroup + 1];
};

// x -> B fragments in shared memory, one unit (256 elements, 8 x-blocks)
// at a time by the warp that uses it.  Local x-block j of the unit, plane h:
//   xb[(2j + h) * 64 + 8i] = half2(x_h[4i], x_h[4i+2]), half2(x_h[4i+1], x_h[4i+3])
// with x' = x * 2^-e, x_0 = fp16(x'), x_1 = fp16(x' - x_0); xm[j] = (sum of x
// over the block, 2^e, sum over its first 16 elements, over its last 16).
// e = 0 unless max|x| of the block reaches 2^15, then the block is scaled
// into [2^14, 2^15).  Lane l takes elements 8q .. 8q + 7 (q = l % 4) of
// local block l / 4; blocks past x are zero.
// The unit's x for lane `lane` (eight floats) copied into its 32-byte slot
// of `xs` without holding registers (cp.async; zeros past x).
__device__ __forceinline__ void load_unit_x(const float* __restrict__ x, int nxb, int u, int lane, float* xs) {
    const int j = 8 * u + (lane >> 2), q = lane & 3;
    float* d = xs + 8 * lane;
    if (j < nxb) {
        cp_async16(d, x + 32 * j + 8 * q);
        cp_async16(d + 4, x + 32 * j + 8 * q + 4);
    } else {
        *reinterpret_cast<float4*>(d) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        *reinterpret_cast<float4*>(d + 4) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
}
__device__ __forceinline__ void prep_unit_x(const float* xs, uint8_t* xb, float4* xm, int lane) {
    const int jl = lane >> 2, q = lane & 3;
    const float4 a = *reinterpret_cast<const float4*>(xs + 8 * lane), b = *reinterpret_cast<const float4*>(xs + 8 * lane + 4);
    const float amax_a = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
    float amax = fmaxf(amax_a, fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
    // The eight elements' sum by packed pair adds (any order: an fp32 block sum).
    const float2 s2 = __fadd2_rn(__fadd2_rn(make_float2(a.x, a.y), make_float2(a.z, a.w)),
                                 __fadd2_rn(make_float2(b.x, b.y), make_float2(b.z, b.w)));
    float sum = s2.x + s2.y;
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);           // sum of 16 elements (one half)
    const float other = __shfl_xor_sync(0xffffffffu, sum, 2);
    // Scale exponent: floor(log2 max|x|) - 14 when that is positive.
    const int ex = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
    const int e = max(0, ex - 14);
    const float down = __uint_as_float((uint32_t)(127 - e) << 23), up = __uint_as_float((uint32_t)(127 + e) << 23);
    // Words 2q and 2q+1: elements 8q + {0,2}, {1,3}, {4,6}, {5,7}; each pair
    // rounded to fp16 by one packed convert, its residual by another.
    constexpr int kPair[4][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}};
    // x' = x 2^-e on the loads' natural register pairs.
    const float2 s01 = __fmul2_rn(make_float2(a.x, a.y), make_float2(down, down));
    const float2 s23 = __fmul2_rn(make_float2(a.z, a.w), make_float2(down, down));
    const float2 s45 = __fmul2_rn(make_float2(b.x, b.y), make_float2(down, down));
    const float2 s67 = __fmul2_rn(make_float2(b.z, b.w), make_float2(down, down));
    const float xs8[8] = {s01.x, s01.y, s23.x, s23.y, s45.x, s45.y, s67.x, s67.y};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a0 = xs8[kPair[k][0]], b0 = xs8[kPair[k][1]];
        const __half2 h = __floats2half2_rn(a0, b0);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(a0 - hf.x, b0 - hf.y);   // x' - hi, exact
        hi[k] = *reinterpret_cast<const uint32_t*>(&h);
        lo[k] = *reinterpret_cast<const uint32_t*>(&l);
    }
    *reinterpret_cast<uint4*>(xb + jl * kXBB + 16 * q) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(xb + jl * kXBB + 64 + 16 * q) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (q == 0) xm[jl] = make_float4(sum + other, up, sum, other);
}

__device__ __forceinline__ void named_sync_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory"); }

// SWI: one matrix pair (W[0] gate, W[1] up, same shape), y[0] = h =
// SiLU(gate x) * (up x); each 16-row tile is walked through the gate matrix
// and then the up matrix.
//
// Order of the work: K chunks outermost, row tiles inside, so that a warp's
// B fragments (its unit of x) stay in registers for all the CTA's tiles of a
// chunk.  Each warp adds its partial sums of a (tile, row) into shared memory
// in chunk order; at the end the warps' partials of a row are added in warp
// order.  The result does not depend on timing.
template <int T, int MT, bool SWI>
__global__ void __launch_bounds__(kThreads, 2) hgemv_kernel(const Args p) {
    static_assert(!SWI || MT == 1, "the SwiGLU form takes one activation row");
    using U = HU<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + p.stages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + p.stages);
    // Partial sums [tile pass][token][kCW][64]: per warp, row g's sums of the
    // four threads of its group t at t * 8 + g, row g + 8's at 32 + t * 8 + g
    // (32 consecutive words for a warp's 32 lanes).
    float* part = reinterpret_cast<float*>(smem + p.off_red);
    uint8_t* xb = smem + p.off_xb;
    float4* xm = reinterpret_cast<float4*>(smem + p.off_xm);
    float* xst = reinterpret_cast<float*>(smem + p.off_xs);   // [warp][token][256] staged x
    uint8_t* ring = smem + p.off_ring;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // My matrix and rows.
    const uint8_t* Wm = p.W[0];
    float* ym = p.y[0];
    int64_t rows = p.rows[0], rq = p.rows_q[0];
    int rr = p.rows_r[0], bx = (int)blockIdx.x;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (!SWI && i < p.n && (int)blockIdx.x >= p.cta0[i]) {
            Wm = p.W[i];
            ym = p.y[i];
            rows = p.rows[i];
            rq = p.rows_q[i];
            rr = p.rows_r[i];
            bx = (int)blockIdx.x - p.cta0[i];
        }
    const int64_t r_begin = bx * rq + min(bx, rr);
    const int nrows = (int)(rq + (bx < rr ? 1 : 0));
    const int ntiles = (nrows + kTileRows - 1) / kTileRows;
    constexpr int npass = SWI ? 2 : 1;
    const uint32_t rb = p.row_bytes;
    const uint32_t CB = (uint32_t)kCW * U::UB;   // bytes of a full chunk (a multiple of 16)
    const uint32_t stage_bytes = kTileRows * p.slot;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kCW) {
        // ---------------- producer ----------------
        const uint64_t pol = policy_evict_first();
        const int64_t total16 = (rows * (int64_t)rb) & ~(int64_t)15;
        int it = 0, s = 0;
        uint32_t ph = 0;   // phase parity of stage s's barriers in this pass over the ring
        bool dead = false;
        for (int c = 0; c < p.nchunks && !dead; ++c) {
            const int64_t coff = (int64_t)c * CB;
            const int64_t len = min((int64_t)CB, (int64_t)rb - coff);
            for (int tile = 0; tile < ntiles && !dead; ++tile) {
                const int nr = min(kTileRows, nrows - tile * kTileRows);
                const int64_t off = (r_begin + tile * kTileRows + lane) * (int64_t)rb + coff;
                for (int pass = 0; pass < npass; ++pass, ++it) {
                    const uint8_t* Wp = (SWI && pass) ? p.W[1] : Wm;
                    if (it >= p.stages && !mbar_wait_abortable(&empty[s], ph ^ 1u, p.status, abort)) {
                        dead = true;
                        break;
                    }
                    uint8_t* st = ring + (uint32_t)s * stage_bytes;
                    uint32_t bytes = 0;
                    const int64_t a = off & ~(int64_t)15;
                    if (lane < nr) {
                        const int64_t e = min((off + len + 15) & ~(int64_t)15, total16);
                        bytes = e > a ? (uint32_t)(e - a) : 0u;
                        // Bytes past the last full 16 bytes of the matrix (its final row).
                        for (int64_t b = max(off, total16); b < off + len; ++b) st[lane * p.slot + (uint32_t)(b - a)] = Wp[b];
                    }
                    uint32_t total = bytes;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], total);
                    __syncwarp();
                    if (bytes) bulk_g2s(st + lane * p.slot, Wp + a, bytes, &full[s], pol);
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        if (dead) {
            // Let the copies already requested land before the CTA exits.
            for (int k = max(0, it - p.stages); k < it; ++k)
                mbar_wait_bounded(&full[k % p.stages], (uint32_t)(k / p.stages) & 1u, p.status);
        }
        return;
    }

    // ---------------- consumers ----------------
    const int ctid = threadIdx.x;
    const int g = lane >> 2, t = lane & 3;
    // This warp's partial sums start at zero (only this warp adds into them
    // until the final barrier).
    for (int i = lane; i < ntiles * npass * MT * kPartW; i += 32)
        part[((i >> 6) * kCW + warp) * kPartW + (i & 63)] = 0.0f;
    // This warp's prepared x: its unit of the current chunk, per token.
    uint8_t* xbw = xb + warp * MT * (8 * kXBB);
    float4* xmw = xm + warp * MT * 8;
    float* xsw = xst + warp * MT * 256;
    pdl_wait_prior();   // x may come from the previous kernel
#pragma unroll
    for (int m = 0; m < MT; ++m) load_unit_x(p.x + (int64_t)m * p.cols, p.nxb, warp, lane, xsw + m * 256);
    cp_async_commit();
    // B fragments: the thread whose column g belongs to its group t (g / 2 ==
    // t) reads plane g % 2 of the group's x-blocks; every other thread
    // supplies zeros.
    const bool owner = (g >> 1) == t;
    // Rows g and g + 8 of every tile start (row * row_bytes) mod 16 bytes
    // into their slots (a chunk is a multiple of 16 bytes; 16 rows move the
    // offset by a multiple of 16).
    const uint32_t o0 = g * p.slot + (uint32_t)(((r_begin + g) * (int64_t)rb) & 15) + warp * U::UB;
    const uint32_t o1 = (g + 8) * p.slot + (uint32_t)(((r_begin + g + 8) * (int64_t)rb) & 15) + warp * U::UB;
    const int units_last = p.nunits - (p.nchunks - 1) * kCW;
    int s = 0;
    uint32_t ph = 0;
    bool dead = false;
    for (int c = 0; c < p.nchunks; ++c) {
        const int u = c * kCW + warp;   // my unit of every row of the chunk
        const bool act = warp < (c == p.nchunks - 1 ? units_last : kCW);
        // One token: its B fragments for the chunk in registers; more: read
        // from shared memory step by step.
        using BP = typename std::conditional<MT == 1, BRegs, BSmem<MT>>::type;
        BP bp = {};
        float4 xm0[MT], xm1[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) xm0[m] = xm1[m] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        // Prepare this chunk's x (loaded one chunk ahead), then request the
        // next chunk's.
        cp_async_wait<0>();   // this lane's staged x of the chunk
        __syncwarp();         // every lane is done reading the previous unit's x
#pragma unroll
        for (int m = 0; m < MT; ++m) prep_unit_x(xsw + m * 256, xbw + m * (8 * kXBB), xmw + m * 8, lane);
        __syncwarp();
        if (c + 1 < p.nchunks) {
#pragma unroll
            for (int m = 0; m < MT; ++m) load_unit_x(p.x + (int64_t)m * p.cols, p.nxb, u + kCW, lane, xsw + m * 256);
            cp_async_commit();
        }
        if (act) {
            const uint32_t xo0 = (U::X0(t) * 2 + (g & 1)) * 64, xo1 = (U::X1(t) * 2 + (g & 1)) * 64;
            if constexpr (MT == 1) {
                if (owner) {
                    load_xb(xbw + xo0, bp.x0);
                    load_xb(xbw + xo1, bp.x1);
                }
            } else {
                bp.own = owner;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    bp.p[m][0] = xbw + m * (8 * kXBB) + xo0;
                    bp.p[m][1] = xbw + m * (8 * kXBB) + xo1;
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                xm0[m] = xmw[m * 8 + U::X0(t)];
                xm1[m] = xmw[m * 8 + U::X1(t)];
            }
        }
        const int nvb = min(8, p.nxb - 8 * u);
        for (int tile = 0; tile < ntiles; ++tile) {
            for (int pass = 0; pass < npass; ++pass) {
                if (!dead && !mbar_wait_abortable(&full[s], ph, p.status, abort)) dead = true;
                float y0[MT], y1[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) y0[m] = y1[m] = 0.0f;
                if (act && !dead) {
                    const uint8_t* st = ring + (uint32_t)s * stage_bytes;
                    run_unit<T, MT>(st + o0, st + o1, bp, xm0, xm1, t, nvb, y0, y1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (++s == p.stages) {
                    s = 0;
                    ph ^= 1u;
                }
                // Each thread keeps its own sums of rows g and g + 8 (the four
                // threads of a row are added at the end).
                if (act) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float* pp = part + (((tile * npass + pass) * MT + m) * kCW + warp) * kPartW + t * 8 + g;
                        pp[0] += y0[m];
                        pp[32] += y1[m];
                    }
                }
            }
        }
    }
    named_sync_consumers();
    if (dead) return;
    for (int i = ctid; i < nrows * MT; i += kCW * 32) {
        const int m = i / nrows, ri = i - m * nrows;
        const int tile = ri / kTileRows, r = ri % kTileRows;
        const float* pp = part + ((tile * npass) * MT + m) * kCW * kPartW + (r < 8 ? r : 24 + r);
        // Warps in order, the four threads of the row in order within each.
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kCW; ++w)
#pragma unroll
            for (int q = 0; q < 4; ++q) v += pp[w * kPartW + 8 * q];
        if (SWI) {   // h = SiLU(g) * u, SiLU(g) = g / (1 + e^-g)
            float uu = 0.0f;
#pragma unroll
            for (int w = 0; w < kCW; ++w)
#pragma unroll
                for (int q = 0; q < 4; ++q) uu += pp[(kCW + w) * kPartW + 8 * q];
            v = v / (1.0f + expf(-v)) * uu;
        }
        ym[(int64_t)m * p.ystride + r_begin + ri] = v;
    }
}

}  // namespace hg

namespace {

bool hg_supported(int type) { return type >= T_Q4_K && type <= T_Q3_K; }

int hg_block_bytes(int type) {
    switch (type) {
    case T_Q4_K: return 144;
    case T_Q6_K: return 210;
    case T_Q8_0: return 34;
    case T_Q5_0: return 22;
    case T_Q4_0: return 18;
    case T_Q5_K: return 176;
    case T_Q2_K: return 84;
    case T_Q3_K: return 110;
    }
    return 0;
}
int hg_block_elems(int type) { return (type == T_Q8_0 || type == T_Q5_0 || type == T_Q4_0) ? 32 : 256; }

// Two CTAs per SM: the rings of both (about 150 KB) keep enough copies in
// flight to cover the loaded HBM latency (about 3 us), and when one CTA of
// an SM finishes, the next launch's CTA (programmatic dependent launch)
// takes its place and starts streaming while the other still runs.
constexpr int64_t kSmemBudget = 113 * 1024;

struct PlanH {
    int grid = 0, stages = 0, nunits = 0, nchunks = 0, nxb = 0;
    uint32_t slot = 0, off_xb = 0, off_xm = 0, off_xs = 0, off_ring = 0, off_bar = 0, off_red = 0, smem = 0;
    int64_t rows_q[hg::kMaxGroup] = {}, rows_r[hg::kMaxGroup] = {};
    int cta0[hg::kMaxGroup + 1] = {};
};

// mt = activation rows (tokens) per launch; swiglu = the two-pass form.
PlanH planh(int type, int n, const int64_t* rows, int64_t cols, int sms, int mt, bool swiglu) {
    PlanH p;
    if (!hg_supported(type) || n < 1 || n > hg::kMaxGroup || cols <= 0 || mt < 1) return p;
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += std::max<int64_t>(rows[i], 0);
    if (total == 0) return p;
    const int BB = hg_block_bytes(type), BE = hg_block_elems(type);
    p.nxb = (int)(cols / 32);
    p.nunits = (int)((cols + hg::kUnitW - 1) / hg::kUnitW);
    // CTAs in proportion to each matrix's rows (at least one per non-empty
    // matrix, at most one per row).
    const int64_t G = 2 * (int64_t)std::max(sms, 1);
    int64_t g0 = 0, per_cta = 0;
    for (int i = 0; i < n; ++i) {
        p.cta0[i] = (int)g0;
        if (rows[i] <= 0) continue;
        const int64_t g = std::max<int64_t>(1, std::min<int64_t>(rows[i], (G * rows[i] + total / 2) / total));
        p.rows_q[i] = rows[i] / g;
        p.rows_r[i] = rows[i] % g;
        per_cta = std::max<int64_t>(per_cta, p.rows_q[i] + (p.rows_r[i] ? 1 : 0));
        g0 += g;
    }
    for (int i = n; i <= hg::kMaxGroup; ++i) p.cta0[i] = (int)g0;
    p.grid = (int)g0;
    // Layout: B fragments of each token, block sums of each token, partial
    // sums [tile pass][token][8 warps][64], mbarriers + abort word, ring.
    const int64_t ntp = (per_cta + hg::kTileRows - 1) / hg::kTileRows * (swiglu ? 2 : 1);
    // Each consumer warp prepares its own unit of x, per token.
    const int64_t xbb = (int64_t)mt * hg::kCW * 8 * hg::kXBB;
    const int64_t xmb = (int64_t)mt * hg::kCW * 8 * 16;
    const int64_t redb = ntp * mt * hg::kCW * hg::kPartW * 4;
    const int64_t barb = 2 * hg::kMaxStages * 8 + 16;
    const int64_t xsb = (int64_t)mt * hg::kCW * 256 * 4;   // staged x, 32 bytes per lane per token
    p.off_xb = 0;
    p.off_xm = (uint32_t)xbb;
    p.off_xs = (uint32_t)(xbb + xmb);
    p.off_red = (uint32_t)(xbb + xmb + xsb);
    p.off_bar = (uint32_t)((p.off_red + redb + 15) & ~(int64_t)15);
    p.off_ring = (uint32_t)((p.off_bar + barb + 127) & ~(int64_t)127);
    const int64_t UB = (int64_t)(hg::kUnitW / BE) * BB;
    const int64_t CB = hg::kCW * UB;
    // Room for the alignment remainder and word reads past the end, and a
    // stride of 16 mod 32 bytes: the 16-byte code loads of rows g and g + 1
    // then fall in different shared-memory banks.
    uint32_t slot = (uint32_t)(((CB + 15 + 15) & ~(int64_t)15) + 16);
    if (slot % 32 == 0) slot += 16;
    const int64_t stage = (int64_t)hg::kTileRows * slot;
    const int64_t ns = (kSmemBudget - p.off_ring) / stage;
    if (ns < hg::kMinStages) return PlanH{};
    p.slot = slot;
    p.nchunks = (p.nunits + hg::kCW - 1) / hg::kCW;
    p.stages = (int)std::min<int64_t>(ns, hg::kMaxStages);
    p.smem = (uint32_t)(p.off_ring + p.stages * stage);
    return p;
}

template <int T, int MT, bool SWI>
cudaError_t launch_h_t(const hg::Args& a, const PlanH& pl, cudaStream_t s) {
    auto kern = hg::hgemv_kernel<T, MT, SWI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(hg::kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int MT, bool SWI>
cudaError_t launch_h_type(int type, const hg::Args& a, const PlanH& pl, cudaStream_t s) {
    switch (type) {
    case T_Q4_K: return launch_h_t<T_Q4_K, MT, SWI>(a, pl, s);
    case T_Q6_K: return launch_h_t<T_Q6_K, MT, SWI>(a, pl, s);
    case T_Q8_0: return launch_h_t<T_Q8_0, MT, SWI>(a, pl, s);
    case T_Q5_0: return launch_h_t<T_Q5_0, MT, SWI>(a, pl, s);
    case T_Q4_0: return launch_h_t<T_Q4_0, MT, SWI>(a, pl, s);
    case T_Q5_K: return launch_h_t<T_Q5_K, MT, SWI>(a, pl, s);
    case T_Q2_K: return launch_h_t<T_Q2_K, MT, SWI>(a, pl, s);
    case T_Q3_K: return launch_h_t<T_Q3_K, MT, SWI>(a, pl, s);
    }
    return cudaErrorInvalidValue;
}

hg::Args make_args(int type, const PlanH& pl, int64_t cols, const float* x, unsigned* status) {
    hg::Args a = {};
    a.x = x;
    a.cols = cols;
    a.row_bytes = (uint32_t)(cols / hg_block_elems(type) * hg_block_bytes(type));
    a.nxb = pl.nxb;
    a.nunits = pl.nunits;
    a.nchunks = pl.nchunks;
    a.stages = pl.stages;
    a.slot = pl.slot;
    a.off_xb = pl.off_xb;
    a.off_xm = pl.off_xm;
    a.off_xs = pl.off_xs;
    a.off_ring = pl.off_ring;
    a.off_bar = pl.off_bar;
    a.off_red = pl.off_red;
    a.status = status;
    for (int i = 0; i <= hg::kMaxGroup; ++i) a.cta0[i] = pl.cta0[i];
    return a;
}
}  // namespace

bool hgemv_ok(int type, int n, const int64_t* rows, int64_t cols, int sms) {
    return planh(type, n, rows, cols, sms, 1, false).stages > 0;
}

cudaError_t launch_hgemv(int type, int n, const uint8_t* const* W, const int64_t* rows, int64_t cols, const float* x,
                         float* const* y, int sms, unsigned* status, cudaStream_t s) {
    const PlanH pl = planh(type, n, rows, cols, sms, 1, false);
    if (pl.stages == 0) return cudaErrorInvalidValue;
    if (pl.grid == 0) return cudaSuccess;
    hg::Args a = make_args(type, pl, cols, x, status);
    a.n = n;
    for (int i = 0; i < n; ++i) {
        a.W[i] = W[i];
        a.y[i] = y[i];
        a.rows[i] = rows[i];
        a.rows_q[i] = pl.rows_q[i];
        a.rows_r[i] = (int)pl.rows_r[i];
    }
    return launch_h_type<1, false>(type, a, pl, s);
}

cudaError_t launch_hgemv_tokens(int type, const uint8_t* W, int64_t rows, int64_t cols, const float* x, int64_t M,
                                float* y, int sms, unsigned* status, cudaStream_t s) {
    // Two activation rows per launch (the fp16 code conversion of a weight
    // is shared by both), one for an odd last row.
    for (int64_t m0 = 0; m0 < M;) {
        const int mt = (M - m0 >= 2 && planh(type, 1, &rows, cols, sms, 2, false).stages > 0) ? 2 : 1;
        const PlanH pl = planh(type, 1, &rows, cols, sms, mt, false);
        if (pl.stages == 0) return cudaErrorInvalidValue;
        hg::Args a = make_args(type, pl, cols, x + m0 * cols, status);
        a.n = 1;
        a.ystride = rows;
        a.W[0] = W;
        a.y[0] = y + m0 * rows;
        a.rows[0] = rows;
        a.rows_q[0] = pl.rows_q[0];
        a.rows_r[0] = (int)pl.rows_r[0];
        const cudaError_t e = mt == 2 ? launch_h_type<2, false>(type, a, pl, s) : launch_h_type<1, false>(type, a, pl, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

cudaError_t launch_hgemv_swiglu(int type, const uint8_t* Wg, const uint8_t* Wu, int64_t rows, int64_t cols,
                                const float* x, float* h, int sms, unsigned* status, cudaStream_t s) {
    const PlanH pl = planh(type, 1, &rows, cols, sms, 1, true);
    if (pl.stages == 0) return cudaErrorInvalidValue;
    if (pl.grid == 0) return cudaSuccess;
    hg::Args a = make_args(type, pl, cols, x, status);
    a.n = 1;
    a.W[0] = Wg;
    a.W[1] = Wu;
    a.y[0] = h;
    a.rows[0] = rows;
    a.rows_q[0] = pl.rows_q[0];
    a.rows_r[0] = (int)pl.rows_r[0];
    return launch_h_type<1, true>(type, a, pl, s);
}

}  // namespace qk
