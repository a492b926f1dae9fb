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
#include "qk_lanes.cuh"
#include "qk_ptx.cuh"

namespace qk {
namespace gv {

constexpr int kCW = 8;                 // consumer warps per CTA
constexpr int kRW = 2;                 // rows per consumer warp
constexpr int kRows = kCW * kRW;       // rows per CTA tile
constexpr int kThreads = (kCW + 1) * 32;

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

}  // namespace gv
}  // namespace qk

namespace qk {

namespace {
int mt_for(int64_t M) { return M >= 4 ? 4 : (M >= 2 ? 2 : 1); }

int64_t nst_for(int type, int64_t cols) {
    switch (type) {
    case T_Q4_K: case T_Q6_K: case T_Q5_K: case T_Q2_K: case T_Q3_K: return (cols / 256 + 7) / 8;
    case T_Q8_0: case T_Q5_0: case T_Q4_0: return (cols / 32 + 63) / 64;
    }
    return 0;
}

int64_t align16(int64_t v) { return (v + 15) & ~(int64_t)15; }
}  // namespace

// Activation rows up to which qk_gemv runs the tensor-core kernel (two rows
// per launch, weights streamed once per launch); beyond, the tiled kernel
// (weights decoded once per tile of up to four rows, prepped x in the
// workspace).
constexpr int64_t kTcMaxM = 64;

GemvPlan plan_gemv(int type, int64_t rows, int64_t cols, int64_t M, int sm_count) {
    GemvPlan pl;
    pl.sms = sm_count;
    if (M <= kTcMaxM && hgemv_ok(type, 1, &rows, cols, sm_count)) {   // tensor-core kernel, prep inside
        pl.decode = M == 1;
        pl.tc = true;
        return pl;
    }
    if (M == 1 && gemv5_ring_pairs(type, 1, &rows, cols, sm_count) > 0) {   // decode kernel, prep inside
        pl.decode = true;
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
static cudaError_t launch_mt(const GemvPlan& pl, const gv::Args& a, cudaStream_t s) {
    switch (pl.mt) {
    case 1: return launch_t<T, 1>(pl, a, s);
    case 2: return launch_t<T, 2>(pl, a, s);
    default: return launch_t<T, 4>(pl, a, s);
    }
}

cudaError_t launch_gemv(int type, const GemvPlan& pl, const uint8_t* W, int64_t rows, int64_t cols, const float* x,
                        int64_t M, float* y, float* ws, unsigned* status, cudaStream_t s) {
    if (pl.tc && M == 1) return launch_hgemv(type, 1, &W, &rows, cols, x, &y, pl.sms, status, s);
    if (pl.tc) return launch_hgemv_tokens(type, W, rows, cols, x, M, y, pl.sms, status, s);
    if (pl.decode) return launch_gemv5(type, 1, &W, &rows, cols, x, &y, pl.sms, s);
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
    case T_Q4_0: a.row_bytes = cols / 32 * 18; break;
    case T_Q5_K: a.row_bytes = cols / 256 * 176; break;
    case T_Q2_K: a.row_bytes = cols / 256 * 84; break;
    case T_Q3_K: a.row_bytes = cols / 256 * 110; break;
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
    switch (type) {
    case T_Q4_K: return launch_mt<T_Q4_K>(pl, a, s);
    case T_Q6_K: return launch_mt<T_Q6_K>(pl, a, s);
    case T_Q8_0: return launch_mt<T_Q8_0>(pl, a, s);
    case T_Q5_0: return launch_mt<T_Q5_0>(pl, a, s);
    case T_Q4_0: return launch_mt<T_Q4_0>(pl, a, s);
    case T_Q5_K: return launch_mt<T_Q5_K>(pl, a, s);
    case T_Q2_K: return launch_mt<T_Q2_K>(pl, a, s);
    case T_Q3_K: return launch_mt<T_Q3_K>(pl, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
