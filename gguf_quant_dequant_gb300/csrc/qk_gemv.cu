// qk_gemv.cu -- fused dequant-GEMV: y[m, n] = sum_k w[n, k] x[m, k].
//
// The packed weights are dequantized inside the dot product ("Local LLM
// inference", "The mmap backend"); each decoded weight is reused across the
// MT activation rows a CTA holds (the same page: decode each projection
// weight once per input batch, reuse it across the batch rows).
//
// Work split.  A warp owns RW = 4 consecutive output rows and walks their K
// range in stages of 1024 weights (4 super-blocks or 32 small blocks per
// row).  Lane 0 of the warp streams each stage's four row segments from HBM
// into a private 4-deep shared-memory ring with bulk async copies
// (cp.async.bulk, completion counted on an mbarrier); the segments need not
// start on 16-byte boundaries (Q6_K rows of 11008 weights are 9030 bytes
// apart), so each copy starts at the aligned-down address and the consumer
// parses from the remainder.  Each lane decodes one 32-weight unit of each
// row per stage, as two 16-weight halves, and accumulates in fp32.  A warp
// shuffle tree sums the lanes.  For skinny problems the K range is split
// over gridDim.z and a second kernel adds the partials in a fixed order.
#include <algorithm>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_ptx.cuh"

namespace qk {

namespace gemv {

constexpr int kWarps = 4;     // warps per CTA
constexpr int kRW = 4;        // rows per warp
constexpr int kStages = 4;    // ring depth per warp
constexpr int kStageW = 1024; // weights per row per stage

template <int T>
struct Geo {
    static constexpr int KB = kStageW / Fmt<T>::BE;               // blocks per row per stage
    static constexpr int SEG = KB * Fmt<T>::BB;                   // bytes per row segment
    static constexpr int SLOT = ((SEG + 32) + 15) / 16 * 16;      // with alignment slack
    static constexpr int WARP_BYTES = kStages * kRW * SLOT;
    static constexpr int SMEM = kWarps * WARP_BYTES + kWarps * kStages * 8;
};

struct Args {
    const uint8_t* W;
    int64_t rows, cols, M;
    int64_t row_bytes;
    int64_t total16;   // total bytes of W rounded down to 16
    int64_t total;     // total bytes of W
    const float* x;
    float* out;        // y (splits == 1) or the partial buffer
    int splits;
    int stages_per_split;
    unsigned* status;
};

// Byte range of row `row`'s segment for global stage `gs`, and the aligned
// window a bulk copy may read: [a, e) with a = start rounded down to 16 and
// e = end rounded up to 16 but never past the last full 16 bytes of W.
template <int T>
struct Seg {
    int64_t start, end, a, e;
    __device__ __forceinline__ Seg(const Args& p, int64_t row, int64_t gs) {
        using G = Geo<T>;
        const int64_t nb = p.cols / Fmt<T>::BE;
        const int64_t b0 = gs * G::KB;
        const int64_t nblk = min((int64_t)G::KB, nb - b0);
        start = row * p.row_bytes + b0 * Fmt<T>::BB;
        end = start + nblk * Fmt<T>::BB;
        a = start & ~(int64_t)15;
        e = min((end + 15) & ~(int64_t)15, p.total16);
    }
};

template <int T>
__device__ __forceinline__ void issue_stage(const Args& p, uint8_t* wbuf, uint64_t* bars, int64_t row0,
                                            int64_t gs, int slot, uint64_t pol) {
    using G = Geo<T>;
    uint32_t bytes = 0;
#pragma unroll
    for (int rr = 0; rr < kRW; ++rr) {
        if (row0 + rr >= p.rows) continue;
        Seg<T> s(p, row0 + rr, gs);
        if (s.e > s.a) bytes += (uint32_t)(s.e - s.a);
    }
    mbar_arrive_expect_tx(&bars[slot], bytes);
#pragma unroll
    for (int rr = 0; rr < kRW; ++rr) {
        if (row0 + rr >= p.rows) continue;
        Seg<T> s(p, row0 + rr, gs);
        if (s.e > s.a)
            bulk_g2s(wbuf + (slot * kRW + rr) * G::SLOT, p.W + s.a, (uint32_t)(s.e - s.a), &bars[slot], pol);
    }
}

template <int T, int MT>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const Args p) {
    using F = Fmt<T>;
    using G = Geo<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wbuf = smem + warp * G::WARP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * G::WARP_BYTES) + warp * kStages;

    const int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * kRW;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    const int64_t nb = p.cols / F::BE;
    const int64_t nstage_all = (nb + G::KB - 1) / G::KB;
    const int64_t gs0 = (int64_t)blockIdx.z * p.stages_per_split;
    const int64_t nloc = max((int64_t)0, min((int64_t)p.stages_per_split, nstage_all - gs0));

    pdl_launch_dependents();
    if (row0 >= p.rows) return;  // whole warp idle (ragged last CTA)

    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        for (int s = 0; s < kStages && s < nloc; ++s) issue_stage<T>(p, wbuf, bars, row0, gs0 + s, s, pol);
    }
    __syncwarp();
    // The activations may come from the previous kernel in the stream.
    pdl_wait_prior();

    float acc[kRW][MT];
#pragma unroll
    for (int rr = 0; rr < kRW; ++rr)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[rr][m] = 0.0f;

    const int bi = lane / F::UPB;  // block of this lane within the stage
    const int u = lane % F::UPB;   // unit of this lane within its block

    for (int64_t i = 0; i < nloc; ++i) {
        const int slot = (int)(i % kStages);
        const int64_t gs = gs0 + i;
        if (!mbar_wait_bounded(&bars[slot], (uint32_t)((i / kStages) & 1), p.status)) {
            // Give up; first let every copy already issued land (bounded).
            for (int64_t j = i + 1; j < min(nloc, i + kStages); ++j)
                mbar_wait_bounded(&bars[j % kStages], (uint32_t)((j / kStages) & 1), p.status);
            return;
        }
        // Bytes past the last full 16 bytes of W cannot be bulk-copied; the
        // lanes fetch them (only ever the final segment of the matrix).
#pragma unroll
        for (int rr = 0; rr < kRW; ++rr) {
            if (row0 + rr >= p.rows) continue;
            Seg<T> s(p, row0 + rr, gs);
            if (s.end > p.total16) {
                uint8_t* dst = wbuf + (slot * kRW + rr) * G::SLOT;
                for (int64_t b = max(s.start, p.total16) + lane; b < s.end; b += 32) dst[b - s.a] = p.W[b];
            }
        }
        __syncwarp();

        const int64_t blk = gs * G::KB + bi;
        if (blk < nb) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t k = blk * F::BE + F::koff(u, h);
                float xv[MT][16];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m0 + m < p.M) {
                        const float4* xp = reinterpret_cast<const float4*>(p.x + (m0 + m) * p.cols + k);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 v = __ldg(xp + q);
                            xv[m][4 * q] = v.x; xv[m][4 * q + 1] = v.y; xv[m][4 * q + 2] = v.z; xv[m][4 * q + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) xv[m][q] = 0.0f;
                    }
                }
#pragma unroll
                for (int rr = 0; rr < kRW; ++rr) {
                    if (row0 + rr >= p.rows) continue;
                    const int64_t start = (row0 + rr) * p.row_bytes + gs * G::KB * (int64_t)F::BB;
                    const uint8_t* b = wbuf + (slot * kRW + rr) * G::SLOT + (int)(start & 15) + bi * F::BB;
                    float w[16];
                    dequant_half<T>(b, u, h, w);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float s = 0.0f;
#pragma unroll
                        for (int q = 0; q < 16; ++q) s = fmaf(w[q], xv[m][q], s);
                        acc[rr][m] += s;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + kStages < nloc) issue_stage<T>(p, wbuf, bars, row0, gs + kStages, slot, pol);
    }

#pragma unroll
    for (int rr = 0; rr < kRW; ++rr)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[rr][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[rr][m] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int rr = 0; rr < kRW; ++rr) {
            if (row0 + rr >= p.rows) continue;
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m0 + m < p.M) p.out[((int64_t)blockIdx.z * p.M + m0 + m) * p.rows + row0 + rr] = acc[rr][m];
        }
    }
}

// y[m, n] = sum over splits z (in order) of part[z, m, n].
__global__ void __launch_bounds__(256) splitk_reduce(const float* __restrict__ part, int splits, int64_t n,
                                                     float* __restrict__ y) {
    pdl_launch_dependents();
    pdl_wait_prior();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float s = part[i];
        for (int z = 1; z < splits; ++z) s += part[(int64_t)z * n + i];
        y[i] = s;
    }
}

}  // namespace gemv
}  // namespace qk

namespace qk {

static int mt_for(int64_t M) { return M >= 4 ? 4 : (M >= 2 ? 2 : 1); }

template <int T>
static int64_t stage_count(int64_t cols) {
    const int64_t nb = cols / Fmt<T>::BE;
    return (nb + gemv::Geo<T>::KB - 1) / gemv::Geo<T>::KB;
}

static int64_t stages_for(int type, int64_t cols) {
    switch (type) {
    case T_Q4_K: return stage_count<T_Q4_K>(cols);
    case T_Q6_K: return stage_count<T_Q6_K>(cols);
    case T_Q8_0: return stage_count<T_Q8_0>(cols);
    case T_Q5_0: return stage_count<T_Q5_0>(cols);
    }
    return 0;
}

GemvPlan plan_gemv(int type, int64_t rows, int64_t cols, int64_t M, int sm_count) {
    GemvPlan pl;
    pl.mt = mt_for(M);
    const int64_t rows_per_cta = gemv::kWarps * gemv::kRW;
    const int64_t ctas = ((rows + rows_per_cta - 1) / rows_per_cta) * ((M + pl.mt - 1) / pl.mt);
    const int64_t nst = stages_for(type, cols);
    const int64_t target = 2 * (int64_t)std::max(sm_count, 1);
    int64_t splits = 1;
    if (ctas > 0 && ctas < target && nst > 1) splits = std::min<int64_t>({(target + ctas - 1) / ctas, nst, 16});
    // Every split must own at least one stage.
    if (splits > 1) {
        const int64_t per = (nst + splits - 1) / splits;
        splits = (nst + per - 1) / per;
    }
    pl.splits = (int)splits;
    pl.ws_bytes = splits > 1 ? splits * M * rows * (int64_t)sizeof(float) : 0;
    return pl;
}

template <int T, int MT>
static cudaError_t launch_t(const GemvPlan& pl, const gemv::Args& a, cudaStream_t s) {
    using G = gemv::Geo<T>;
    auto kern = gemv::gemv_kernel<T, MT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t rows_per_cta = gemv::kWarps * gemv::kRW;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.rows + rows_per_cta - 1) / rows_per_cta), (unsigned)((a.M + MT - 1) / MT),
                       (unsigned)pl.splits);
    cfg.blockDim = dim3(gemv::kWarps * 32);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int T>
static cudaError_t launch_mt(const GemvPlan& pl, const gemv::Args& a, cudaStream_t s) {
    switch (pl.mt) {
    case 1: return launch_t<T, 1>(pl, a, s);
    case 2: return launch_t<T, 2>(pl, a, s);
    default: return launch_t<T, 4>(pl, a, s);
    }
}

cudaError_t launch_gemv(int type, const GemvPlan& pl, const uint8_t* W, int64_t rows, int64_t cols, const float* x,
                        int64_t M, float* y, float* ws, unsigned* status, cudaStream_t s) {
    gemv::Args a;
    a.W = W;
    a.rows = rows;
    a.cols = cols;
    a.M = M;
    const int64_t nst = stages_for(type, cols);
    a.stages_per_split = (int)((nst + pl.splits - 1) / pl.splits);
    a.splits = pl.splits;
    a.x = x;
    a.out = pl.splits > 1 ? ws : y;
    a.status = status;
    switch (type) {
    case T_Q4_K: a.row_bytes = cols / 256 * 144; break;
    case T_Q6_K: a.row_bytes = cols / 256 * 210; break;
    case T_Q8_0: a.row_bytes = cols / 32 * 34; break;
    case T_Q5_0: a.row_bytes = cols / 32 * 22; break;
    default: return cudaErrorInvalidValue;
    }
    a.total = rows * a.row_bytes;
    a.total16 = a.total & ~(int64_t)15;
    cudaError_t e = cudaErrorInvalidValue;
    switch (type) {
    case T_Q4_K: e = launch_mt<T_Q4_K>(pl, a, s); break;
    case T_Q6_K: e = launch_mt<T_Q6_K>(pl, a, s); break;
    case T_Q8_0: e = launch_mt<T_Q8_0>(pl, a, s); break;
    case T_Q5_0: e = launch_mt<T_Q5_0>(pl, a, s); break;
    }
    if (e != cudaSuccess || pl.splits == 1) return e;
    const int64_t n = M * rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((n + 255) / 256, 65535));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv::splitk_reduce, (const float*)ws, pl.splits, n, y);
}

}  // namespace qk
