// qk_gemm.cu -- tensor-core dequant-GEMM for prefill: Y[m, n] = sum_k w[n, k] X[m, k].
//
// Prefill turns the per-token GEMV into a real dense contraction ("12 --
// llama.cpp / GGUF": prompt processing is big GEMMs of high arithmetic
// intensity; decode is bandwidth-bound).  A CTA owns 128 weight rows x 256
// tokens and walks K in blocks of 64:
//   * 8 dequant warps unpack the packed blocks of the 128 weight rows, round
//     the fp32 weights to bf16 and store them straight into shared memory in
//     the tensor core's K-major 128-byte-swizzled layout (operand A);
//   * one thread loads the 256 x 64 bf16 activation tile with TMA (operand B);
//   * one thread issues tcgen05.mma (M = 128, N = 256, K = 16 per instruction)
//     into an fp32 accumulator in tensor memory and releases each stage with
//     tcgen05.commit;
//   * four warps read the accumulator back (tcgen05.ld) and write Y.
// Every mbarrier wait is bounded; tensor memory is always released.
#include <algorithm>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "qk_formats.cuh"
#include "qk_internal.h"
#include "qk_ptx.cuh"
#include "qk_tc.cuh"

namespace qk {
namespace gm {

constexpr int kBM = 128;          // weight rows per CTA (MMA M)
constexpr int kBN = 256;          // tokens per CTA (MMA N)
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int kNS = 4;            // pipeline stages
constexpr int kA = kBM * kBK * 2; // 16 KB
constexpr int kB = kBN * kBK * 2; // 32 KB
constexpr int kStage = kA + kB;
constexpr int kDeqWarps = 8;
constexpr int kThreads = (2 + kDeqWarps) * 32;
constexpr int kTmemCols = 256;
constexpr int kSmem = 1024 + kNS * kStage + (3 * kNS + 1) * 8 + 16;

struct Args {
    const uint8_t* W;
    int64_t rows, cols, row_bytes, M;
    float* Y;
    unsigned* status;
    int nkb;
};

// (unit, half) of the 16 weights that start `o` weights into a block.
template <int T>
__device__ __forceinline__ void locate(int o, int& u, int& h) {
    if constexpr (T == T_Q4_K) {          // koff = 64(u>>1) + 32h + 16(u&1)
        u = 2 * (o >> 6) + ((o >> 4) & 1);
        h = (o >> 5) & 1;
    } else if constexpr (T == T_Q6_K) {   // koff = 128(u>>2) + 32((u>>1&1) + 2h) + 16(u&1)
        const int t = o >> 7, g = (o >> 5) & 3;
        u = 4 * t + 2 * (g & 1) + ((o >> 4) & 1);
        h = g >> 1;
    } else {                              // 32-weight blocks: koff = 16h
        u = 0;
        h = (o >> 4) & 1;
    }
}

// 32 bf16 weights of row `row`, k in [k0, k0 + 32), into 4 swizzled 16-byte
// chunks of the A stage (chunks cbase..cbase+3 of the row).  Rows past the
// matrix and k past cols are zero.
template <int T>
__device__ __forceinline__ void dequant32(const Args& p, uint8_t* A, int r, int64_t row, int64_t k0, int cbase) {
    using F = Fmt<T>;
    uint32_t packed[16];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int64_t k = k0 + 16 * hf;
        float w[16];
        if (row < p.rows && k < p.cols) {
            const int64_t b = k / F::BE;
            int u, h;
            locate<T>((int)(k % F::BE), u, h);
            dequant_half<T>(p.W + row * p.row_bytes + b * F::BB, u, h, w);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(w[2 * i], w[2 * i + 1]);
            packed[8 * hf + i] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
    uint8_t* rowp = A + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int chunk = (cbase + c) ^ (r & 7);
        *reinterpret_cast<uint4*>(rowp + chunk * 16) =
            make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
    }
}

template <int T>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Args p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (the 128-byte swizzle atoms must be aligned).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* full_x = reinterpret_cast<uint64_t*>(smem + kNS * kStage);
    uint64_t* full_w = full_x + kNS;
    uint64_t* empty = full_w + kNS;
    uint64_t* accum = empty + kNS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kBM;
    const int64_t tok0 = (int64_t)blockIdx.y * kBN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&full_w[s], kDeqWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
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
            int issued = 0;
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int s = kb % kNS;
                if (kb >= kNS && !mbar_wait_bounded(&empty[s], (uint32_t)((kb / kNS - 1) & 1), p.status)) break;
                mbar_arrive_expect_tx(&full_x[s], (uint32_t)kB);
                tc::tma_load_2d(smem + s * kStage + kA, &xmap, kb * kBK, (int)tok0, &full_x[s]);
                issued = kb + 1;
            }
            // Every load issued must land before the CTA may exit.
            for (int kb = issued > kNS ? issued - kNS : 0; kb < issued; ++kb)
                mbar_wait_bounded(&full_x[kb % kNS], (uint32_t)((kb / kNS) & 1), p.status);
        }
    } else if (warp == 1) {
        // MMA issuer.
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int s = kb % kNS;
                const uint32_t par = (uint32_t)((kb / kNS) & 1);
                if (!mbar_wait_bounded(&full_x[s], par, p.status) || !mbar_wait_bounded(&full_w[s], par, p.status))
                    break;
                tc::fence_after_sync();
                const uint32_t a = smem_u32(smem + s * kStage), b = a + kA;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc::mma_bf16(tmem, tc::sdesc_k128(a + 32 * kk), tc::sdesc_k128(b + 32 * kk), idesc,
                                 (kb | kk) != 0 ? 1u : 0u);
                tc::commit(&empty[s]);
            }
            tc::commit(accum);   // fires once every MMA issued above has completed
            // Tensor memory may only be released after the MMAs are done.
            mbar_wait_bounded(accum, 0, p.status);
        }
    } else {
        // Dequant warps: thread -> (tile row r, half hh of the 64-wide k-block).
        const int t = threadIdx.x - 64;
        const int r = t & (kBM - 1), hh = t >> 7;
        const int64_t row = row0 + r;
        for (int kb = 0; kb < p.nkb; ++kb) {
            const int s = kb % kNS;
            if (kb >= kNS && !mbar_wait_bounded(&empty[s], (uint32_t)((kb / kNS - 1) & 1), p.status)) break;
            dequant32<T>(p, smem + s * kStage, r, row, (int64_t)kb * kBK + 32 * hh, 4 * hh);
            fence_proxy_async_smem();   // generic stores -> visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_w[s]);
        }
        // Epilogue: warps 2..5 cover the four 32-lane quarters of the accumulator.
        if (warp < 6) {
            const int q = warp & 3;
            mbar_wait_bounded(accum, 0, p.status);
            tc::fence_after_sync();
            const int64_t orow = row0 + 32 * q + lane;
#pragma unroll 1
            for (int j = 0; j < kBN / 16; ++j) {
                uint32_t v[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * j, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int64_t tok = tok0 + 16 * j + i;
                    if (tok < p.M && orow < p.rows) p.Y[tok * p.rows + orow] = __uint_as_float(v[i]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace gm
}  // namespace qk

namespace qk {

namespace {
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
}  // namespace

template <int T>
static cudaError_t gemm_t(const gm::Args& a, const CUtensorMap& map, cudaStream_t s) {
    auto kern = gm::gemm_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gm::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.rows + gm::kBM - 1) / gm::kBM), (unsigned)((a.M + gm::kBN - 1) / gm::kBN));
    cfg.blockDim = dim3(gm::kThreads);
    cfg.dynamicSmemBytes = gm::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

cudaError_t launch_gemm(int type, const uint8_t* W, int64_t rows, int64_t cols, const void* X, int64_t M, float* Y,
                        unsigned* status, cudaStream_t s) {
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    // X: bf16 [M, cols] row-major; tiles of 64 (k) x 256 (tokens), 128-byte swizzle.
    CUtensorMap map;
    cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)M};
    cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)gm::kBK, (cuuint32_t)gm::kBN};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    gm::Args a;
    a.W = W;
    a.rows = rows;
    a.cols = cols;
    a.M = M;
    a.Y = Y;
    a.status = status;
    a.nkb = (int)((cols + gm::kBK - 1) / gm::kBK);
    switch (type) {
    case T_Q4_K: a.row_bytes = cols / 256 * 144; return gemm_t<T_Q4_K>(a, map, s);
    case T_Q6_K: a.row_bytes = cols / 256 * 210; return gemm_t<T_Q6_K>(a, map, s);
    case T_Q8_0: a.row_bytes = cols / 32 * 34; return gemm_t<T_Q8_0>(a, map, s);
    case T_Q5_0: a.row_bytes = cols / 32 * 22; return gemm_t<T_Q5_0>(a, map, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
