// qk_quant.cu -- the write side: fp32 weights -> packed GGUF blocks.
//
// The pages name the k-quant quantizer ("Quantization formats", the
// quantize_row_q4_K reference) without giving it; this is the plain min/max
// scheme (group parameters from plain_params, the block from assemble, both
// in qk_qlanes.cuh, where the formulas are listed).
//
// One warp quantizes a tile of 32 consecutive 32-weight groups (1024
// weights): four super-blocks for the K types, 32 blocks otherwise.  The
// grid is persistent: warp w takes tiles w, w + W, w + 2W, ... (W warps in
// all), streaming the next two tiles' 4 KB each into shared memory with
// coalesced 16-byte cp.async copies while it quantizes the current one (a
// ring of three buffers per warp), so that each SM keeps about 128 KB of
// loads in flight.
// 16-byte chunk c of a tile (group c / 8, columns 4(c % 8) ..) is stored at
// group * 128 + 16 * ((c % 8) ^ (group % 8)): lane l then reads its group's
// eight chunks without shared-memory bank conflicts.  Per-super-block maxima
// and the nibble / bit packing cross lanes with shuffles; the packed bytes
// are staged in shared memory and written out as 4-byte words.  The work is
// HBM-bound: 4 bytes read and BB/BE bytes written per weight; the codes take
// one reciprocal per group instead of a division per weight.
#include <algorithm>

#include "qk_internal.h"
#include "qk_ptx.cuh"
#include "qk_qlanes.cuh"

namespace qk {
namespace qz {

constexpr int kWarps = 4;                    // per CTA
constexpr int kCtasPerSm = 4;
constexpr int kStages = 3;                   // tiles in flight or in use per warp
constexpr int kBufWords = 32 * 34 / 4;      // largest warp output: 32 Q8_0 blocks = 1088 bytes
// Dynamic shared memory: [warp][stage] 4 KB input tiles, then [warp] staged
// output bytes.
constexpr int kSmemBytes = kWarps * kStages * 4096 + kWarps * kBufWords * 4;

// Request tile `tile` (valid groups ng) into the 4 KB buffer `xs`.
__device__ __forceinline__ void fetch_tile(const float* __restrict__ w, int64_t tile, int ng, float* xs, int lane) {
    const float* src = w + tile * 1024;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = lane + 32 * j, row = c >> 3, col = c & 7;
        if (row < ng) cp_async16(xs + row * 32 + 4 * (col ^ (row & 7)), src + 4 * c);
    }
}

template <int T>
__global__ void __launch_bounds__(kWarps * 32) quantize_kernel(const float* __restrict__ w, int64_t ngroups,
                                                                uint8_t* __restrict__ out) {
    constexpr bool kK = ql::LaneGeo<T>::K;
    constexpr int kBB = Fmt<T>::BB;
    extern __shared__ __align__(128) float qsm[];
    float* xw = qsm + (threadIdx.x >> 5) * (kStages * 1024);   // this warp's input tiles
    uint32_t* bw = reinterpret_cast<uint32_t*>(qsm + kWarps * kStages * 1024) + (threadIdx.x >> 5) * kBufWords;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (ngroups + 31) / 32;
    const int64_t stride = (int64_t)gridDim.x * kWarps;
    int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
    if (tile >= ntiles) return;   // whole warp
    auto groups_of = [&](int64_t t) { const int64_t left = ngroups - t * 32; return left < 32 ? (int)left : 32; };
#pragma unroll
    for (int j = 0; j < kStages - 1; ++j) {   // the first kStages - 1 tiles
        const int64_t t = tile + j * stride;
        if (t < ntiles) fetch_tile(w, t, groups_of(t), xw + j * 1024, lane);
        cp_async_commit();
    }
    uint8_t* sb = reinterpret_cast<uint8_t*>(bw);
    int st = 0;   // stage of the current tile
    for (; tile < ntiles; tile += stride) {
        const int64_t ahead = tile + (kStages - 1) * stride;
        const int sa = st == 0 ? kStages - 1 : st - 1;   // the stage freed by the previous tile
        if (ahead < ntiles) fetch_tile(w, ahead, groups_of(ahead), xw + sa * 1024, lane);
        cp_async_commit();
        cp_async_wait<kStages - 1>();   // this tile's copies (older than the kStages - 1 groups after them)
        __syncwarp();
        const int ng = groups_of(tile);
        const bool live = lane < ng;
        float v[32];
        const float* mine = xw + st * 1024 + lane * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = live ? *reinterpret_cast<const float4*>(mine + 4 * (i ^ (lane & 7)))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
        float sp[2], mp[2];
        ql::plain_params<T>(v, sp, mp);
        ql::assemble<T>(v, sp, mp, lane, live, sb + (kK ? (lane >> 3) : lane) * kBB);
        __syncwarp();
        // This tile's bytes: [first block * BB, + nb), 4-byte aligned (every
        // tile but the last covers a multiple of 4 bytes).
        const int64_t ob = (kK ? tile * 4 : tile * 32) * kBB;
        const int nb = (kK ? ng / 8 : ng) * kBB;
        uint8_t* dst = out + ob;
        for (int i = lane; i < nb / 4; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = bw[i];
        if (lane < (nb & 3)) dst[(nb & ~3) + lane] = sb[(nb & ~3) + lane];
        __syncwarp();   // the staged bytes and this tile's buffer are free again
        st = st == kStages - 1 ? 0 : st + 1;
    }
}

template <int T>
static cudaError_t launch_t(const float* w, int64_t ngroups, uint8_t* out, int sms, cudaStream_t s) {
    const int64_t tiles = (ngroups + 31) / 32;
    const int64_t need = (tiles + kWarps - 1) / kWarps;
    const int64_t blocks = std::min<int64_t>(need, (int64_t)std::max(sms, 1) * kCtasPerSm);
    const cudaError_t e = cudaFuncSetAttribute(quantize_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    quantize_kernel<T><<<(unsigned)blocks, kWarps * 32, kSmemBytes, s>>>(w, ngroups, out);
    return cudaGetLastError();
}

}  // namespace qz

cudaError_t launch_quantize(int type, const float* w, int64_t rows, int64_t cols, uint8_t* out, int sms,
                            cudaStream_t s) {
    const int64_t ngroups = rows * (cols / 32);
    switch (type) {
    case T_Q4_K: return qz::launch_t<T_Q4_K>(w, ngroups, out, sms, s);
    case T_Q6_K: return qz::launch_t<T_Q6_K>(w, ngroups, out, sms, s);
    case T_Q8_0: return qz::launch_t<T_Q8_0>(w, ngroups, out, sms, s);
    case T_Q5_0: return qz::launch_t<T_Q5_0>(w, ngroups, out, sms, s);
    case T_Q4_0: return qz::launch_t<T_Q4_0>(w, ngroups, out, sms, s);
    case T_Q5_K: return qz::launch_t<T_Q5_K>(w, ngroups, out, sms, s);
    case T_Q2_K: return qz::launch_t<T_Q2_K>(w, ngroups, out, sms, s);
    case T_Q3_K: return qz::launch_t<T_Q3_K>(w, ngroups, out, sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
