// qk_dequant.cu -- streaming dequantization (blocks -> fp32 / bf16 rows) and
// the integer unpack test hook.  One thread per 16-weight half; the output
// of a half is 16 consecutive values of a row, written with 16-byte stores.
#include <cuda_bf16.h>

#include "qk_formats.cuh"
#include "qk_internal.h"

namespace qk {

template <int T, bool BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int64_t nhalves,
                                                      int64_t nb_row, int64_t cols, void* __restrict__ out) {
    using F = Fmt<T>;
    constexpr int HPB = 2 * F::UPB;  // halves per block
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < nhalves;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = g / HPB;
        const int within = (int)(g % HPB), u = within >> 1, h = within & 1;
        const int64_t row = blk / nb_row, bi = blk % nb_row;
        float w[16];
        dequant_half<T>(W + blk * F::BB, u, h, w);
        const int64_t o = row * cols + bi * F::BE + F::koff(u, h);
        if (BF16) {
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(w[2 * i], w[2 * i + 1]);
                p[i] = *reinterpret_cast<const uint32_t*>(&v);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
        } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    }
}

template <int T>
__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ W, int64_t nblocks, int16_t* codes,
                                                     int16_t* sc, uint8_t* mins, float* d, float* dmin) {
    using F = Fmt<T>;
    const int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* blk = W + b * F::BB;
    if (codes) {
        for (int u = 0; u < F::UPB; ++u)
            for (int h = 0; h < 2; ++h) {
                int c[16];
                F::codes16(blk, u, h, c);
                for (int i = 0; i < 16; ++i) codes[b * F::BE + F::koff(u, h) + i] = (int16_t)c[i];
            }
    }
    if (sc)
        for (int j = 0; j < 16; ++j) {
            int v = 0;
            if constexpr (T == T_Q4_K || T == T_Q5_K) {
                uint32_t s, m;
                if (j < 8) { Fmt<T_Q4_K>::scale_min(blk, j, s, m); v = (int)s; }
            } else if constexpr (T == T_Q6_K) {
                v = (int)(int8_t)blk[192 + j];
            } else if constexpr (T == T_Q2_K) {
                v = (int)(blk[j] & 15u);
            } else if constexpr (T == T_Q3_K) {
                v = Fmt<T_Q3_K>::scale(blk, j);
            }
            sc[b * 16 + j] = (int16_t)v;
        }
    if (mins)
        for (int j = 0; j < 16; ++j) {
            uint32_t s = 0, m = 0;
            if constexpr (T == T_Q4_K || T == T_Q5_K) {
                if (j < 8) Fmt<T_Q4_K>::scale_min(blk, j, s, m);
            } else if constexpr (T == T_Q2_K) {
                m = blk[j] >> 4;
            }
            mins[b * 16 + j] = (uint8_t)m;
        }
    if (d) {
        if constexpr (T == T_Q6_K) d[b] = h2f(ld_u16(blk + 208));
        else if constexpr (T == T_Q2_K) d[b] = h2f(ld_u16(blk + 80));
        else if constexpr (T == T_Q3_K) d[b] = h2f(ld_u16(blk + 108));
        else d[b] = h2f(ld_u16(blk));
    }
    if (dmin) {
        if constexpr (T == T_Q4_K || T == T_Q5_K) dmin[b] = h2f(ld_u16(blk + 2));
        else if constexpr (T == T_Q2_K) dmin[b] = h2f(ld_u16(blk + 82));
        else dmin[b] = 0.0f;
    }
}

template <int T>
static cudaError_t dequant_t(const uint8_t* W, int64_t rows, int64_t cols, void* out, int bf16, cudaStream_t s) {
    using F = Fmt<T>;
    const int64_t nb_row = cols / F::BE;
    const int64_t nhalves = rows * nb_row * 2 * F::UPB;
    if (nhalves == 0) return cudaSuccess;
    const int64_t want = (nhalves + 255) / 256;
    const unsigned grid = (unsigned)(want < 65536 * 8 ? want : 65536 * 8);
    if (bf16) dequant_kernel<T, true><<<grid, 256, 0, s>>>(W, nhalves, nb_row, cols, out);
    else dequant_kernel<T, false><<<grid, 256, 0, s>>>(W, nhalves, nb_row, cols, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int type, const uint8_t* W, int64_t rows, int64_t cols, void* out, int out_bf16,
                           cudaStream_t s) {
    switch (type) {
    case T_Q4_K: return dequant_t<T_Q4_K>(W, rows, cols, out, out_bf16, s);
    case T_Q6_K: return dequant_t<T_Q6_K>(W, rows, cols, out, out_bf16, s);
    case T_Q8_0: return dequant_t<T_Q8_0>(W, rows, cols, out, out_bf16, s);
    case T_Q5_0: return dequant_t<T_Q5_0>(W, rows, cols, out, out_bf16, s);
    case T_Q4_0: return dequant_t<T_Q4_0>(W, rows, cols, out, out_bf16, s);
    case T_Q5_K: return dequant_t<T_Q5_K>(W, rows, cols, out, out_bf16, s);
    case T_Q2_K: return dequant_t<T_Q2_K>(W, rows, cols, out, out_bf16, s);
    case T_Q3_K: return dequant_t<T_Q3_K>(W, rows, cols, out, out_bf16, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_unpack(int type, const uint8_t* W, int64_t nblocks, int16_t* codes, int16_t* sc, uint8_t* mins,
                          float* d, float* dmin, cudaStream_t s) {
    if (nblocks == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((nblocks + 255) / 256);
    switch (type) {
    case T_Q4_K: unpack_kernel<T_Q4_K><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q6_K: unpack_kernel<T_Q6_K><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q8_0: unpack_kernel<T_Q8_0><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q5_0: unpack_kernel<T_Q5_0><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q4_0: unpack_kernel<T_Q4_0><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q5_K: unpack_kernel<T_Q5_K><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q2_K: unpack_kernel<T_Q2_K><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    case T_Q3_K: unpack_kernel<T_Q3_K><<<grid, 256, 0, s>>>(W, nblocks, codes, sc, mins, d, dmin); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qk
