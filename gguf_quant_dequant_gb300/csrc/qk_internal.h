// qk_internal.h -- launchers shared between the C-ABI layer (qk_api.cu) and
// the kernel translation units.  Host code only; no torch types anywhere.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/qk.h"

namespace qk {

// The driver's cuTensorMapEncodeTiled (looked up once; nullptr if missing).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

// Sets the calling thread's qk_last_error() text; returns st.
qk_status set_error(qk_status st, const char* msg);
// qk_gemv's argument checks (type, shape, NULL and alignment), in its order;
// sets the error text on failure.
qk_status gemv_check_args(int type, const void* W, int64_t rows, int64_t cols, const float* x, int64_t M,
                          const float* y);

cudaError_t launch_dequant(int type, const uint8_t* W, int64_t rows, int64_t cols, void* out,
                           int out_bf16, cudaStream_t s);

// Plain quantizer: a persistent grid of at most 4 CTAs per SM (sms SMs).
cudaError_t launch_quantize(int type, const float* w, int64_t rows, int64_t cols, uint8_t* out, int sms,
                            cudaStream_t s);
int64_t attn_decode_ws_bytes(int64_t T_len, int n_heads, int d);
bool attn_decode_shape_ok(int n_heads, int n_kv, int d);
cudaError_t launch_attn_decode(int type, const float* q, const uint8_t* K, const uint8_t* V, int64_t T_len, int n_heads,
                               int n_kv, int d, float scale, float* out, float* ws, unsigned* status, int sms,
                               cudaStream_t s);
cudaError_t launch_quantize_imatrix(int type, const float* w, const float* imp, int64_t rows, int64_t cols,
                                   uint8_t* out, cudaStream_t s);

cudaError_t launch_unpack(int type, const uint8_t* W, int64_t nblocks, int16_t* codes, int16_t* sc,
                          uint8_t* mins, float* d, float* dmin, cudaStream_t s);

// qk_gemv's plan: whether the tensor-core GEMV takes the shape (it needs
// no workspace for any shape).
struct GemvPlan {
    bool ok = false;
    int sms = 0;         // SM count the plan was made for
    int64_t ws_bytes = 0;
};
GemvPlan plan_gemv(int type, int64_t rows, int64_t cols, int64_t M, int sm_count);
// Tensor-core GEMV (qk_hgemv.cu): whether it takes this shape (type
// supported, two ring stages fit shared memory), the plain / batched launch
// (n <= QK_GEMV_BATCH_MAX matrices sharing x) and the SwiGLU launch.
bool hgemv_ok(int type, int n, const int64_t* rows, int64_t cols, int sms);
cudaError_t launch_hgemv(int type, int n, const uint8_t* const* W, const int64_t* rows, int64_t cols, const float* x,
                         float* const* y, int sms, unsigned* status, cudaStream_t s);
cudaError_t launch_hgemv_swiglu(int type, const uint8_t* Wg, const uint8_t* Wu, int64_t rows, int64_t cols,
                                const float* x, float* h, int sms, unsigned* status, cudaStream_t s);
// M activation rows through the same kernel (two per launch), y [M, rows].
cudaError_t launch_hgemv_tokens(int type, const uint8_t* W, int64_t rows, int64_t cols, const float* x, int64_t M,
                                float* y, int sms, unsigned* status, cudaStream_t s);
cudaError_t launch_gemv(int type, const GemvPlan& plan, const uint8_t* W, int64_t rows, int64_t cols,
                        const float* x, int64_t M, float* y, unsigned* status, cudaStream_t s);

// One thread waiting on an mbarrier nothing arrives on (bounded by limit_ns).
cudaError_t launch_stalled_wait(unsigned* status, uint64_t limit_ns, cudaStream_t s);

// Tensor-core dequant-GEMM (bf16 activations, fp32 output).  Small problems
// split K over CTAs; the partials [splits, M, rows] live in the workspace.
struct GemmPlan {
    int splits = 1;
    int kb_per_split = 0;   // 64-wide k-blocks per split
    int nmma = 256;         // MMA N
    bool skinny = false;    // M <= 64: deep pipeline, one small accumulator
    int64_t ws_bytes = 0;
};
GemmPlan plan_gemm(int type, int64_t rows, int64_t cols, int64_t M, int sm_count);
cudaError_t launch_gemm(int type, const GemmPlan& plan, const uint8_t* W, int64_t rows, int64_t cols, const void* X,
                        int64_t M, float* Y, float* ws, unsigned* status, cudaStream_t s);

}  // namespace qk
