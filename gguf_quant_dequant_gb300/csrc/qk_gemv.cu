// qk_gemv.cu -- qk_gemv's plan and launch: y[m, n] = sum_k w[n, k] x[m, k].
//
// The packed weights are dequantized inside the dot product ("Local LLM
// inference", "The mmap backend").  Every activation batch runs the
// tensor-core GEMV of qk_hgemv.cu: one launch for a single token, else one
// launch per pair of tokens (each weight decoded once per launch and used
// for both).  The kernel prepares x itself, one 256-element unit per warp,
// so no shape needs a workspace and no row length is too long.
#include "qk_internal.h"

namespace qk {

GemvPlan plan_gemv(int type, int64_t rows, int64_t cols, int64_t M, int sm_count) {
    GemvPlan pl;
    pl.sms = sm_count;
    pl.ok = M > 0 && hgemv_ok(type, 1, &rows, cols, sm_count);
    return pl;
}

cudaError_t launch_gemv(int type, const GemvPlan& pl, const uint8_t* W, int64_t rows, int64_t cols, const float* x,
                        int64_t M, float* y, unsigned* status, cudaStream_t s) {
    if (!pl.ok) return cudaErrorInvalidValue;
    if (M == 1) return launch_hgemv(type, 1, &W, &rows, cols, x, &y, pl.sms, status, s);
    return launch_hgemv_tokens(type, W, rows, cols, x, M, y, pl.sms, status, s);
}

}  // namespace qk
