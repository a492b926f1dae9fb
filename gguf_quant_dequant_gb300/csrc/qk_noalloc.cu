// qk_noalloc.cu -- qk_gemv_noalloc: the fused dequant-GEMV for callers that
// cannot allocate device memory.  The GEMV kernel prepares its activations
// in shared memory and needs no workspace for any shape, so this entry point
// is qk_gemv with none, after the same argument checks.
#include "../../include/qk.h"
#include "qk_internal.h"

extern "C" qk_status qk_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols, const float* x,
                                     int64_t M, float* y, void* stream) {
    const qk_status st = qk::gemv_check_args(type, W, rows, cols, x, M, y);
    if (st != QK_OK) return st;
    return qk_gemv(type, W, rows, cols, x, M, y, nullptr, 0, stream);
}
