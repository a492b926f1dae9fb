// qk_noalloc.cu -- qk_gemv_noalloc: the fused dequant-GEMV for callers that
// cannot allocate device memory.  Its scratch (prepped activations, split-K
// partials and tile counters) lives in one fixed array in this library's
// device image instead of a caller-provided workspace.
#include <cstdio>
#include <mutex>

#include "../../include/qk.h"
#include "qk_internal.h"

namespace {

// The shared scratch of every qk_gemv_noalloc call on a device.  It belongs
// to the loaded module, so each GPU that loads libqk holds it until exit.
static __device__ __align__(256) unsigned char g_gemv_scratch[QK_GEMV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" qk_status qk_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols, const float* x,
                                     int64_t M, float* y, void* stream) {
    // Argument errors first, in qk_gemv's order, so that a bad pointer is
    // reported as such whatever the problem's size.
    const qk_status st = qk::gemv_check_args(type, W, rows, cols, x, M, y);
    if (st != QK_OK) return st;
    const size_t need = qk_gemv_workspace(type, rows, cols, M);
    if (need > QK_GEMV_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "qk_gemv_noalloc: this problem needs %zu bytes of scratch; the static scratch holds %zu "
                 "(use qk_gemv with a workspace)",
                 need, (size_t)QK_GEMV_NOALLOC_SCRATCH_BYTES);
        return qk::set_error(QK_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qk::set_error(QK_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return qk::set_error(QK_ERR_ARG, "qk_gemv_noalloc: device id out of range");
    void* scratch = nullptr;
    {
        // First call on this device (which must be current): look up the
        // device address of the array.  Host code cannot use the symbol itself.
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_gemv_scratch);
            if (e != cudaSuccess) return qk::set_error(QK_ERR_CUDA, cudaGetErrorString(e));
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    return qk_gemv(type, W, rows, cols, x, M, y, scratch, QK_GEMV_NOALLOC_SCRATCH_BYTES, stream);
}
