// qk_api.cu -- the extern "C" entry points of libqk (include/qk.h): argument
// validation on the host, then a launch on the caller's stream.  Nothing here
// allocates device memory; scratch comes from the caller's workspace.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/qk.h"
#include "qk_internal.h"

namespace {

thread_local std::string g_last_error;

// Kernel status word (bit 0: a bounded wait ran out).  One per device; its
// address is looked up once per device and passed to the kernels.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

qk_status fail(qk_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
qk_status fail(qk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

qk_status cuda_fail(cudaError_t e, const char* where) {
    return fail(QK_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool known_type(int t) { return t >= QK_Q4_K && t <= QK_Q3_K; }

size_t block_bytes(int t) {
    switch (t) {
    case QK_Q4_K: return 144;
    case QK_Q6_K: return 210;
    case QK_Q8_0: return 34;
    case QK_Q5_0: return 22;
    case QK_Q4_0: return 18;
    case QK_Q5_K: return 176;
    case QK_Q2_K: return 84;
    case QK_Q3_K: return 110;
    }
    return 0;
}

int block_elems(int t) {
    switch (t) {
    case QK_Q4_K: case QK_Q6_K: case QK_Q5_K: case QK_Q2_K: case QK_Q3_K: return 256;
    case QK_Q8_0: case QK_Q5_0: case QK_Q4_0: return 32;
    }
    return 0;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-device state: status-word address and SM count, set up on first use.
qk_status device_state(unsigned** status, int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QK_ERR_ARG, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_sm_count[dev] = n;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    if (status) *status = g_status_ptr[dev];
    if (sms) *sms = g_sm_count[dev];
    return QK_OK;
}

int sm_count_or_default() {
    int sms = 0;
    if (device_state(nullptr, &sms) != QK_OK || sms <= 0) return 148;
    return sms;
}

// Shared validation of (type, rows, cols, W).
qk_status check_matrix(int type, const void* W, int64_t rows, int64_t cols) {
    if (!known_type(type)) return fail(QK_ERR_TYPE, "unknown quant type %d", type);
    if (rows < 0 || cols < 0) return fail(QK_ERR_SHAPE, "negative shape rows=%lld cols=%lld", (long long)rows,
                                          (long long)cols);
    if (cols % block_elems(type) != 0)
        return fail(QK_ERR_SHAPE, "cols=%lld is not a multiple of %d", (long long)cols, block_elems(type));
    if (rows > 0 && cols > 0) {
        if (!W) return fail(QK_ERR_NULL, "W is NULL");
        if (!aligned(W, 16)) return fail(QK_ERR_ALIGN, "W is not 16-byte aligned");
    }
    return QK_OK;
}

}  // namespace

namespace qk {
// Record `msg` as the calling thread's last error and return `st` (for entry
// points defined in other translation units).
qk_status set_error(qk_status st, const char* msg) { return fail(st, "%s", msg); }

// The argument checks of qk_gemv, in its order (no launch, no device call).
qk_status gemv_check_args(int type, const void* W, int64_t rows, int64_t cols, const float* x, int64_t M,
                          const float* y) {
    qk_status st = check_matrix(type, W, rows, cols);
    if (st != QK_OK) return st;
    if (M < 0) return fail(QK_ERR_SHAPE, "negative M=%lld", (long long)M);
    if (rows == 0 || M == 0) return QK_OK;
    if (!y) return fail(QK_ERR_NULL, "y is NULL");
    if (!aligned(y, 4)) return fail(QK_ERR_ALIGN, "y is not 4-byte aligned");
    if (cols == 0) return QK_OK;
    if (!x) return fail(QK_ERR_NULL, "x is NULL");
    if (!aligned(x, 16)) return fail(QK_ERR_ALIGN, "x is not 16-byte aligned");
    return QK_OK;
}
}  // namespace qk

extern "C" {

int qk_version(void) { return 1; }

size_t qk_block_bytes(int type) { return block_bytes(type); }

int qk_block_elems(int type) { return block_elems(type); }

size_t qk_row_bytes(int type, int64_t cols) {
    if (!known_type(type) || cols < 0 || cols % block_elems(type) != 0) return 0;
    return (size_t)(cols / block_elems(type)) * block_bytes(type);
}

const char* qk_last_error(void) { return g_last_error.c_str(); }

qk_status qk_dequant(int type, const void* W, int64_t rows, int64_t cols, void* out, int out_dtype, void* stream) {
    qk_status st = check_matrix(type, W, rows, cols);
    if (st != QK_OK) return st;
    if (out_dtype != QK_OUT_F32 && out_dtype != QK_OUT_BF16) return fail(QK_ERR_ARG, "bad out_dtype %d", out_dtype);
    if (rows == 0 || cols == 0) return QK_OK;
    if (!out) return fail(QK_ERR_NULL, "out is NULL");
    if (!aligned(out, 16)) return fail(QK_ERR_ALIGN, "out is not 16-byte aligned");
    cudaError_t e = qk::launch_dequant(type, static_cast<const uint8_t*>(W), rows, cols, out,
                                       out_dtype == QK_OUT_BF16, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_dequant launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_quantize(int type, const float* w, int64_t rows, int64_t cols, void* out, void* stream) {
    if (!known_type(type)) return fail(QK_ERR_TYPE, "unknown type %d", type);
    if (rows < 0 || cols < 0 || cols % block_elems(type) != 0)
        return fail(QK_ERR_SHAPE, "bad shape rows=%lld cols=%lld", (long long)rows, (long long)cols);
    if (rows == 0 || cols == 0) return QK_OK;
    if (rows > (int64_t(1) << 46) / cols)   // 2^46 weights: far beyond any device memory
        return fail(QK_ERR_SHAPE, "rows * cols too large (rows=%lld cols=%lld)", (long long)rows, (long long)cols);
    if (!w) return fail(QK_ERR_NULL, "w is NULL");
    if (!out) return fail(QK_ERR_NULL, "out is NULL");
    if (!aligned(w, 16)) return fail(QK_ERR_ALIGN, "w is not 16-byte aligned");
    if (!aligned(out, 4)) return fail(QK_ERR_ALIGN, "out is not 4-byte aligned");
    int sms = 0;
    const qk_status st = device_state(nullptr, &sms);
    if (st != QK_OK) return st;
    cudaError_t e = qk::launch_quantize(type, w, rows, cols, static_cast<uint8_t*>(out), sms,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_quantize launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_quantize_imatrix(int type, const float* w, int64_t rows, int64_t cols, const float* imp, void* out,
                              void* stream) {
    if (!known_type(type)) return fail(QK_ERR_TYPE, "unknown type %d", type);
    if (rows < 0 || cols < 0 || cols % block_elems(type) != 0)
        return fail(QK_ERR_SHAPE, "bad shape rows=%lld cols=%lld", (long long)rows, (long long)cols);
    if (rows == 0 || cols == 0) return QK_OK;
    if (rows > (int64_t(1) << 46) / cols)
        return fail(QK_ERR_SHAPE, "rows * cols too large (rows=%lld cols=%lld)", (long long)rows, (long long)cols);
    if (!w) return fail(QK_ERR_NULL, "w is NULL");
    if (!imp) return fail(QK_ERR_NULL, "imp is NULL");
    if (!out) return fail(QK_ERR_NULL, "out is NULL");
    if (!aligned(w, 16)) return fail(QK_ERR_ALIGN, "w is not 16-byte aligned");
    if (!aligned(imp, 4) || !aligned(out, 4)) return fail(QK_ERR_ALIGN, "imp or out is not 4-byte aligned");
    cudaError_t e = qk::launch_quantize_imatrix(type, w, imp, rows, cols, static_cast<uint8_t*>(out),
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_quantize_imatrix launch");
    g_last_error.clear();
    return QK_OK;
}

size_t qk_attn_decode_workspace(int type, int64_t T, int n_heads, int n_kv, int d) {
    if ((type != QK_Q8_0 && type != QK_Q5_0 && type != QK_Q4_0) || T < 1 || !qk::attn_decode_shape_ok(n_heads, n_kv, d))
        return 0;
    return (size_t)qk::attn_decode_ws_bytes(T, n_heads, d);
}

qk_status qk_attn_decode(int type, const float* q, const void* K, const void* V, int64_t T, int n_heads, int n_kv, int d,
                         float scale, float* out, void* ws, size_t ws_bytes, void* stream) {
    if (type != QK_Q8_0 && type != QK_Q5_0 && type != QK_Q4_0)
        return fail(QK_ERR_TYPE, "KV cache type %d: Q8_0, Q5_0 or Q4_0 expected", type);
    if (T < 1 || T > (int64_t)65535 * 256 || !qk::attn_decode_shape_ok(n_heads, n_kv, d))
        return fail(QK_ERR_SHAPE, "bad attention shape T=%lld n_heads=%d n_kv=%d d=%d", (long long)T, n_heads, n_kv, d);
    if (!q || !K || !V || !out || !ws) return fail(QK_ERR_NULL, "NULL pointer argument");
    if (!aligned(q, 4) || !aligned(out, 4) || !aligned(ws, 4) || !aligned(K, 16) || !aligned(V, 16))
        return fail(QK_ERR_ALIGN, "q, out and ws must be 4-byte aligned, K and V 16-byte aligned");
    const int64_t need = qk::attn_decode_ws_bytes(T, n_heads, d);
    if (ws_bytes < (size_t)need) return fail(QK_ERR_WORKSPACE, "workspace %zu bytes < %lld needed", ws_bytes, (long long)need);
    unsigned* status = nullptr;
    int sms = 0;
    const qk_status st = device_state(&status, &sms);
    if (st != QK_OK) return st;
    cudaError_t e = qk::launch_attn_decode(type, q, static_cast<const uint8_t*>(K), static_cast<const uint8_t*>(V), T,
                                           n_heads, n_kv, d, scale, out, static_cast<float*>(ws), status, sms,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_attn_decode launch");
    g_last_error.clear();
    return QK_OK;
}

size_t qk_gemv_workspace(int type, int64_t rows, int64_t cols, int64_t M) {
    if (!known_type(type) || rows <= 0 || cols <= 0 || M <= 0 || cols % block_elems(type) != 0) return 0;
    return (size_t)qk::plan_gemv(type, rows, cols, M, sm_count_or_default()).ws_bytes;
}

qk_status qk_gemv(int type, const void* W, int64_t rows, int64_t cols, const float* x, int64_t M, float* y,
                  void* ws, size_t ws_bytes, void* stream) {
    qk_status st = qk::gemv_check_args(type, W, rows, cols, x, M, y);
    if (st != QK_OK) return st;
    if (rows == 0 || M == 0) return QK_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, (size_t)(M * rows) * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e, "qk_gemv zero fill");
        return QK_OK;
    }
    unsigned* status = nullptr;
    int sms = 0;
    st = device_state(&status, &sms);
    if (st != QK_OK) return st;
    (void)ws;   // no shape needs one
    (void)ws_bytes;
    const qk::GemvPlan pl = qk::plan_gemv(type, rows, cols, M, sms);
    if (!pl.ok) return fail(QK_ERR_SHAPE, "rows=%lld cols=%lld: no GEMV launch fits", (long long)rows, (long long)cols);
    cudaError_t e = qk::launch_gemv(type, pl, static_cast<const uint8_t*>(W), rows, cols, x, M, y, status, s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_gemv launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_gemv_batch(int type, int n_mat, const void* const* W, const int64_t* rows, int64_t cols,
                        const float* x, float* const* y, void* stream) {
    if (!known_type(type)) return fail(QK_ERR_TYPE, "unknown quant type %d", type);
    if (n_mat < 1 || n_mat > QK_GEMV_BATCH_MAX)
        return fail(QK_ERR_ARG, "n_mat=%d outside 1..%d", n_mat, QK_GEMV_BATCH_MAX);
    if (!W || !rows || !y) return fail(QK_ERR_NULL, "W, rows or y array is NULL");
    int64_t total = 0;
    for (int i = 0; i < n_mat; ++i) {
        qk_status st = check_matrix(type, W[i], rows[i], cols);
        if (st != QK_OK) return st;
        if (rows[i] > 0) {
            if (!y[i]) return fail(QK_ERR_NULL, "y[%d] is NULL", i);
            if (!aligned(y[i], 4)) return fail(QK_ERR_ALIGN, "y[%d] is not 4-byte aligned", i);
        }
        total += rows[i];
    }
    if (total == 0) return QK_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0) {
        for (int i = 0; i < n_mat; ++i) {
            if (rows[i] == 0) continue;
            cudaError_t e = cudaMemsetAsync(y[i], 0, (size_t)rows[i] * sizeof(float), s);
            if (e != cudaSuccess) return cuda_fail(e, "qk_gemv_batch zero fill");
        }
        return QK_OK;
    }
    if (!x) return fail(QK_ERR_NULL, "x is NULL");
    if (!aligned(x, 16)) return fail(QK_ERR_ALIGN, "x is not 16-byte aligned");
    int sms = 0;
    unsigned* status = nullptr;
    qk_status st = device_state(&status, &sms);
    if (st != QK_OK) return st;
    cudaError_t e;
    if (!qk::hgemv_ok(type, n_mat, rows, cols, sms))
        return fail(QK_ERR_SHAPE, "cols=%lld: no batched GEMV launch fits", (long long)cols);
    e = qk::launch_hgemv(type, n_mat, reinterpret_cast<const uint8_t* const*>(W), rows, cols, x, y, sms, status, s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_gemv_batch launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_gemv_swiglu(int type, const void* Wg, const void* Wu, int64_t rows, int64_t cols, const float* x,
                         float* h, void* stream) {
    qk_status st = check_matrix(type, Wg, rows, cols);
    if (st != QK_OK) return st;
    st = check_matrix(type, Wu, rows, cols);
    if (st != QK_OK) return st;
    if (rows == 0) return QK_OK;
    if (!h) return fail(QK_ERR_NULL, "h is NULL");
    if (!aligned(h, 4)) return fail(QK_ERR_ALIGN, "h is not 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0) {   // g = u = 0, SiLU(0) * 0 = 0
        cudaError_t e = cudaMemsetAsync(h, 0, (size_t)rows * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e, "qk_gemv_swiglu zero fill");
        return QK_OK;
    }
    if (!x) return fail(QK_ERR_NULL, "x is NULL");
    if (!aligned(x, 16)) return fail(QK_ERR_ALIGN, "x is not 16-byte aligned");
    int sms = 0;
    unsigned* status = nullptr;
    st = device_state(&status, &sms);
    if (st != QK_OK) return st;
    if (!qk::hgemv_ok(type, 1, &rows, cols, sms))
        return fail(QK_ERR_SHAPE, "rows=%lld cols=%lld: no SwiGLU launch fits", (long long)rows, (long long)cols);
    const cudaError_t e = qk::launch_hgemv_swiglu(type, static_cast<const uint8_t*>(Wg), static_cast<const uint8_t*>(Wu),
                                                  rows, cols, x, h, sms, status, s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_gemv_swiglu launch");
    g_last_error.clear();
    return QK_OK;
}

size_t qk_gemm_workspace(int type, int64_t rows, int64_t cols, int64_t M) {
    if (!known_type(type) || rows <= 0 || cols <= 0 || M <= 0 || cols % block_elems(type) != 0) return 0;
    return (size_t)qk::plan_gemm(type, rows, cols, M, sm_count_or_default()).ws_bytes;
}

qk_status qk_gemm(int type, const void* W, int64_t rows, int64_t cols, const void* X_bf16, int64_t M, float* Y,
                  void* ws, size_t ws_bytes, void* stream) {
    qk_status st = check_matrix(type, W, rows, cols);
    if (st != QK_OK) return st;
    if (M < 0) return fail(QK_ERR_SHAPE, "negative M=%lld", (long long)M);
    if (rows == 0 || M == 0) return QK_OK;
    if (!Y) return fail(QK_ERR_NULL, "Y is NULL");
    if (!aligned(Y, 4)) return fail(QK_ERR_ALIGN, "Y is not 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0) {
        cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)(M * rows) * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e, "qk_gemm zero fill");
        return QK_OK;
    }
    if (!X_bf16) return fail(QK_ERR_NULL, "X is NULL");
    if (!aligned(X_bf16, 16)) return fail(QK_ERR_ALIGN, "X is not 16-byte aligned");
    if (rows > (int64_t)1 << 31 || M > (int64_t)1 << 31 || cols > (int64_t)1 << 31)
        return fail(QK_ERR_SHAPE, "qk_gemm: dimensions must be below 2^31");
    if ((rows + 127) / 128 > 65535)
        return fail(QK_ERR_SHAPE, "qk_gemm: rows=%lld above 65535 tiles of 128", (long long)rows);
    unsigned* status = nullptr;
    int sms = 0;
    st = device_state(&status, &sms);
    if (st != QK_OK) return st;
    const qk::GemmPlan pl = qk::plan_gemm(type, rows, cols, M, sms);
    if (pl.ws_bytes > 0) {
        if (ws_bytes < (size_t)pl.ws_bytes)
            return fail(QK_ERR_WORKSPACE, "workspace %zu bytes < %lld needed", ws_bytes, (long long)pl.ws_bytes);
        if (!ws) return fail(QK_ERR_NULL, "workspace is NULL");
        if (!aligned(ws, 16)) return fail(QK_ERR_ALIGN, "workspace is not 16-byte aligned");
    }
    cudaError_t e = qk::launch_gemm(type, pl, static_cast<const uint8_t*>(W), rows, cols, X_bf16, M, Y,
                                    static_cast<float*>(ws), status, s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_gemm launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_unpack(int type, const void* W, int64_t nblocks, int16_t* codes, int16_t* sc, uint8_t* mins, float* d,
                    float* dmin, void* stream) {
    if (!known_type(type)) return fail(QK_ERR_TYPE, "unknown quant type %d", type);
    if (nblocks < 0) return fail(QK_ERR_SHAPE, "negative nblocks");
    if (nblocks == 0) return QK_OK;
    if (!W) return fail(QK_ERR_NULL, "W is NULL");
    if (!aligned(W, 16)) return fail(QK_ERR_ALIGN, "W is not 16-byte aligned");
    cudaError_t e = qk::launch_unpack(type, static_cast<const uint8_t*>(W), nblocks, codes, sc, mins, d, dmin,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_unpack launch");
    return QK_OK;
}

qk_status qk_test_stalled_wait(uint32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 10000000u) return fail(QK_ERR_ARG, "limit_us=%u outside 1..10000000", limit_us);
    unsigned* status = nullptr;
    qk_status st = device_state(&status, nullptr);
    if (st != QK_OK) return st;
    cudaError_t e = qk::launch_stalled_wait(status, (uint64_t)limit_us * 1000u, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "qk_test_stalled_wait launch");
    g_last_error.clear();
    return QK_OK;
}

qk_status qk_device_status(void* stream) {
    unsigned* status = nullptr;
    qk_status st = device_state(&status, nullptr);
    if (st != QK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof v, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_device_status");
    if (v & 1u) return fail(QK_ERR_TIMEOUT, "a bounded wait inside a kernel ran out (status 0x%x)", v);
    return QK_OK;
}

}  // extern "C"
