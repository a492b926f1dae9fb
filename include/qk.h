/*
 * qk.h -- C ABI of libqk: matrix products over GGUF block-quantized weights
 * on one GB300 (sm_103a), with the blocks unpacked inside the dot product.
 *
 * Block formats (one block = a fixed number of weights along a row):
 *   Q4_K  256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes holding eight
 *         6-bit sub-block scales and eight 6-bit mins, 128 bytes of 4-bit
 *         codes; weight = (d*sc)*q - dmin*m.  ("Hitchhiker's Guide -- Lab 01:
 *         Air-Gapped LLM Serving", section 11.2, Q4_K super-block figure;
 *         "12 -- llama.cpp / GGUF / Local Inference Mastery", "Q4_K_M -- bit
 *         layout in exquisite detail", figure and dequantization pseudo-code.)
 *   Q6_K  256 weights in 210 bytes: 128 bytes of low code nibbles, 64 bytes
 *         of high code bit pairs, sixteen int8 scales (one per 16 weights),
 *         fp16 d; weight = d*sc*(q - 32).  ("12 -- llama.cpp / GGUF", "Other
 *         k-quants at a glance": 256-weight super-block, 6.6 bits/weight.)
 *   Q8_0  32 weights in 34 bytes: fp16 d, 32 int8 codes; weight = d*q.
 *         ("Hitchhiker's Guide", section 11.1: the Q4_0 structure with 8-bit
 *         codes.)
 *   Q5_0  32 weights in 22 bytes: fp16 d, a 32-bit word of fifth bits, 16
 *         bytes of nibbles; weight = d*(q - 16).  ("Local LLM inference",
 *         "The mmap backend": one of the block types of a Q4_K_M file.)
 *   Q4_0  32 weights in 18 bytes: fp16 d, 16 bytes of nibbles (low nibbles
 *         elements 0-15, high nibbles 16-31); weight = d*(q - 8).
 *         ("Hitchhiker's Guide", section 11.1, Q4_0 block figure; "How LLM
 *         Inference Engines Work", "Loading GGUF Models", the Q4_0
 *         dequantizer.)
 *   Q5_K  256 weights in 176 bytes: fp16 d, fp16 dmin, the 12 scale bytes
 *         of Q4_K, 32 bytes of fifth code bits (bit 2c + h of byte l for
 *         weight 64c + 32h + l), 128 bytes of low nibbles placed as Q4_K's
 *         codes; weight = (d*sc)*q - dmin*m, q in 0..31.  The pages give only
 *         its size ("12 -- llama.cpp / GGUF", "Other k-quants at a glance":
 *         256-weight super-block, 5.5-5.7 bits/weight); the layout is the
 *         GGUF k-quant one.
 *   Q2_K  256 weights in 84 bytes, sixteen 16-weight groups: 16 bytes of
 *         (4-bit scale, 4-bit min) per group, 64 bytes of 2-bit codes (code
 *         l of group 8t + 2j + k is bits 2j.. of byte 32t + 16k + l), fp16 d,
 *         fp16 dmin; weight = (d*sc)*q - dmin*m.  (Pages: 2.5-2.6 bits/weight
 *         on 256-weight super-blocks, same table; layout: GGUF.)
 *   Q3_K  256 weights in 110 bytes: 32 bytes of high-bit mask, 64 bytes of
 *         2-bit codes placed as Q2_K's, 12 bytes of sixteen 6-bit scales
 *         (stored + 32), fp16 d; a code is its 2 bits minus 4 unless its
 *         mask bit (bit 4t + j of byte 16k + l) is set; weight = (d*sc)*q.
 *         (Pages: 3.4-4.0 bits/weight, same table; layout: GGUF.)
 * The bit placement inside the Q4_K scale bytes, the Q6_K code bytes and the
 * Q5_0 block is the k-quant / GGUF packing: low nibbles of a group of bytes
 * are the first weights, high nibbles the next ("How LLM Inference Engines
 * Work", "Loading GGUF Models").
 *
 * Matrix layout: a weight matrix W has `rows` output rows and `cols` inputs.
 * Each row is cols / block_elems blocks laid back to back along cols; row r
 * starts at byte r * qk_row_bytes(type, cols).  Rows follow each other with
 * no padding (so Q6_K rows of 11008 weights start at 9030-byte steps, not on
 * 16-byte boundaries).
 *
 * Ownership and memory: every pointer argument is DEVICE memory owned by the
 * caller, except where a function says otherwise.  The library allocates no
 * device memory; scratch space comes from the caller as a workspace.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Every compute call is asynchronous on it and returns once the work is
 * queued.  Argument errors are detected on the host before anything is
 * queued; nothing is launched when a call returns an error.
 *
 * Errors: every call returns a qk_status; qk_last_error() gives a text for
 * the last failure on the calling thread.  Waits inside the kernels are
 * bounded; a wait that runs out sets a device status word instead of
 * hanging, and qk_device_status() reports it as QK_ERR_TIMEOUT.
 */
#ifndef QK_H_
#define QK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Quant types.  The numbers are this library's own. */
typedef enum {
    QK_Q4_K = 1, QK_Q6_K = 2, QK_Q8_0 = 3, QK_Q5_0 = 4, QK_Q4_0 = 5, QK_Q5_K = 6, QK_Q2_K = 7, QK_Q3_K = 8
} qk_type;

typedef enum {
    QK_OK = 0,
    QK_ERR_TYPE = 1,      /* unknown quant type                                 */
    QK_ERR_SHAPE = 2,     /* negative size, cols not a multiple of block_elems  */
    QK_ERR_ALIGN = 3,     /* a pointer breaks its stated alignment              */
    QK_ERR_NULL = 4,      /* a required pointer is NULL                         */
    QK_ERR_WORKSPACE = 5, /* workspace smaller than the matching *_workspace()  */
    QK_ERR_CUDA = 6,      /* the CUDA runtime reported an error                 */
    QK_ERR_TIMEOUT = 7,   /* a bounded wait inside a kernel ran out             */
    QK_ERR_ARG = 8,       /* any other invalid argument                         */
    QK_ERR_FORMAT = 9,    /* a GGUF image is malformed or truncated             */
    QK_ERR_IO = 10        /* a file could not be opened or mapped               */
} qk_status;

/* Output element types of qk_dequant. */
enum { QK_OUT_F32 = 0, QK_OUT_BF16 = 1 };

/* Version of this ABI. */
int qk_version(void);

/* Bytes per block (144, 210, 34, 22) and weights per block (256, 256, 32,
 * 32); 0 for an unknown type.  ("Hitchhiker's Guide", 11.2: 144 bytes =
 * 4.5 bits per weight.) */
size_t qk_block_bytes(int type);
int qk_block_elems(int type);

/* Bytes of one row of `cols` weights; 0 for an unknown type or when cols is
 * not a multiple of the block size. */
size_t qk_row_bytes(int type, int64_t cols);

/* Dequantize W [rows, cols] into out [rows, cols] row-major, as fp32
 * (out_dtype QK_OUT_F32) or bf16 (QK_OUT_BF16, round to nearest even).
 * Each weight is computed in fp32 by the type's formula above, in the order
 * written ((d*sc)*q - dmin*m for Q4_K); fp32 results are exact except for
 * the final subtraction of Q4_K.
 * W: 16-byte aligned.  out: 16-byte aligned.  rows == 0 queues nothing. */
qk_status qk_dequant(int type, const void* W, int64_t rows, int64_t cols,
                     void* out, int out_dtype, void* stream);

/* Quantize fp32 weights into packed blocks: the write side of the format.
 * The pages name the k-quant quantizer ("12 -- llama.cpp / GGUF / Local
 * Inference Mastery", reading list: quantize_row_q4_K) without giving it,
 * and describe plain quantization as minimising the weight-space error
 * ("Hitchhiker's Guide -- Lab 01", 11.3); this is the plain min/max scheme,
 * each quotient an IEEE fp32 division and each code clamp(round half away
 * from zero(quotient)):
 *   Q4_K per 32-weight sub-block: lo = min(0, min w), hi = max w,
 *        sc_f = (hi - lo)/15, m_f = -lo; d = fp16(max sc_f / 63),
 *        dmin = fp16(max m_f / 63); sc = cr(sc_f/d, 0..63),
 *        m = cr(m_f/dmin, 0..63); q = cr((w + dmin*m) / (d*sc), 0..15).
 *   Q5_K the same with 31 in place of 15.
 *   Q2_K per 16 weights: the Q4_K scheme with 3 in place of 15 and 4-bit
 *        sc, m (d = fp16(max sc_f / 15), dmin = fp16(max m_f / 15)).
 *   Q3_K per 16 weights: s = max|w| / 4, d = fp16(max s / 31),
 *        sc = cr(s/d, -32..31), q = cr(w / (d*sc), -4..3).
 *   Q6_K per 16 weights: s = max|w| / 32, d = fp16(max s / 127),
 *        sc = cr(s/d, -128..127), q = cr(w / (d*sc), -32..31) + 32.
 *   Q8_0 / Q5_0 / Q4_0 per 32: d = fp16(max|w| / 127 | 15 | 7),
 *        q = cr(w/d) + 0 | 16 | 8, clamped to the code range.
 * A zero divisor gives the offset code; NaN inputs are not rejected (they are
 * skipped by the maxima and a NaN quotient takes the lowest code).
 *   w   fp32 [rows, cols] row-major, 16-byte aligned.
 *   out rows * qk_row_bytes(type, cols) bytes, 4-byte aligned; fully
 *       overwritten.
 * Deterministic; the bytes do not depend on the launch.  rows == 0 or
 * cols == 0 queues nothing.  Errors: QK_ERR_TYPE, QK_ERR_SHAPE (cols not a
 * multiple of the block size, negative sizes), QK_ERR_NULL, QK_ERR_ALIGN. */
qk_status qk_quantize(int type, const float* w, int64_t rows, int64_t cols, void* out, void* stream);

/* Decode attention over a block-quantized KV cache ("Hitchhiker's Guide --
 * Lab 01", 13.2: K and V cached as q8_0, or q4_0 at a quality cost, and read
 * inside attention; grouped-query attention shares each kv head among
 * n_heads / n_kv query heads).  One query token:
 *   s_t = scale * sum_i q[h, i] K[t, g, i],  g = h / (n_heads / n_kv),
 *   p = softmax(s) over t = 0 .. T-1,  out[h, i] = sum_t p_t V[t, g, i].
 *   type   QK_Q8_0, QK_Q5_0 or QK_Q4_0 (the cache's block type).
 *   q      fp32 [n_heads, d], device, 4-byte aligned.
 *   K, V   [T, n_kv, d]: each (t, g) row is d / 32 blocks (so a cache row
 *          of all kv heads is qk_row_bytes(type, n_kv * d) bytes, written by
 *          qk_quantize from fp32 [T, n_kv * d]); device, 16-byte aligned.
 *   d      32, 64, 128 or 256; n_heads a multiple of n_kv, at most 8 query
 *          heads per kv head; 1 <= T <= 65535 * 256.
 *   out    fp32 [n_heads, d]; ws at least qk_attn_decode_workspace bytes.
 * Positions are split over CTAs (one CTA per kv head and range of
 * positions, about T / (2 SMs / n_kv) of them; shapes whose per-thread state
 * does not fit take chunks of 192 or 256), the cache streamed once; each
 * range keeps its max score, sum of exponentials and weighted value sum, and
 * a second launch combines the ranges (log-sum-exp) in a fixed order:
 * deterministic.  Scores on the fp16 tensor-core MMA (exact codes, each
 * query element as two fp16 terms after a power-of-two scale per 32-block),
 * fp32 softmax; the p V sums in fp32, or for Q8_0 / Q4_0 with d = 128 and
 * up to four query heads per kv head on the MMA with p d as two fp16 terms
 * after a power-of-two scale per 128 positions.  Accuracy: |out - out_exact|
 * <= 2e-4 * sum_t p_t |V[t, g, i]| + 1e-6.
 * Errors: QK_ERR_TYPE, QK_ERR_SHAPE, QK_ERR_NULL, QK_ERR_ALIGN,
 * QK_ERR_WORKSPACE. */
size_t qk_attn_decode_workspace(int type, int64_t T, int n_heads, int n_kv, int d);
qk_status qk_attn_decode(int type, const float* q, const void* K, const void* V, int64_t T, int n_heads, int n_kv, int d,
                         float scale, float* out, void* ws, size_t ws_bytes, void* stream);

/* Importance-weighted quantization ("Hitchhiker's Guide -- Lab 01", 11.3,
 * the importance matrix: minimise sum_i E[x_i^2] (w_i - w^_i)^2 rather than
 * the plain weight-space error).  imp[c] is the mean squared activation met
 * by weight column c (fp32 [cols], finite and >= 0; the same for every row).
 * The page gives the objective, not the search; per group (the 32-weight
 * block of Q8_0 / Q5_0 / Q4_0, the 32-weight sub-block of Q4_K / Q5_K, the
 * 16-weight group of Q6_K / Q3_K / Q2_K):
 *   s0 (and m0) = the plain quantizer's group scale (and min); for k = 0..20
 *   the candidate scale s0 * (90 + k) / 100 rounds the codes, a weighted
 *   least-squares refit gives the scale (scale and min jointly where the type
 *   has a min; kept only with a positive determinant, a positive scale and a
 *   non-negative min), and the candidate of least weighted error wins (the
 *   first on ties).  The block is then assembled as by qk_quantize with
 *   those group values, and kept only if its weighted error (summed per
 *   group, then over groups) is no more than the plain block's; otherwise
 *   the plain block is written.  fp32 throughout, sums in index order, so
 *   the bytes are deterministic.  All-zero importances give qk_quantize's
 *   bytes.
 *   w    device fp32 [rows, cols], 16-byte aligned.
 *   imp  device fp32 [cols], 4-byte aligned.
 *   out  rows * qk_row_bytes(type, cols) bytes, 4-byte aligned.
 * One lane per 32 weights (it searches its own groups; the codes of a
 * candidate take one reciprocal of its scale, with the division's rounding
 * reproduced exactly), a warp per 32 groups.
 * Errors as qk_quantize. */
qk_status qk_quantize_imatrix(int type, const float* w, int64_t rows, int64_t cols, const float* imp, void* out,
                              void* stream);

/* Fused decode FFN gate: h[n] = SiLU(g[n]) * u[n] with g = Wg x, u = Wu x
 * (batch 1) and SiLU(z) = z / (1 + e^-z) ("How LLM Inference Engines
 * Work", "SwiGLU Feed-Forward Network": the gate projection passes through
 * SiLU and multiplies the up projection element-wise; SiLU is not written
 * out on the page, the standard z * sigmoid(z) is used).  One launch: the
 * same CTAs walk their rows of Wg and then of Wu (x prepared once), and
 * write h only; g and u never reach memory.
 *   Wg, Wu [rows, cols] packed blocks of the same type, 16-byte aligned.
 *   x      fp32 [cols], 16-byte aligned.
 *   h      fp32 [rows], 4-byte aligned; fully overwritten.
 * Accuracy: g and u each as qk_gemv (1e-4 * sum|w x| + 1e-6), then the fp32
 * epilogue (expf, one division, one product).  No limit on cols beyond the
 * format's.
 * rows == 0 queues nothing; cols == 0 zero-fills h. */
qk_status qk_gemv_swiglu(int type, const void* Wg, const void* Wu, int64_t rows, int64_t cols,
                         const float* x, float* h, void* stream);

/* Workspace bytes qk_gemv needs for this problem: 0 for every shape (the
 * kernel prepares its activations in shared memory).  Kept so that callers
 * written against a workspace-taking GEMV need no change. */
size_t qk_gemv_workspace(int type, int64_t rows, int64_t cols, int64_t M);

/* Fused dequant-GEMV: y[m, n] = sum_k w[n, k] * x[m, k] for m < M,
 * n < rows, with every weight unpacked in registers inside the dot product
 * and never written out ("Local LLM inference", "The mmap backend": blocks
 * dequantized inside the dot product; each weight decoded once per input
 * batch and reused across its rows).  fp32 activations, fp32 accumulation.
 *   W  [rows, cols] packed blocks, 16-byte aligned.
 *   x  fp32 [M, cols] row-major, 16-byte aligned.
 *   y  fp32 [M, rows] row-major, 4-byte aligned; fully overwritten.
 *   ws, ws_bytes  ignored (no shape needs a workspace; NULL, 0 is fine).
 * Kernel: the fp16 warp MMA with exact integer codes (the code minus an
 * integer offset) and x as two fp16 terms per element after a power-of-two
 * scale per 32-element block; one launch for M == 1, one per pair of
 * activation rows otherwise (each launch streams W once).
 * Accuracy: |y - y_exact| <= 1e-4 * sum_k |w x| + 1e-6 per output.  The
 * per-element error model behind it: |x - (hi + lo) 2^e| <= 2^-22 |x| +
 * 2^(e-25), with 2^e <= 2^-14 times the block's largest magnitude when e > 0
 * (so elements down to 2^-17 of that magnitude keep 22 significant bits);
 * codes are exact, and a weight that is exactly zero contributes exactly
 * zero.  So blocks holding massive activations (tested at 1e3, 1e4
 * and 1e5 times the others, beside zero and tiny weights) stay within the
 * bound; the remaining terms are fp32 roundings of the block sums and scales.
 * Results are deterministic run to run (fixed reduction order).
 * rows == 0 or M == 0 queues nothing; cols == 0 zero-fills y. */
qk_status qk_gemv(int type, const void* W, int64_t rows, int64_t cols,
                  const float* x, int64_t M, float* y,
                  void* ws, size_t ws_bytes, void* stream);

/* Most matrices one qk_gemv_batch call takes. */
#define QK_GEMV_BATCH_MAX 8

/* Decode GEMV over several matrices that read the same activation vector, in
 * one launch: y_i[n] = sum_k W_i[n, k] * x[k] for i < n_mat, n < rows[i].
 * In a decoder layer the query, key and value projections are applied to the
 * same hidden state ("How LLM Inference Engines Work", Grouped-Query
 * Attention (GQA) and KV Cache), and so are the gate and up projections of
 * the feed-forward block (same page, SwiGLU Feed-Forward Network).  One call
 * per such group prepares x once and spreads the rows of all its matrices
 * over the GPU, instead of paying a launch and a ramp per matrix.
 *   type, cols  common to all matrices.
 *   W     host array of n_mat device pointers, W[i] = packed blocks
 *         [rows[i], cols], 16-byte aligned.
 *   rows  host array of n_mat row counts (0 allowed: that matrix is skipped).
 *   x     fp32 [cols] (one activation row), 16-byte aligned, device.
 *   y     host array of n_mat device pointers, y[i] = fp32 [rows[i]], 4-byte
 *         aligned; fully overwritten.
 * The host arrays are read during the call only.  No workspace, no limit on
 * cols beyond the format's.  n_mat outside 1..QK_GEMV_BATCH_MAX is
 * QK_ERR_ARG.  Kernel, accuracy and determinism as qk_gemv with M == 1. */
qk_status qk_gemv_batch(int type, int n_mat, const void* const* W, const int64_t* rows, int64_t cols,
                        const float* x, float* const* y, void* stream);

/* qk_gemv for callers that cannot allocate device memory.  The pages have no
 * counterpart; this is a convenience of this library.  Some callers of a
 * decode GEMV are not allowed to allocate: plug-in code running inside a
 * host runtime that owns every device allocation, code under a fixed memory
 * budget that must not grow its footprint while serving, and paths that
 * cannot afford the device-wide synchronization that cudaMalloc / cudaFree
 * can cause.  They call this instead of qk_gemv and pass no workspace.
 *   Arguments, results, accuracy and errors are those of qk_gemv; argument
 *   errors are reported exactly as qk_gemv reports them.
 *   Scratch: none.  The GEMV kernel prepares its activations in shared
 *   memory, so no shape needs a workspace; this call allocates nothing and
 *   holds no device memory of its own.
 *   Set-up: the first qk_* call on a device looks up the library's device
 *   status word; make it before starting any stream capture.  A
 *   cudaDeviceReset() unloads the module and leaves that address stale, so
 *   make no qk_* call on a device after resetting it. */
qk_status qk_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols,
                          const float* x, int64_t M, float* y, void* stream);

/* Workspace bytes qk_gemm needs (0 when none). */
size_t qk_gemm_workspace(int type, int64_t rows, int64_t cols, int64_t M);

/* Tensor-core dequant-GEMM for prefill: Y[m, n] = sum_k w[n, k] * X[m, k]
 * with X in bf16 and fp32 accumulation; weight tiles are unpacked to bf16 in
 * shared memory and fed to the tensor cores.  ("12 -- llama.cpp / GGUF":
 * prompt processing is big GEMMs of high arithmetic intensity.)
 *   W  [rows, cols] packed blocks, 16-byte aligned.
 *   X  bf16 [M, cols] row-major, 16-byte aligned; cols * 2 bytes must be a
 *      multiple of 16 (always true: cols is a multiple of 32).
 *   Y  fp32 [M, rows] row-major, 16-byte aligned; fully overwritten.
 *   ws as for qk_gemv.
 * Accuracy: |Y - Y_exact(bf16 X)| <= 5e-3 * sum_k |w x|; the weights are
 * rounded to bf16 before the product (Q8_0, Q5_0 and Q6_K codes and most
 * Q4_K weights are exact in bf16 up to the block scale).
 * M == 0 or rows == 0 queues nothing; cols == 0 zero-fills Y.  rows above
 * 65535 * 128 = 8,388,480 is QK_ERR_SHAPE. */
qk_status qk_gemm(int type, const void* W, int64_t rows, int64_t cols,
                  const void* X_bf16, int64_t M, float* Y,
                  void* ws, size_t ws_bytes, void* stream);

/* Test hook: unpack nblocks consecutive blocks into their integer fields.
 *   codes int16 [nblocks * block_elems]: Q4_K 0..15, Q5_K 0..31, Q6_K 0..63,
 *         Q8_0 -128..127, Q5_0 0..31, Q4_0 0..15, Q2_K 0..3, Q3_K -4..3.
 *   sc    int16 [nblocks * 16]: Q4_K / Q5_K 6-bit scales in slots 0..7, Q6_K
 *         the sixteen int8 scales, Q2_K the 4-bit scales, Q3_K the scales
 *         (-32..31); other slots and types 0.
 *   mins  uint8 [nblocks * 16]: Q4_K / Q5_K 6-bit mins (8 used), Q2_K 4-bit
 *         mins; 0 elsewhere.
 *   d, dmin fp32 [nblocks]: the decoded binary16 fields (dmin 0 unless the
 *         type has one: Q4_K, Q5_K, Q2_K).
 * All outputs device memory, any may be NULL.  W 16-byte aligned. */
qk_status qk_unpack(int type, const void* W, int64_t nblocks, int16_t* codes,
                    int16_t* sc, uint8_t* mins, float* d, float* dmin, void* stream);

/* Diagnostic of the failure-detection path; the pages have no counterpart.
 * Every mbarrier wait inside the library's kernels is bounded (2 s): when it
 * runs out the kernel records a timeout in the device status word, drains
 * its copies in flight, releases its tensor memory and returns, so the
 * context stays usable.  This call queues one thread that waits, through
 * the same bounded wait, on a barrier nothing arrives on, with the limit
 * shortened to limit_us microseconds (1 .. 10,000,000; else QK_ERR_ARG).
 * Afterwards qk_device_status() reports QK_ERR_TIMEOUT (and clears it). */
qk_status qk_test_stalled_wait(uint32_t limit_us, void* stream);

/* Synchronize `stream`, then read and clear this device's kernel status
 * word: QK_OK, or QK_ERR_TIMEOUT when a bounded wait ran out since the last
 * call (the affected outputs are then invalid). */
qk_status qk_device_status(void* stream);

/* ------------------------------------------------------------------------
 * GGUF container reader (host code; no GPU involved).  The file the blocks
 * come in ("12 -- llama.cpp / GGUF / Local Inference Mastery", "Part 1 --
 * The GGUF format (bit-level)"): header (magic "GGUF", version uint32,
 * tensor_count uint64, metadata_kv_count uint64), metadata entries
 * (length-prefixed key, value type, value), tensor infos (name, n_dims,
 * shape, ggml type, offset), padding to the alignment, tensor data.
 * Versions 2 and 3, little-endian.  The value-type codes (0 u8, 1 i8, 2 u16,
 * 3 i16, 4 u32, 5 i32, 6 f32, 7 bool, 8 string, 9 array, 10 u64, 11 i64,
 * 12 f64), the ggml tensor types (0 F32, 1 F16, 2 Q4_0, 6 Q5_0, 8 Q8_0,
 * 10 Q2_K, 11 Q3_K, 12 Q4_K, 13 Q5_K, 14 Q6_K, 30 BF16 are sized here;
 * others are listed with nbytes 0)
 * and the "general.alignment" key (uint32 power of two, default 32) follow
 * the GGUF specification the page cites.
 * Every length, count and offset is checked against the image before use;
 * a malformed or truncated image gives QK_ERR_FORMAT and no handle.  Tensor
 * data is never copied: qk_gguf_tensor gives a pointer into the image.  A
 * handle is read-only and may be used from several threads. */
typedef struct qk_gguf qk_gguf;

typedef struct {
    const char* name;      /* NUL-terminated, valid while the handle is open      */
    uint32_t n_dims;       /* 1..4                                                */
    int64_t dims[4];       /* dims[0] innermost (a weight matrix: cols, rows); 1 past n_dims */
    uint32_t ggml_type;
    int qk_type;           /* this library's type id (QK_Q4_K ...), -1 for others */
    uint64_t offset;       /* absolute byte offset in the image                   */
    uint64_t nbytes;       /* data bytes; 0 when the type's size is not known here */
    const void* data;      /* image + offset                                      */
} qk_gguf_tensor_info;

/* Open `path` read-only (memory-mapped) and parse it.  *out is NULL on error
 * (QK_ERR_IO, QK_ERR_FORMAT, QK_ERR_NULL). */
qk_status qk_gguf_open(const char* path, qk_gguf** out);
/* Parse an image the caller owns; it must outlive the handle. */
qk_status qk_gguf_parse(const void* data, uint64_t size, qk_gguf** out);
/* Release the handle (and its mapping).  NULL is ignored. */
void qk_gguf_close(qk_gguf* g);

uint32_t qk_gguf_version(const qk_gguf* g);
int64_t qk_gguf_n_kv(const qk_gguf* g);
int64_t qk_gguf_n_tensors(const qk_gguf* g);
uint64_t qk_gguf_alignment(const qk_gguf* g);
uint64_t qk_gguf_data_offset(const qk_gguf* g);   /* start of the tensor data section */
const void* qk_gguf_image(const qk_gguf* g);

/* Metadata entry i (0 .. n_kv-1); the index of `key`, or -1. */
int64_t qk_gguf_find_kv(const qk_gguf* g, const char* key);
const char* qk_gguf_kv_key(const qk_gguf* g, int64_t i);   /* NULL when out of range */
int qk_gguf_kv_type(const qk_gguf* g, int64_t i);          /* -1 when out of range */
/* Scalar values: integers of any width and bools as int64 (a uint64 above
 * INT64_MAX gives QK_ERR_TYPE), floats as double; QK_ERR_TYPE for another
 * type, QK_ERR_ARG for a bad index. */
qk_status qk_gguf_kv_int(const qk_gguf* g, int64_t i, int64_t* v);
qk_status qk_gguf_kv_float(const qk_gguf* g, int64_t i, double* v);
/* A string value (not NUL-terminated: *len bytes), NULL when not a string. */
const char* qk_gguf_kv_str(const qk_gguf* g, int64_t i, uint64_t* len);
/* Arrays: element type and count; element j as int64 / double / string. */
qk_status qk_gguf_kv_array(const qk_gguf* g, int64_t i, int* elem_type, uint64_t* n);
qk_status qk_gguf_kv_array_int(const qk_gguf* g, int64_t i, uint64_t j, int64_t* v);
qk_status qk_gguf_kv_array_float(const qk_gguf* g, int64_t i, uint64_t j, double* v);
const char* qk_gguf_kv_array_str(const qk_gguf* g, int64_t i, uint64_t j, uint64_t* len);

/* Tensor i (0 .. n_tensors-1); the index of `name`, or -1. */
int64_t qk_gguf_find_tensor(const qk_gguf* g, const char* name);
qk_status qk_gguf_tensor(const qk_gguf* g, int64_t i, qk_gguf_tensor_info* info);

/* Text of the last error on the calling thread ("" if none). */
const char* qk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* QK_H_ */
