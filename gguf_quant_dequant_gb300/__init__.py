"""Python binding of libqk (include/qk.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; this module passes
device pointers, sizes and the current CUDA stream of PyTorch tensors, and
raises QKError on a non-zero status.  There is no CPU fallback: if libqk.so
has not been built, load() raises.

Type ids: Q4_K = 1, Q6_K = 2, Q8_0 = 3, Q5_0 = 4, Q4_0 = 5, Q5_K = 6, Q2_K = 7, Q3_K = 8.
"""
from __future__ import annotations

import ctypes
import os
import threading

Q4_K, Q6_K, Q8_0, Q5_0, Q4_0, Q5_K, Q2_K, Q3_K = 1, 2, 3, 4, 5, 6, 7, 8
TYPES = {"Q4_K": Q4_K, "Q6_K": Q6_K, "Q8_0": Q8_0, "Q5_0": Q5_0, "Q4_0": Q4_0, "Q5_K": Q5_K, "Q2_K": Q2_K,
         "Q3_K": Q3_K}
OUT_F32, OUT_BF16 = 0, 1
STATUS = {0: "QK_OK", 1: "QK_ERR_TYPE", 2: "QK_ERR_SHAPE", 3: "QK_ERR_ALIGN", 4: "QK_ERR_NULL",
          5: "QK_ERR_WORKSPACE", 6: "QK_ERR_CUDA", 7: "QK_ERR_TIMEOUT", 8: "QK_ERR_ARG",
          9: "QK_ERR_FORMAT", 10: "QK_ERR_IO"}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqk.so")
_lib = None
_lock = threading.Lock()

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_int = ctypes.c_int
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u64p = ctypes.POINTER(ctypes.c_uint64)


class GGUFTensorInfo(ctypes.Structure):
    """qk_gguf_tensor_info."""
    _fields_ = [("name", ctypes.c_char_p), ("n_dims", ctypes.c_uint32), ("dims", ctypes.c_int64 * 4),
                ("ggml_type", ctypes.c_uint32), ("qk_type", ctypes.c_int), ("offset", ctypes.c_uint64),
                ("nbytes", ctypes.c_uint64), ("data", ctypes.c_void_p)]


# name: (restype, argtypes), exactly as declared in include/qk.h
SIGNATURES = {
    "qk_version": (_int, []),
    "qk_block_bytes": (_sz, [_int]),
    "qk_block_elems": (_int, [_int]),
    "qk_row_bytes": (_sz, [_int, _i64]),
    "qk_dequant": (_int, [_int, _p, _i64, _i64, _p, _int, _p]),
    "qk_quantize": (_int, [_int, _p, _i64, _i64, _p, _p]),
    "qk_quantize_imatrix": (_int, [_int, _p, _i64, _i64, _p, _p, _p]),
    "qk_attn_decode_workspace": (ctypes.c_size_t, [_int, _i64, _int, _int, _int]),
    "qk_attn_decode": (_int, [_int, _p, _p, _p, _i64, _int, _int, _int, ctypes.c_float, _p, _p, ctypes.c_size_t, _p]),
    "qk_gemv_workspace": (_sz, [_int, _i64, _i64, _i64]),
    "qk_gemv": (_int, [_int, _p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "qk_gemv_noalloc": (_int, [_int, _p, _i64, _i64, _p, _i64, _p, _p]),
    "qk_gemv_batch": (_int, [_int, _int, ctypes.POINTER(_p), ctypes.POINTER(_i64), _i64, _p,
                             ctypes.POINTER(_p), _p]),
    "qk_gemv_swiglu": (_int, [_int, _p, _p, _i64, _i64, _p, _p, _p]),
    "qk_gemm_workspace": (_sz, [_int, _i64, _i64, _i64]),
    "qk_gemm": (_int, [_int, _p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "qk_unpack": (_int, [_int, _p, _i64, _p, _p, _p, _p, _p, _p]),
    "qk_device_status": (_int, [_p]),
    "qk_test_stalled_wait": (_int, [ctypes.c_uint32, _p]),
    "qk_last_error": (ctypes.c_char_p, []),
    "qk_gguf_open": (_int, [ctypes.c_char_p, ctypes.POINTER(_p)]),
    "qk_gguf_parse": (_int, [_p, _u64, ctypes.POINTER(_p)]),
    "qk_gguf_close": (None, [_p]),
    "qk_gguf_version": (_u32, [_p]),
    "qk_gguf_n_kv": (_i64, [_p]),
    "qk_gguf_n_tensors": (_i64, [_p]),
    "qk_gguf_alignment": (_u64, [_p]),
    "qk_gguf_data_offset": (_u64, [_p]),
    "qk_gguf_image": (_p, [_p]),
    "qk_gguf_find_kv": (_i64, [_p, ctypes.c_char_p]),
    "qk_gguf_kv_key": (ctypes.c_char_p, [_p, _i64]),
    "qk_gguf_kv_type": (_int, [_p, _i64]),
    "qk_gguf_kv_int": (_int, [_p, _i64, _i64p]),
    "qk_gguf_kv_float": (_int, [_p, _i64, _f64p]),
    "qk_gguf_kv_str": (_p, [_p, _i64, _u64p]),
    "qk_gguf_kv_array": (_int, [_p, _i64, ctypes.POINTER(_int), _u64p]),
    "qk_gguf_kv_array_int": (_int, [_p, _i64, _u64, _i64p]),
    "qk_gguf_kv_array_float": (_int, [_p, _i64, _u64, _f64p]),
    "qk_gguf_kv_array_str": (_p, [_p, _i64, _u64, _u64p]),
    "qk_gguf_find_tensor": (_i64, [_p, ctypes.c_char_p]),
    "qk_gguf_tensor": (_int, [_p, _i64, ctypes.POINTER(GGUFTensorInfo)]),
}


class QKError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libqk.so (built in-tree by build.build()); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m gguf_quant_dequant_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(st: int, where: str) -> None:
    if st != 0:
        raise QKError(st, where, load().qk_last_error().decode())


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def block_bytes(t: int) -> int:
    return load().qk_block_bytes(t)


def block_elems(t: int) -> int:
    return load().qk_block_elems(t)


def row_bytes(t: int, cols: int) -> int:
    return load().qk_row_bytes(t, cols)


def dequant(t: int, W, rows: int, cols: int, out=None, bf16: bool = False, stream=None):
    """W: uint8 CUDA tensor of packed blocks -> out [rows, cols] fp32 / bf16."""
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16 if bf16 else torch.float32, device=W.device)
    _check(load().qk_dequant(t, _ptr(W), rows, cols, _ptr(out), OUT_BF16 if bf16 else OUT_F32,
                             _stream(stream)), "qk_dequant")
    return out


def quantize(t: int, w, out=None, stream=None):
    """w: fp32 CUDA tensor [rows, cols] -> out: uint8 packed blocks, rows *
    row_bytes(t, cols) bytes (allocated when not given)."""
    import torch
    rows, cols = w.shape
    if out is None:
        out = torch.empty(rows * row_bytes(t, cols), dtype=torch.uint8, device=w.device)
    _check(load().qk_quantize(t, _ptr(w), rows, cols, _ptr(out), _stream(stream)), "qk_quantize")
    return out


def quantize_imatrix(t: int, w, imp, out=None, stream=None):
    """w: fp32 CUDA [rows, cols], imp: fp32 CUDA [cols] column importances
    (mean squared activations) -> packed blocks minimising the
    importance-weighted error (qk_quantize_imatrix)."""
    import torch
    rows, cols = w.shape
    if out is None:
        out = torch.empty(rows * row_bytes(t, cols), dtype=torch.uint8, device=w.device)
    _check(load().qk_quantize_imatrix(t, _ptr(w), rows, cols, _ptr(imp), _ptr(out), _stream(stream)),
           "qk_quantize_imatrix")
    return out


def attn_decode_workspace(t: int, T: int, n_heads: int, n_kv: int, d: int) -> int:
    return load().qk_attn_decode_workspace(t, T, n_heads, n_kv, d)


def attn_decode(t: int, q, K, V, T: int, n_heads: int, n_kv: int, d: int, scale: float, out=None, ws=None,
                stream=None):
    """Decode attention over a block-quantized KV cache (qk_attn_decode):
    q fp32 CUDA [n_heads, d]; K, V packed caches [T, n_kv, d] -> out fp32
    [n_heads, d]."""
    import torch
    if out is None:
        out = torch.empty((n_heads, d), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace(t, T, n_heads, n_kv, d)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(load().qk_attn_decode(t, _ptr(q), _ptr(K), _ptr(V), T, n_heads, n_kv, d, scale, _ptr(out), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "qk_attn_decode")
    return out


def gemv_swiglu(t: int, Wg, Wu, rows: int, cols: int, x, h=None, stream=None):
    """Decode SwiGLU: x fp32 CUDA [cols] -> h = SiLU(Wg x) * (Wu x), fp32 [rows]."""
    import torch
    if h is None:
        h = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(load().qk_gemv_swiglu(t, _ptr(Wg), _ptr(Wu), rows, cols, _ptr(x), _ptr(h), _stream(stream)),
           "qk_gemv_swiglu")
    return h


def gemv_workspace(t: int, rows: int, cols: int, M: int) -> int:
    return load().qk_gemv_workspace(t, rows, cols, M)


def gemv(t: int, W, rows: int, cols: int, x, y=None, ws=None, stream=None):
    """x fp32 CUDA [M, cols] -> y fp32 [M, rows]; ws allocated if needed."""
    import torch
    M = x.shape[0] if x.dim() == 2 else 1
    if y is None:
        y = torch.empty((M, rows), dtype=torch.float32, device=x.device)
    need = gemv_workspace(t, rows, cols, M)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qk_gemv(t, _ptr(W), rows, cols, _ptr(x), M, _ptr(y), _ptr(ws), nbytes, _stream(stream)),
           "qk_gemv")
    return y


def gemv_noalloc(t: int, W, rows: int, cols: int, x, y=None, stream=None):
    """qk_gemv_noalloc: qk_gemv for callers that cannot allocate device
    memory (no workspace; the GEMV needs none)."""
    import torch
    M = x.shape[0] if x.dim() == 2 else 1
    if y is None:
        y = torch.empty((M, rows), dtype=torch.float32, device=x.device)
    _check(load().qk_gemv_noalloc(t, _ptr(W), rows, cols, _ptr(x), M, _ptr(y), _stream(stream)),
           "qk_gemv_noalloc")
    return y


def gemv_batch(t: int, Ws, rows, cols: int, x, ys=None, stream=None):
    """qk_gemv_batch: y_i = W_i x for matrices sharing one fp32 activation row
    x [cols] (or [1, cols]); returns the list of fp32 outputs [rows_i]."""
    import torch
    n = len(Ws)
    if ys is None:
        ys = [torch.empty(r, dtype=torch.float32, device=x.device) for r in rows]
    Wp = (_p * n)(*[_ptr(w) for w in Ws])
    rp = (_i64 * n)(*rows)
    yp = (_p * n)(*[_ptr(y) for y in ys])
    _check(load().qk_gemv_batch(t, n, Wp, rp, cols, _ptr(x), yp, _stream(stream)), "qk_gemv_batch")
    return ys


def gemm_workspace(t: int, rows: int, cols: int, M: int) -> int:
    return load().qk_gemm_workspace(t, rows, cols, M)


def gemm(t: int, W, rows: int, cols: int, X, Y=None, ws=None, stream=None):
    """X bf16 CUDA [M, cols] -> Y fp32 [M, rows]."""
    import torch
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, rows), dtype=torch.float32, device=X.device)
    need = gemm_workspace(t, rows, cols, M)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qk_gemm(t, _ptr(W), rows, cols, _ptr(X), M, _ptr(Y), _ptr(ws), nbytes, _stream(stream)),
           "qk_gemm")
    return Y


def unpack(t: int, W, nblocks: int, stream=None):
    """-> (codes int16 [nblocks, elems], sc int16 [nblocks, 16], mins uint8
    [nblocks, 16], d f32 [nblocks], dmin f32 [nblocks]) as CUDA tensors."""
    import torch
    dev = W.device
    codes = torch.empty((nblocks, block_elems(t)), dtype=torch.int16, device=dev)
    sc = torch.empty((nblocks, 16), dtype=torch.int16, device=dev)
    mins = torch.empty((nblocks, 16), dtype=torch.uint8, device=dev)
    d = torch.empty(nblocks, dtype=torch.float32, device=dev)
    dmin = torch.empty(nblocks, dtype=torch.float32, device=dev)
    _check(load().qk_unpack(t, _ptr(W), nblocks, _ptr(codes), _ptr(sc), _ptr(mins), _ptr(d), _ptr(dmin),
                            _stream(stream)), "qk_unpack")
    return codes, sc, mins, d, dmin


def test_stalled_wait(limit_us: int, stream=None) -> None:
    """qk_test_stalled_wait: a bounded wait on a barrier nothing arrives on."""
    _check(load().qk_test_stalled_wait(limit_us, _stream(stream)), "qk_test_stalled_wait")


def device_status(stream=None) -> None:
    _check(load().qk_device_status(_stream(stream)), "qk_device_status")


# ------------------------------------------------------------ GGUF reader --

_V_STR, _V_ARR, _V_F32, _V_F64 = 8, 9, 6, 12


class GGUF:
    """A parsed GGUF image (qk_gguf_*): header, metadata and tensor infos.
    Open a file (memory-mapped) with GGUF(path=...) or parse bytes the object
    keeps alive with GGUF(data=...).  Tensor data stays in the image."""

    def __init__(self, path: str | None = None, data: bytes | None = None):
        L = load()
        h = _p()
        self._buf = None
        if path is not None:
            _check(L.qk_gguf_open(os.fsencode(path), ctypes.byref(h)), "qk_gguf_open")
        else:
            self._buf = ctypes.create_string_buffer(bytes(data), len(data))
            _check(L.qk_gguf_parse(ctypes.cast(self._buf, _p), len(data), ctypes.byref(h)), "qk_gguf_parse")
        self._h = h

    def close(self) -> None:
        if self._h:
            load().qk_gguf_close(self._h)
            self._h = _p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def version(self) -> int:
        return load().qk_gguf_version(self._h)

    @property
    def alignment(self) -> int:
        return load().qk_gguf_alignment(self._h)

    @property
    def data_offset(self) -> int:
        return load().qk_gguf_data_offset(self._h)

    def keys(self) -> list:
        L = load()
        return [L.qk_gguf_kv_key(self._h, i).decode() for i in range(L.qk_gguf_n_kv(self._h))]

    def kv_type(self, key: str) -> int:
        L = load()
        return L.qk_gguf_kv_type(self._h, L.qk_gguf_find_kv(self._h, key.encode()))

    def _str(self, ptr, n) -> str:
        return ctypes.string_at(ptr, n.value).decode("utf-8", "surrogateescape") if n.value else ""

    def kv(self, key: str):
        """The value of `key` as int / float / str / list (KeyError if absent)."""
        L = load()
        i = L.qk_gguf_find_kv(self._h, key.encode())
        if i < 0:
            raise KeyError(key)
        t = L.qk_gguf_kv_type(self._h, i)
        n = ctypes.c_uint64()
        if t == _V_STR:
            return self._str(L.qk_gguf_kv_str(self._h, i, ctypes.byref(n)), n)
        if t in (_V_F32, _V_F64):
            v = ctypes.c_double()
            _check(L.qk_gguf_kv_float(self._h, i, ctypes.byref(v)), "qk_gguf_kv_float")
            return v.value
        if t == _V_ARR:
            et = _int()
            _check(L.qk_gguf_kv_array(self._h, i, ctypes.byref(et), ctypes.byref(n)), "qk_gguf_kv_array")
            out = []
            for j in range(n.value):
                if et.value == _V_STR:
                    m = ctypes.c_uint64()
                    out.append(self._str(L.qk_gguf_kv_array_str(self._h, i, j, ctypes.byref(m)), m))
                elif et.value in (_V_F32, _V_F64):
                    v = ctypes.c_double()
                    _check(L.qk_gguf_kv_array_float(self._h, i, j, ctypes.byref(v)), "qk_gguf_kv_array_float")
                    out.append(v.value)
                elif et.value == _V_ARR:
                    raise QKError(1, "GGUF.kv", "nested arrays are not exposed")
                else:
                    v = ctypes.c_int64()
                    _check(L.qk_gguf_kv_array_int(self._h, i, j, ctypes.byref(v)), "qk_gguf_kv_array_int")
                    out.append(v.value)
            return out
        v = ctypes.c_int64()
        _check(L.qk_gguf_kv_int(self._h, i, ctypes.byref(v)), "qk_gguf_kv_int")
        return v.value

    def tensors(self) -> list:
        L = load()
        return [self._info(i) for i in range(L.qk_gguf_n_tensors(self._h))]

    def _info(self, i: int) -> dict:
        info = GGUFTensorInfo()
        _check(load().qk_gguf_tensor(self._h, i, ctypes.byref(info)), "qk_gguf_tensor")
        return {"name": info.name.decode(), "dims": list(info.dims[:info.n_dims]), "ggml_type": info.ggml_type,
                "qk_type": info.qk_type, "offset": info.offset, "nbytes": info.nbytes, "data": info.data}

    def tensor(self, name: str) -> dict:
        i = load().qk_gguf_find_tensor(self._h, name.encode())
        if i < 0:
            raise KeyError(name)
        return self._info(i)

    def tensor_bytes(self, name: str) -> bytes:
        """A copy of the tensor's data bytes."""
        t = self.tensor(name)
        return ctypes.string_at(t["data"], t["nbytes"])
