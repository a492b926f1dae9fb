"""Plain CPU oracle for GGUF block-quantized weights (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product: the two share no code.

The arithmetic lives in ``qk_oracle.c`` (scalar C, fp32 weights in the order
the formulas state, fp64 accumulation).  This module compiles it with gcc on
first use and wraps it with numpy in / numpy out functions.

Type ids: Q4_K=1, Q6_K=2, Q8_0=3, Q5_0=4, Q4_0=5, Q5_K=6, Q2_K=7, Q3_K=8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K, Q6_K, Q8_0, Q5_0, Q4_0, Q5_K, Q2_K, Q3_K = 1, 2, 3, 4, 5, 6, 7, 8
TYPES = {"Q4_K": Q4_K, "Q6_K": Q6_K, "Q8_0": Q8_0, "Q5_0": Q5_0, "Q4_0": Q4_0, "Q5_K": Q5_K, "Q2_K": Q2_K,
         "Q3_K": Q3_K}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile qk_oracle.c into liboracle.so beside it (plain -O2, no fast-math,
    no fused multiply-add contraction, no ISA-specific flags)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.oq_block_bytes.argtypes = [ctypes.c_int]
            L.oq_block_elems.argtypes = [ctypes.c_int]
            L.oq_half_to_float.argtypes = [ctypes.c_uint16]
            L.oq_half_to_float.restype = ctypes.c_float
            L.oq_float_to_half.argtypes = [ctypes.c_float]
            L.oq_float_to_half.restype = ctypes.c_uint16
            L.oq_float_to_bf16.argtypes = [ctypes.c_float]
            L.oq_float_to_bf16.restype = ctypes.c_uint16
            L.oq_bf16_to_float.argtypes = [ctypes.c_uint16]
            L.oq_bf16_to_float.restype = ctypes.c_float
            L.oq_unpack.argtypes = [ctypes.c_int, _p, _i64, _p, _p, _p, _p, _p]
            L.oq_dequant.argtypes = [ctypes.c_int, _p, _i64, _i64, _p]
            L.oq_gemv.argtypes = [ctypes.c_int, _p, _i64, _i64, _p, _i64, _p, _p]
            L.oq_gemm_bf16.argtypes = [ctypes.c_int, _p, _i64, _i64, _p, _i64, _p, _p]
            L.oq_entries.argtypes = [ctypes.c_int, _p, _i64, _i64, _p, _p, _i64,
                                     _p, _p, _i64, _p, _p]
            L.oq_pack.argtypes = [ctypes.c_int, _i64, _p, _p, _p, _p, _p, _p]
            L.oq_quantize.argtypes = [ctypes.c_int, _p, _i64, _i64, _p]
            L.oq_quantize_imatrix.argtypes = [ctypes.c_int, _p, _i64, _i64, _p, _p]
            L.oq_attn_decode.argtypes = [ctypes.c_int, _p, _p, _p, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_float, _p, _p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def block_bytes(t: int) -> int:
    return lib().oq_block_bytes(t)


def block_elems(t: int) -> int:
    return lib().oq_block_elems(t)


def row_bytes(t: int, cols: int) -> int:
    return cols // block_elems(t) * block_bytes(t)


def half_to_float(bits: int) -> float:
    return lib().oq_half_to_float(bits)


def float_to_half(v: float) -> int:
    return lib().oq_float_to_half(v)


def float_to_bf16(v: float) -> int:
    return lib().oq_float_to_bf16(v)


def bf16_to_float(bits: int) -> float:
    return lib().oq_bf16_to_float(bits)


def float_to_bf16_array(a: np.ndarray) -> np.ndarray:
    """Element-wise fp32 -> bf16 bits (uint16), via the oracle's rounding."""
    L = lib()
    flat = np.ascontiguousarray(a, dtype=np.float32).ravel()
    out = np.fromiter((L.oq_float_to_bf16(float(v)) for v in flat), dtype=np.uint16,
                      count=flat.size)
    return out.reshape(np.shape(a))


def unpack(t: int, blocks: np.ndarray, nblocks: int):
    """Returns (codes int16 [nblocks, elems], sc int16 [nblocks, 16],
    mins uint8 [nblocks, 16], d f32 [nblocks], dmin f32 [nblocks])."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size >= nblocks * block_bytes(t)
    be = block_elems(t)
    codes = np.zeros((nblocks, be), np.int16)
    sc = np.zeros((nblocks, 16), np.int16)
    mins = np.zeros((nblocks, 16), np.uint8)
    d = np.zeros(nblocks, np.float32)
    dmin = np.zeros(nblocks, np.float32)
    _check(lib().oq_unpack(t, _ptr(blocks), nblocks, _ptr(codes), _ptr(sc), _ptr(mins),
                           _ptr(d), _ptr(dmin)), "unpack")
    return codes, sc, mins, d, dmin


def pack(t: int, codes: np.ndarray, sc: np.ndarray | None = None, mins: np.ndarray | None = None,
         d_bits: np.ndarray | None = None, dmin_bits: np.ndarray | None = None) -> np.ndarray:
    be, bb = block_elems(t), block_bytes(t)
    codes = np.ascontiguousarray(codes, dtype=np.int16).reshape(-1, be)
    nb = codes.shape[0]
    sc = np.zeros((nb, 16), np.int16) if sc is None else np.ascontiguousarray(sc, np.int16).reshape(nb, 16)
    mins = np.zeros((nb, 16), np.uint8) if mins is None else np.ascontiguousarray(mins, np.uint8).reshape(nb, 16)
    d_bits = np.zeros(nb, np.uint16) if d_bits is None else np.ascontiguousarray(d_bits, np.uint16).reshape(nb)
    dmin_bits = (np.zeros(nb, np.uint16) if dmin_bits is None
                 else np.ascontiguousarray(dmin_bits, np.uint16).reshape(nb))
    out = np.zeros(nb * bb, np.uint8)
    _check(lib().oq_pack(t, nb, _ptr(codes), _ptr(sc), _ptr(mins), _ptr(d_bits), _ptr(dmin_bits),
                         _ptr(out)), "pack")
    return out


def dequant(t: int, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= rows * row_bytes(t, cols)
    out = np.zeros((rows, cols), np.float32)
    _check(lib().oq_dequant(t, _ptr(W), rows, cols, _ptr(out)), "dequant")
    return out


def gemv(t: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray):
    """x fp32 [M, cols] (or [cols]) -> (y fp64 [M, rows], S fp64 [M, rows])."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= rows * row_bytes(t, cols)
    x2 = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
    M = x2.shape[0]
    y = np.zeros((M, rows), np.float64)
    S = np.zeros((M, rows), np.float64)
    _check(lib().oq_gemv(t, _ptr(W), rows, cols, _ptr(x2), M, _ptr(y), _ptr(S)), "gemv")
    return y, S


def silu(z) -> np.ndarray:
    """SiLU(z) = z / (1 + e^-z) in fp64: the gate nonlinearity of the SwiGLU
    feed-forward ("How LLM Inference Engines Work", "SwiGLU Feed-Forward
    Network"; the page names SiLU without writing it out, this is its standard
    definition z * sigmoid(z)).  e^-z overflowing to inf gives -0."""
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(t: int, Wg: np.ndarray, Wu: np.ndarray, rows: int, cols: int, x: np.ndarray):
    """Decode SwiGLU gate (same page and section): h = SiLU(Wg x) * (Wu x)
    over the exactly dequantized weights, fp64.  x fp32 [cols].  Returns
    (h, g, u, Sg, Su), each fp64 [rows]; Sg, Su = sum_k |w x| of the two
    products (for the tolerance)."""
    g, Sg = gemv(t, Wg, rows, cols, x)
    u, Su = gemv(t, Wu, rows, cols, x)
    g, u, Sg, Su = g[0], u[0], Sg[0], Su[0]
    return silu(g) * u, g, u, Sg, Su


def gemm_bf16(t: int, W: np.ndarray, rows: int, cols: int, X_bits: np.ndarray):
    """X_bits uint16 bf16 bit patterns [M, cols] -> (Y fp64 [M, rows], S)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= rows * row_bytes(t, cols)
    X = np.ascontiguousarray(X_bits, dtype=np.uint16).reshape(-1, cols)
    M = X.shape[0]
    Y = np.zeros((M, rows), np.float64)
    S = np.zeros((M, rows), np.float64)
    _check(lib().oq_gemm_bf16(t, _ptr(W), rows, cols, _ptr(X), M, _ptr(Y), _ptr(S)), "gemm")
    return Y, S


def entries(t: int, W: np.ndarray, rows: int, cols: int, mi, ni, x=None, X_bits=None):
    """Selected outputs (mi[e], ni[e]) of the GEMV (x fp32 [M, cols]) or of the
    bf16 GEMM (X_bits uint16 [M, cols]).  Returns (y fp64 [count], S)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    assert mi.shape == ni.shape
    if X_bits is not None:
        xb = np.ascontiguousarray(X_bits, dtype=np.uint16).reshape(-1, cols)
        M, xf = xb.shape[0], None
    else:
        xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
        M, xb = xf.shape[0], None
    y = np.zeros(mi.size, np.float64)
    S = np.zeros(mi.size, np.float64)
    _check(lib().oq_entries(t, _ptr(W), rows, cols, _ptr(xf), _ptr(xb), M, _ptr(mi), _ptr(ni),
                            mi.size, _ptr(y), _ptr(S)), "entries")
    return y, S


def quantize(t: int, w: np.ndarray) -> np.ndarray:
    """fp32 [rows, cols] -> packed blocks (uint8), by the plain min/max scheme."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    out = np.zeros(rows * row_bytes(t, cols), np.uint8)
    _check(lib().oq_quantize(t, _ptr(w), rows, cols, _ptr(out)), "quantize")
    return out


def quantize_imatrix(t: int, w: np.ndarray, imp: np.ndarray) -> np.ndarray:
    """fp32 [rows, cols] and column importances fp32 [cols] (finite, >= 0)
    -> packed blocks minimising the importance-weighted error (see
    oq_quantize_imatrix)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    imp = np.ascontiguousarray(imp, dtype=np.float32).reshape(cols)
    out = np.zeros(rows * row_bytes(t, cols), np.uint8)
    _check(lib().oq_quantize_imatrix(t, _ptr(w), rows, cols, _ptr(imp), _ptr(out)), "quantize_imatrix")
    return out


def attn_decode(t: int, q: np.ndarray, K: np.ndarray, V: np.ndarray, T: int, n_heads: int, n_kv: int, d: int,
                scale: float):
    """Decode attention over a block-quantized KV cache (oq_attn_decode):
    q fp32 [n_heads, d]; K, V packed [T, n_kv, d] rows of 32-weight blocks.
    Returns (out fp64 [n_heads, d], Sv fp64 [n_heads, d])."""
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(n_heads, d)
    K = np.ascontiguousarray(K, dtype=np.uint8)
    V = np.ascontiguousarray(V, dtype=np.uint8)
    assert K.size >= T * n_kv * row_bytes(t, d) and V.size >= T * n_kv * row_bytes(t, d)
    out = np.zeros((n_heads, d), np.float64)
    Sv = np.zeros((n_heads, d), np.float64)
    _check(lib().oq_attn_decode(t, _ptr(q), _ptr(K), _ptr(V), T, n_heads, n_kv, d, scale, _ptr(out), _ptr(Sv)),
           "attn_decode")
    return out, Sv
