"""The C-ABI boundary without a GPU: the library loads, exports every entry
point include/qk.h declares, reports sizes, and rejects bad arguments on the
host before any CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import gguf_quant_dequant_gb300 as qk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def _declared():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(qk_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from gguf_quant_dequant_gb300 import build
    build.build()
    return qk.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"qk_dequant", "qk_gemv", "qk_gemm"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(qk.SIGNATURES) == names


def test_sizes(lib):
    assert [qk.block_bytes(t) for t in (1, 2, 3, 4, 5)] == [144, 210, 34, 22, 18]
    assert [qk.block_elems(t) for t in (1, 2, 3, 4, 5)] == [256, 256, 32, 32, 32]
    assert qk.block_bytes(9) == 0 and qk.block_elems(0) == 0
    assert qk.row_bytes(qk.Q6_K, 11008) == 9030
    assert qk.row_bytes(qk.Q4_K, 4096) == 2304
    assert qk.row_bytes(qk.Q4_K, 100) == 0
    assert lib.qk_version() == 1


def _status(fn, *args):
    return fn(*args)


def test_argument_errors_are_caught_on_host(lib):
    fake = ctypes.c_void_p(0x10000)          # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x10008)           # 8-byte aligned only
    # bad type
    assert lib.qk_gemv(99, fake, 4, 256, fake, 1, fake, None, 0, None) == 1
    assert b"type" in lib.qk_last_error()
    # cols not a multiple of the block
    assert lib.qk_gemv(qk.Q4_K, fake, 4, 100, fake, 1, fake, None, 0, None) == 2
    assert lib.qk_dequant(qk.Q8_0, fake, 4, 40, fake, 0, None) == 2
    # negative sizes
    assert lib.qk_gemv(qk.Q4_K, fake, -1, 256, fake, 1, fake, None, 0, None) == 2
    assert lib.qk_gemv(qk.Q4_K, fake, 4, 256, fake, -2, fake, None, 0, None) == 2
    # NULL weights / outputs / activations
    assert lib.qk_gemv(qk.Q4_K, None, 4, 256, fake, 1, fake, None, 0, None) == 4
    assert lib.qk_gemv(qk.Q4_K, fake, 4, 256, fake, 1, None, None, 0, None) == 4
    assert lib.qk_gemv(qk.Q4_K, fake, 4, 256, None, 1, fake, None, 0, None) == 4
    assert lib.qk_dequant(qk.Q4_K, fake, 4, 256, None, 0, None) == 4
    # misaligned pointers
    assert lib.qk_gemv(qk.Q4_K, odd, 4, 256, fake, 1, fake, None, 0, None) == 3
    assert lib.qk_gemv(qk.Q4_K, fake, 4, 256, odd, 1, fake, None, 0, None) == 3
    assert lib.qk_dequant(qk.Q4_K, fake, 4, 256, odd, 0, None) == 3
    # bad output dtype
    assert lib.qk_dequant(qk.Q4_K, fake, 4, 256, fake, 5, None) == 8
    # unpack
    assert lib.qk_unpack(0, fake, 1, None, None, None, None, None, None) == 1
    assert lib.qk_unpack(qk.Q4_K, odd, 1, None, None, None, None, None, None) == 3
    assert lib.qk_unpack(qk.Q4_K, fake, -1, None, None, None, None, None, None) == 2


def test_batch_argument_errors_are_caught_on_host(lib):
    fake, odd = 0x10000, 0x10008
    P = ctypes.c_void_p

    def call(t, n, Ws, rows, cols, x, ys):
        Wa = (P * max(len(Ws), 1))(*Ws)
        ra = (ctypes.c_int64 * max(len(rows), 1))(*rows)
        ya = (P * max(len(ys), 1))(*ys)
        return lib.qk_gemv_batch(t, n, Wa, ra, cols, x, ya, None)

    assert call(9, 1, [fake], [4], 256, fake, [fake]) == 1
    assert call(qk.Q4_K, 0, [fake], [4], 256, fake, [fake]) == 8
    assert call(qk.Q4_K, 9, [fake] * 9, [4] * 9, 256, fake, [fake] * 9) == 8
    assert b"n_mat" in lib.qk_last_error()
    assert call(qk.Q4_K, 2, [fake, odd], [4, 4], 256, fake, [fake, fake]) == 3
    assert call(qk.Q4_K, 2, [fake, fake], [4, 4], 256, fake, [fake, None]) == 4
    assert call(qk.Q4_K, 2, [fake, fake], [4, 4], 100, fake, [fake, fake]) == 2
    assert call(qk.Q4_K, 2, [fake, fake], [4, -1], 256, fake, [fake, fake]) == 2
    assert call(qk.Q4_K, 1, [fake], [4], 256, None, [fake]) == 4
    assert call(qk.Q4_K, 1, [fake], [4], 256, odd, [fake]) == 3
    assert lib.qk_gemv_batch(qk.Q4_K, 1, None, None, 256, fake, None, None) == 4
    # all-empty batches queue nothing
    assert call(qk.Q4_K, 2, [None, None], [0, 0], 256, None, [None, None]) == 0


def test_quantize_argument_errors_are_caught_on_host(lib):
    fake = ctypes.c_void_p(0x10000)          # 16-byte aligned, never dereferenced
    odd4 = ctypes.c_void_p(0x10004)          # 4-byte aligned only
    odd2 = ctypes.c_void_p(0x10002)          # 2-byte aligned only
    assert lib.qk_quantize(0, fake, 4, 256, fake, None) == 1
    assert lib.qk_quantize(qk.Q4_K, fake, 4, 100, fake, None) == 2
    assert lib.qk_quantize(qk.Q8_0, fake, -1, 32, fake, None) == 2
    assert lib.qk_quantize(qk.Q8_0, fake, 1 << 40, 1 << 10, fake, None) == 2   # 2^50 weights
    assert b"too large" in lib.qk_last_error()
    assert lib.qk_quantize(qk.Q4_K, None, 4, 256, fake, None) == 4
    assert lib.qk_quantize(qk.Q4_K, fake, 4, 256, None, None) == 4
    assert lib.qk_quantize(qk.Q4_K, odd4, 4, 256, fake, None) == 3     # w needs 16 bytes
    assert lib.qk_quantize(qk.Q4_K, fake, 4, 256, odd2, None) == 3     # out needs 4 bytes
    assert lib.qk_quantize(qk.Q5_0, fake, 0, 64, fake, None) == 0       # nothing to do
    assert lib.qk_quantize(qk.Q5_0, fake, 3, 0, fake, None) == 0


def test_swiglu_argument_errors_are_caught_on_host(lib):
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    odd2 = ctypes.c_void_p(0x10002)
    assert lib.qk_gemv_swiglu(9, fake, fake, 4, 256, fake, fake, None) == 1
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 4, 100, fake, fake, None) == 2
    assert lib.qk_gemv_swiglu(qk.Q4_K, None, fake, 4, 256, fake, fake, None) == 4
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, None, 4, 256, fake, fake, None) == 4
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, odd, 4, 256, fake, fake, None) == 3
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 4, 256, fake, None, None) == 4
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 4, 256, fake, odd2, None) == 3
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 4, 256, None, fake, None) == 4
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 4, 256, odd, fake, None) == 3
    assert lib.qk_gemv_swiglu(qk.Q4_K, fake, fake, 0, 256, fake, fake, None) == 0


def test_gemm_row_tile_limit_is_checked_on_host(lib):
    fake = ctypes.c_void_p(0x10000)
    assert lib.qk_gemm(qk.Q4_K, fake, 65535 * 128 + 1, 256, fake, 4, fake, None, 0, None) == 2
    assert b"65535" in lib.qk_last_error()


def test_empty_problems_queue_nothing(lib):
    fake = ctypes.c_void_p(0x10000)
    # rows == 0 or M == 0: success without touching the device.
    assert lib.qk_gemv(qk.Q4_K, fake, 0, 256, fake, 1, fake, None, 0, None) == 0
    assert lib.qk_gemv(qk.Q4_K, fake, 8, 256, fake, 0, fake, None, 0, None) == 0
    assert lib.qk_dequant(qk.Q6_K, fake, 0, 256, fake, 0, None) == 0
    assert lib.qk_unpack(qk.Q8_0, fake, 0, None, None, None, None, None, None) == 0


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.reload(qk)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError):
        mod.load()
    importlib.reload(qk)


def test_new_block_type_sizes(lib):
    assert [qk.block_bytes(t) for t in (6, 7, 8)] == [176, 84, 110]
    assert [qk.block_elems(t) for t in (6, 7, 8)] == [256, 256, 256]
    assert qk.row_bytes(qk.Q5_K, 4096) == 2816 and qk.row_bytes(qk.Q2_K, 4096) == 1344
    assert qk.row_bytes(qk.Q3_K, 4096) == 1760


def test_imatrix_and_attention_argument_errors_are_caught_on_host(lib):
    fake = ctypes.c_void_p(0x10000)
    odd1 = ctypes.c_void_p(0x10001)
    odd2 = ctypes.c_void_p(0x10002)
    f = ctypes.c_float
    assert lib.qk_quantize_imatrix(0, fake, 4, 256, fake, fake, None) == 1
    assert lib.qk_quantize_imatrix(qk.Q4_K, fake, 4, 100, fake, fake, None) == 2
    assert lib.qk_quantize_imatrix(qk.Q4_K, fake, 4, 256, None, fake, None) == 4
    assert lib.qk_quantize_imatrix(qk.Q4_K, odd2, 4, 256, fake, fake, None) == 3
    assert lib.qk_quantize_imatrix(qk.Q4_K, fake, 0, 256, None, None, None) == 0
    ws = qk.attn_decode_workspace(qk.Q8_0, 300, 32, 8, 128)
    assert ws == 3 * 32 * 130 * 4   # chunks of 128 (the smallest chunk) x heads x (d + 2) floats
    assert qk.attn_decode_workspace(qk.Q4_K, 300, 32, 8, 128) == 0
    call = lib.qk_attn_decode
    assert call(qk.Q4_K, fake, fake, fake, 300, 32, 8, 128, f(0.1), fake, fake, ws, None) == 1
    assert call(qk.Q8_0, fake, fake, fake, 300, 32, 8, 96, f(0.1), fake, fake, ws, None) == 2     # d
    assert call(qk.Q8_0, fake, fake, fake, 300, 30, 8, 128, f(0.1), fake, fake, ws, None) == 2    # groups
    assert call(qk.Q8_0, fake, fake, fake, 300, 32, 2, 128, f(0.1), fake, fake, ws, None) == 2    # 16 per kv
    assert call(qk.Q8_0, fake, fake, fake, 0, 32, 8, 128, f(0.1), fake, fake, ws, None) == 2      # T
    big = qk.attn_decode_workspace(qk.Q8_0, 65535 * 256 + 1, 32, 8, 128)
    assert call(qk.Q8_0, fake, fake, fake, 65535 * 256 + 1, 32, 8, 128, f(0.1), fake, fake, big, None) == 2
    assert call(qk.Q8_0, None, fake, fake, 300, 32, 8, 128, f(0.1), fake, fake, ws, None) == 4
    assert call(qk.Q8_0, fake, odd1, fake, 300, 32, 8, 128, f(0.1), fake, fake, ws, None) == 3
    assert call(qk.Q8_0, fake, fake, odd2, 300, 32, 8, 128, f(0.1), fake, fake, ws, None) == 3
    assert call(qk.Q8_0, fake, fake, fake, 300, 32, 8, 128, f(0.1), fake, fake, ws - 4, None) == 5
