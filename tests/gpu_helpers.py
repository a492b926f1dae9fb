"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
call the library through its binding, compare with the oracle under the
stated tolerances."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import synth

GEMV_RTOL, GEMV_ATOL = 1e-4, 1e-6     # |y - y_ref| <= 1e-4 * sum|w x| + 1e-6
GEMM_RTOL = 5e-3                      # |Y - Y_ref| <= 5e-3 * sum|w x| (bf16 x)


@pytest.fixture(scope="session")
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from gguf_quant_dequant_gb300 import build
    build.build()
    qk.load()
    return torch.device("cuda:0")


def dev_u8(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device)


def dev_f32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def assert_gemv_close(y: np.ndarray, y_ref: np.ndarray, S: np.ndarray, rtol=GEMV_RTOL, atol=GEMV_ATOL, what=""):
    err = np.abs(y.astype(np.float64) - y_ref)
    bound = rtol * S + atol
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs out of tolerance; "
                           f"worst err/bound {np.max(err / bound):.3g}")
    return float(np.max(err / bound)) if err.size else 0.0


def type_id(name: str) -> int:
    return synth.TYPE_IDS[name]
