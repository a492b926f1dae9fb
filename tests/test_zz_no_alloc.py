"""qk_gemv_noalloc, the GEMV entry point for callers that cannot allocate
device memory (plug-ins inside a runtime that owns all allocations, code
under a fixed memory budget, paths that cannot take the synchronization an
allocation can cause).  It keeps its scratch in a fixed array inside the
library, so these tests call it through the C ABI and check that two calls
in a row match the oracle within the GEMV tolerance, including a problem
whose scratch fills the array almost to its end.  This file is collected
last on purpose."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu
SCRATCH = 8 << 20

# Decode and small batches (no scratch needed), a misaligned Q6_K case, and
# two batches beyond 64 activation rows that use the scratch: prepped
# activations, and for the 16-row one split-K partials and tile counters.
CASES = [("Q4_K", 4096, 4096, 1), ("Q6_K", 9, 11008, 2), ("Q5_0", 300, 1024, 5), ("Q8_0", 16, 8192, 72),
         ("Q4_K", 200, 2048, 70)]


def _near_full_case():
    """A batched problem whose scratch is the largest of a few candidates
    that still fit the array, with K split over CTAs (16 output rows)."""
    best = None
    for cols in (8192, 12288, 16384, 20480):
        for M in (72, 96, 112, 128, 160):
            ws = qk.gemv_workspace(qk.Q4_K, 16, cols, M)
            if ws <= SCRATCH and (best is None or ws > best[0]):
                best = (ws, cols, M)
    return best


def _check(lib, gpu, name, rows, cols, M, seed):
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, seed)
    x = synth.activations(M, cols, seed + 100)
    Wd, xd = dev_u8(W, gpu), dev_f32(x, gpu)
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    stream = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full((M, rows), float("nan"), device=gpu)
        st = lib.qk_gemv_noalloc(t, Wd.data_ptr(), rows, cols, xd.data_ptr(), M, y.data_ptr(), stream.cuda_stream)
        assert st == 0, lib.qk_last_error()
        stream.synchronize()
        assert_gemv_close(y.cpu().numpy(), y_ref, S, what=f"{name} {rows}x{cols} M={M} call {call}")
    qk.device_status()


@pytest.mark.parametrize("name,rows,cols,M", CASES)
def test_noalloc_matches_oracle(gpu, name, rows, cols, M):
    _check(qk.load(), gpu, name, rows, cols, M, 8800 + rows + M)


def test_noalloc_scratch_nearly_full(gpu):
    ws, cols, M = _near_full_case()
    assert ws > SCRATCH // 2, "the case should use most of the array"
    _check(qk.load(), gpu, "Q4_K", 16, cols, M, 8700)


def test_noalloc_rejects_problems_larger_than_its_scratch(gpu):
    lib = qk.load()
    t, rows, cols, M = qk.Q4_K, 16, 16384, 256      # prepped activations alone: 14.7 MB
    assert qk.gemv_workspace(t, rows, cols, M) > SCRATCH
    W = torch.zeros(rows * qk.row_bytes(t, cols), dtype=torch.uint8, device=gpu)
    x = torch.zeros((M, cols), device=gpu)
    y = torch.full((M, rows), 7.0, device=gpu)
    st = lib.qk_gemv_noalloc(t, W.data_ptr(), rows, cols, x.data_ptr(), M, y.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == 5 and b"static scratch" in lib.qk_last_error()
    torch.cuda.synchronize()
    assert (y == 7.0).all()


def test_noalloc_reports_argument_errors_before_scratch_size(gpu):
    # An oversized problem with a NULL W: the NULL is reported (as qk_gemv would).
    lib = qk.load()
    t, rows, cols, M = qk.Q4_K, 16, 16384, 256
    x = torch.zeros((M, cols), device=gpu)
    y = torch.zeros((M, rows), device=gpu)
    st = lib.qk_gemv_noalloc(t, None, rows, cols, x.data_ptr(), M, y.data_ptr(), None)
    assert st == 4, lib.qk_last_error()
