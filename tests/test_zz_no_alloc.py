"""qk_gemv_noalloc, the GEMV entry point for callers that cannot allocate
device memory (plug-ins inside a runtime that owns all allocations, code
under a fixed memory budget, paths that cannot take the synchronization an
allocation can cause).  The GEMV needs no workspace for any shape, so the
entry point holds no scratch of its own; these tests call it through the C
ABI and check that two calls in a row match the oracle within the GEMV
tolerance, for decode, small and large activation batches and a problem
that a workspace-taking design would have had to reject.  This file is
collected last on purpose."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

# Decode, small batches, a misaligned Q6_K case and batches beyond 64
# activation rows (one launch per pair of rows).
CASES = [("Q4_K", 4096, 4096, 1), ("Q6_K", 9, 11008, 2), ("Q5_0", 300, 1024, 5), ("Q8_0", 16, 8192, 72),
         ("Q4_K", 200, 2048, 70)]


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


def test_noalloc_large_batch_needs_no_scratch(gpu):
    # 256 activation rows of a 16384-column matrix: 14.7 MB of prepared
    # activations in a design that keeps them in a workspace; here none.
    t, rows, cols, M = qk.Q4_K, 16, 16384, 256
    assert qk.gemv_workspace(t, rows, cols, M) == 0
    _check(qk.load(), gpu, "Q4_K", rows, cols, M, 8700)


def test_noalloc_reports_argument_errors(gpu):
    # A NULL W is reported as qk_gemv would report it, and nothing is queued.
    lib = qk.load()
    t, rows, cols, M = qk.Q4_K, 16, 16384, 256
    x = torch.zeros((M, cols), device=gpu)
    y = torch.full((M, rows), 7.0, device=gpu)
    st = lib.qk_gemv_noalloc(t, None, rows, cols, x.data_ptr(), M, y.data_ptr(), None)
    assert st == 4, lib.qk_last_error()
    torch.cuda.synchronize()
    assert (y == 7.0).all()
