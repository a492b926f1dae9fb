"""qk_gemv_noalloc, the GEMV entry point for callers that cannot allocate
device memory (plug-ins inside a runtime that owns all allocations, code
under a fixed memory budget, paths that cannot take the synchronization an
allocation can cause).  It keeps its scratch in a fixed array inside the
library, so these tests call it through the C ABI and check that two calls
in a row give what the workspace entry point gives, within the GEMV
tolerance.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

# One unsplit decode GEMV, one split-K case with non-16-byte-aligned Q6_K rows
# (partials and tile counters in the scratch), a batched case and a Q8_0 one.
CASES = [("Q4_K", 4096, 4096, 1), ("Q6_K", 9, 11008, 2), ("Q5_0", 300, 1024, 5), ("Q8_0", 16, 8192, 1)]


@pytest.mark.parametrize("name,rows,cols,M", CASES)
def test_noalloc_matches_workspace_entry_point(gpu, name, rows, cols, M):
    lib = qk.load()
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, 8800 + rows)
    x = synth.activations(M, cols, 8900 + rows)
    Wd, xd = dev_u8(W, gpu), dev_f32(x, gpu)
    y_ws = qk.gemv(t, Wd, rows, cols, xd).cpu().numpy()
    _, S = oracle.gemv(t, W, rows, cols, x)
    stream = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full((M, rows), float("nan"), device=gpu)
        st = lib.qk_gemv_noalloc(t, Wd.data_ptr(), rows, cols, xd.data_ptr(), M, y.data_ptr(), stream.cuda_stream)
        assert st == 0, lib.qk_last_error()
        stream.synchronize()
        assert_gemv_close(y.cpu().numpy(), y_ws, S, what=f"{name} call {call}")
    qk.device_status()


def test_noalloc_rejects_problems_larger_than_its_scratch(gpu):
    lib = qk.load()
    t, rows, cols, M = qk.Q4_K, 16, 16384, 256      # prepped activations alone: 14.7 MB
    assert qk.gemv_workspace(t, rows, cols, M) > qk.load().qk_gemv_workspace(t, 16, 256, 1)
    W = torch.zeros(rows * qk.row_bytes(t, cols), dtype=torch.uint8, device=gpu)
    x = torch.zeros((M, cols), device=gpu)
    y = torch.full((M, rows), 7.0, device=gpu)
    st = lib.qk_gemv_noalloc(t, W.data_ptr(), rows, cols, x.data_ptr(), M, y.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == 5 and b"static scratch" in lib.qk_last_error()
    torch.cuda.synchronize()
    assert (y == 7.0).all()
