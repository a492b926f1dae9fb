"""Failure detection without a GPU fault: a bounded wait that nothing
releases runs out, the kernel records the timeout and returns, the host
reads QK_ERR_TIMEOUT from the device status word, and the context keeps
working (a GEMV right after it is exact to tolerance)."""
import time

import numpy as np
import pytest

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu  # noqa: F401

pytestmark = pytest.mark.gpu


def test_stalled_wait_times_out_and_context_survives(gpu):
    qk.device_status()                       # start clean
    t0 = time.perf_counter()
    qk.test_stalled_wait(20000)              # 20 ms limit
    with pytest.raises(qk.QKError) as e:
        qk.device_status()
    dt = time.perf_counter() - t0
    assert e.value.status == 7
    assert dt < 5.0                          # bounded: returned long before any watchdog
    qk.device_status()                       # the word was cleared
    rows, cols = 64, 2048
    W = synth.random_blocks("Q4_K", rows, cols, 9911)
    x = synth.activations(1, cols, 9912)
    y = qk.gemv(qk.Q4_K, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(qk.Q4_K, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what="after a timeout")
    qk.device_status()


def test_stalled_wait_argument_check(gpu):
    with pytest.raises(qk.QKError) as e:
        qk.test_stalled_wait(0)
    assert e.value.status == 8
