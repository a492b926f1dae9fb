"""qk_gemv against the oracle on small seeded problems that span several
stages, ragged row tiles and tails, every activation-batch width, split and
unsplit K, misaligned Q6_K rows; plus invariants and edge cases."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu
NAMES = ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"]


def run(gpu, name, rows, cols, M, seed, W=None, x=None):
    t = type_id(name)
    if W is None:
        W = synth.random_blocks(name, rows, cols, seed)
    if x is None:
        x = synth.activations(M, cols, seed + 1)
    y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    return y, y_ref, S


# Shapes: one block; one stage plus a one-block tail; many rows with a ragged
# last CTA (rows % 16 != 0) and several stages; a 11008-wide Q6_K case whose
# rows start 6 bytes off 16-byte alignment and whose total size is not a
# multiple of 16 (the last bytes are not bulk-copyable).
SHAPES = {
    "Q4_K": [(1, 256), (5, 1280), (37, 3328), (300, 1024)],
    "Q6_K": [(1, 256), (5, 1280), (37, 3328), (9, 11008)],
    "Q8_0": [(1, 32), (5, 1056), (37, 3104), (300, 1024)],
    "Q5_0": [(1, 32), (5, 1056), (37, 3104), (300, 1024)],
    "Q4_0": [(1, 32), (5, 1056), (37, 3104), (300, 1024)],
    "Q5_K": [(1, 256), (5, 1280), (37, 3328), (300, 1024)],
    "Q2_K": [(1, 256), (5, 1280), (37, 3328), (300, 1024)],
    "Q3_K": [(1, 256), (5, 1280), (37, 3328), (300, 1024)],
}


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("shape_i", range(4))
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 9, 67])
def test_gemv_parity(gpu, name, shape_i, M):
    rows, cols = SHAPES[name][shape_i]
    y, y_ref, S = run(gpu, name, rows, cols, M, 1000 + 10 * shape_i + M)
    assert y.shape == (M, rows)
    assert_gemv_close(y, y_ref, S, what=f"{name} {rows}x{cols} M={M}")


@pytest.mark.parametrize("name", NAMES)
def test_gemv_quantized_codes(gpu, name):
    # Codes from the plain quantizer applied to N(0, 0.02) weights.
    rows, cols = 64, 2048
    W = oracle.quantize(type_id(name), synth.normal_weights(rows, cols, 77))
    y, y_ref, S = run(gpu, name, rows, cols, 2, 78, W=W)
    assert_gemv_close(y, y_ref, S, what=name)


def test_gemv_needs_no_workspace_for_any_batch(gpu):
    # Every batch size runs the tensor-core kernel (one launch per one or two
    # activation rows), which prepares x in shared memory: no workspace.
    for M in (1, 2, 3, 64, 72, 200):
        assert qk.gemv_workspace(qk.Q4_K, 16, 8192, M) == 0
        assert qk.gemv_workspace(qk.Q6_K, 8192, 8192, M) == 0
    for rows in (16, 1024):
        for M in (1, 2, 3, 72):
            y, y_ref, S = run(gpu, "Q4_K", rows, 8192, M, 2000 + rows)
            assert_gemv_close(y, y_ref, S, what=f"rows={rows} M={M}")


def test_exact_integer_case_is_near_exact(gpu):
    # Q8_0 with d = 2^-3 and integer x in [-8, 8]: the exact result is an
    # integer multiple of 2^-3.  Codes and such x are exact in fp16 and every
    # partial sum is an integer the fp32 accumulators hold exactly, so only
    # the scale steps can round: far inside the 1e-4 bound.
    g = synth.rng(90)
    rows, cols = 48, 4096
    codes = g.integers(-128, 128, (rows * cols // 32, 32)).astype(np.int16)
    W = oracle.pack(qk.Q8_0, codes, None, None, np.full(rows * cols // 32, 0x3000, np.uint16))
    x = g.integers(-8, 9, (3, cols)).astype(np.float32)
    y, y_ref, S = run(gpu, "Q8_0", rows, cols, 3, 0, W=W, x=x)
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -20 * S)
    assert np.array_equal(y_ref, np.round(y_ref * 8) / 8)


def test_linearity_and_batch_rows(gpu):
    name, rows, cols = "Q6_K", 40, 2048
    t = type_id(name)
    W = dev_u8(synth.random_blocks(name, rows, cols, 91), gpu)
    x = synth.activations(4, cols, 92)
    Y = qk.gemv(t, W, rows, cols, dev_f32(x, gpu)).cpu().numpy()
    _, S4 = oracle.gemv(t, W.cpu().numpy(), rows, cols, x)
    for m in range(4):
        # A single row may run on another kernel than the batch (decode
        # kernel vs tiled kernel): each result is within its own bound of the
        # exact product, so the two differ by at most the sum of the bounds.
        y1 = qk.gemv(t, W, rows, cols, dev_f32(x[m:m + 1], gpu)).cpu().numpy()[0]
        assert np.all(np.abs(Y[m] - y1) <= 2e-4 * S4[m] + 2e-6)
    # Linearity, within the sum of the three results' error bounds.
    a, b = 0.5, -2.0
    yc = qk.gemv(t, W, rows, cols, dev_f32(a * x[0:1] + b * x[1:2], gpu)).cpu().numpy()[0]
    _, S = oracle.gemv(t, W.cpu().numpy(), rows, cols, x[:2])
    bound = 2e-4 * (abs(a) * S[0] + abs(b) * S[1]) + 3e-6
    assert np.all(np.abs(yc - (a * Y[0] + b * Y[1])) <= bound)


def test_deterministic(gpu):
    name, rows, cols = "Q4_K", 64, 8192   # split-K path included
    t = type_id(name)
    W = dev_u8(synth.random_blocks(name, rows, cols, 93), gpu)
    x = dev_f32(synth.activations(1, cols, 94), gpu)
    y0 = qk.gemv(t, W, rows, cols, x).cpu().numpy()
    for _ in range(3):
        assert np.array_equal(qk.gemv(t, W, rows, cols, x).cpu().numpy(), y0)


def test_output_canaries_and_empty(gpu):
    name, rows, cols, M = "Q5_0", 21, 1024, 2
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, 95)
    x = synth.activations(M, cols, 96)
    buf = torch.full((M * rows + 8,), float("nan"), device=gpu)
    y = buf[4:4 + M * rows].view(M, rows)
    qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu), y=y)
    b = buf.cpu().numpy()
    assert np.isnan(b[:4]).all() and np.isnan(b[-4:]).all() and not np.isnan(b[4:-4]).any()
    # cols == 0 zero-fills, rows == 0 and M == 0 are no-ops
    y0 = torch.full((2, 3), 7.0, device=gpu)
    qk.gemv(t, torch.zeros(16, dtype=torch.uint8, device=gpu), 3, 0,
            torch.zeros((2, 0), device=gpu), y=y0)
    assert (y0 == 0).all()
    qk.gemv(t, dev_u8(W, gpu), 0, cols, dev_f32(x, gpu), y=torch.empty((2, 0), device=gpu))
    qk.device_status()


def test_workspace_argument_is_not_needed(gpu):
    # No shape needs a workspace: a NULL or a 16-byte one are both fine.
    t, rows, cols, M = qk.Q4_K, 16, 4096, 72
    W = synth.random_blocks("Q4_K", rows, cols, 97)
    x = synth.activations(M, cols, 98)
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    Wd, xd = dev_u8(W, gpu), dev_f32(x, gpu)
    tiny = torch.empty(16, dtype=torch.uint8, device=gpu)
    for ws in (None, tiny):
        y = qk.gemv(t, Wd, rows, cols, xd, ws=ws).cpu().numpy()
        assert_gemv_close(y, y_ref, S, what=f"ws={'NULL' if ws is None else '16 B'}")


@pytest.mark.parametrize("name,rows,cols", [("Q6_K", 24, 20480), ("Q4_K", 40, 65536), ("Q8_0", 17, 40960)])
def test_decode_needs_no_workspace_at_any_k(gpu, name, rows, cols):
    # M = 1 prepares x inside the decode kernel, one 256-element unit per
    # warp and chunk, so its shared memory does not grow with K: no
    # workspace, whatever the row length.
    t = type_id(name)
    assert qk.gemv_workspace(t, 4096, 4096, 1) == 0
    assert qk.gemv_workspace(t, rows, cols, 1) == 0
    W = synth.random_blocks(name, rows, cols, 4321 + rows)
    x = synth.activations(1, cols, 4322 + rows)
    y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what=f"{name} K={cols}")


@pytest.mark.parametrize("name,rows,cols", [("Q6_K", 9, 11008), ("Q4_K", 151, 4096), ("Q4_K", 153, 2304),
                                            ("Q5_K", 151, 4096), ("Q5_K", 1000, 11008),
                                            ("Q2_K", 151, 4096), ("Q3_K", 1000, 11008),
                                            ("Q8_0", 1000, 4128), ("Q5_0", 3, 96)])
def test_decode_row_splits(gpu, name, rows, cols):
    # Fewer rows than SMs, one row more than the SMs on some CTAs, a K whose
    # last 2048-slice is short, and a K that is a single 32-block short of
    # full slices.
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, 4400 + rows)
    x = synth.activations(1, cols, 4500 + rows)
    y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what=f"{name} {rows}x{cols}")


@pytest.mark.parametrize("name,rows_list,cols", [
    ("Q4_K", [512, 128, 128], 4096),                       # q / k / v (grouped-query shapes)
    ("Q4_K", [700, 700], 2048),                            # gate / up
    ("Q6_K", [300, 0, 45], 11008),                         # an empty member
    ("Q8_0", [1, 2, 3, 5, 8, 13, 21, 34], 1024),           # the most members, tiny ones
    ("Q5_0", [333, 77], 1056),
])
def test_gemv_batch_matches_oracle(gpu, name, rows_list, cols):
    # One launch over matrices that share x gives each matrix's GEMV.
    t = type_id(name)
    x = synth.activations(1, cols, 4600 + cols)
    xd = dev_f32(x, gpu)
    Ws = [synth.random_blocks(name, r, cols, 4700 + 31 * i + r) if r else np.zeros(0, np.uint8)
          for i, r in enumerate(rows_list)]
    Wd = [dev_u8(W, gpu) if W.size else torch.zeros(16, dtype=torch.uint8, device=gpu) for W in Ws]
    ys = qk.gemv_batch(t, Wd, rows_list, cols, xd[0])
    qk.device_status()
    for i, (W, r) in enumerate(zip(Ws, rows_list)):
        if r == 0:
            continue
        y_ref, S = oracle.gemv(t, W, r, cols, x)
        assert_gemv_close(ys[i].cpu().numpy()[None, :], y_ref, S, what=f"{name} member {i}")
        # and the same as the single-matrix entry point, to the tolerance
        y1 = qk.gemv(t, Wd[i], r, cols, xd).cpu().numpy()
        assert_gemv_close(ys[i].cpu().numpy()[None, :], y1.astype(np.float64), S, what=f"{name} member {i} vs qk_gemv")


def test_gemv_batch_at_large_k(gpu):
    # K = 20480 (Q6_K): the batched kernel prepares x per unit, so long rows fit.
    t, cols = qk.Q6_K, 20480
    rows = [8, 24]
    x = synth.activations(1, cols, 4700)
    Ws = [synth.random_blocks("Q6_K", r, cols, 4701 + i) for i, r in enumerate(rows)]
    ys = qk.gemv_batch(t, [dev_u8(W, gpu) for W in Ws], rows, cols, dev_f32(x[0], gpu))
    for W, r, y in zip(Ws, rows, ys):
        y_ref, S = oracle.gemv(t, W, r, cols, x)
        assert_gemv_close(y.cpu().numpy()[None, :], y_ref, S, what=f"Q6_K batch {r}x{cols}")


