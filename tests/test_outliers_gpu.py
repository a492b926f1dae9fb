"""Parity with massive activations: in every 32-element block of x (and of
the attention query) one coordinate is 1e3, 1e4 or 1e5 times the typical
magnitude, as the hidden states of large language models have.  Some rows
carry an exactly zero weight at each outlier column (a Q8_0 code 0, a Q6_K
code 32, a Q4_K sub-block with d*sc*q == dmin*m, ...), others a tiny
non-zero one, so that sum|w x| of those rows holds no outlier term and the
bound 1e-4 * sum|w x| + 1e-6 tests the rounding of everything else.

The matrices are built by unpacking seeded random blocks with the oracle,
setting the fields at the outlier columns, and packing them back; a
precondition checks that the oracle's weights there are exactly zero."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu
NAMES = ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"]
RATIOS = [1e3, 1e4, 1e5]
# The code whose weight is zero whatever the scale (types with a code offset).
ZERO_CODE = {"Q8_0": 0, "Q6_K": 32, "Q5_0": 16, "Q4_0": 8, "Q3_K": 0}


def _half_bits(W, name, nb, off):
    bb = synth.GEOMETRY[name][0]
    return W.reshape(nb, bb)[:, off:off + 2].copy().view(np.uint16).reshape(nb)


def zero_weights_at(name, W, rows, cols, pos, block=32):
    """W with, for rows r % 4 == 0, a zero weight at every column
    32 b + pos[b] (pos: outlier position per 32-block of x), and for rows
    r % 4 == 1 a tiny non-zero one; other rows unchanged."""
    t = type_id(name)
    bb, be, d_off, dmin_off = synth.GEOMETRY[name]
    nbr = cols // be
    nb = rows * nbr
    codes, sc, mins, _, _ = oracle.unpack(t, W, nb)
    d_bits = _half_bits(W, name, nb, d_off)
    dmin_bits = _half_bits(W, name, nb, dmin_off) if dmin_off is not None else None
    for r in range(rows):
        kind = r % 4
        if kind > 1:
            continue
        tiny = kind == 1
        for b, p in enumerate(pos):
            c = block * b + int(p)
            bi, e = r * nbr + c // be, c % be
            if name in ZERO_CODE:
                codes[bi, e] = ZERO_CODE[name] + (1 if tiny else 0)
                if tiny and name in ("Q6_K", "Q3_K") and sc[bi, e // 16] == 0:
                    sc[bi, e // 16] = 1   # a zero group scale would zero the tiny weight too
                if tiny and (d_bits[bi] & 0x7FFF) == 0:
                    d_bits[bi] = 0x1400   # so would a zero d (fp16 underflow of the draw)
            elif name in ("Q4_K", "Q5_K"):
                j = e // 32
                dmin_bits[bi] = d_bits[bi] + (1 if tiny else 0)   # tiny: dmin one fp16 step above d
                sc[bi, j], mins[bi, j], codes[bi, e] = 3, 15, 5    # d*3*5 == dmin*15
            elif name == "Q2_K":
                g = e // 16
                dmin_bits[bi] = d_bits[bi] + (1 if tiny else 0)
                sc[bi, g], mins[bi, g], codes[bi, e] = 2, 6, 3     # d*2*3 == dmin*6
    W2 = oracle.pack(t, codes, sc, mins, d_bits, dmin_bits)
    w = oracle.dequant(t, W2, rows, cols)
    zcols = block * np.arange(len(pos)) + pos
    assert (w[0::4][:, zcols] == 0).all(), "construction: weights at the outlier columns must be zero"
    assert (w[1::4][:, zcols] != 0).all(), "construction: tiny weights must be non-zero"
    return W2


def outlier_problem(name, rows, cols, ratio, seed, M=1):
    x, pos = synth.activations_outliers(M, cols, seed, ratio)
    W = synth.random_blocks(name, rows, cols, seed + 1)
    # One set of outlier columns for the matrix: those of the first row of x
    # (every row of x has its outliers there too, so that M > 1 is covered).
    for m in range(1, M):
        x[m] = synth.activations(1, cols, seed + 10 + m)[0]
        x[m, 32 * np.arange(cols // 32) + pos[0]] = x[0, 32 * np.arange(cols // 32) + pos[0]] * (m + 1) / M
    return zero_weights_at(name, W, rows, cols, pos[0]), x


SHAPES = {  # (rows, cols): one block of the type, several blocks, a Llama-sized matrix
    "Q4_K": [(64, 256), (48, 1024), (4096, 4096)],
    "Q6_K": [(64, 256), (48, 1024), (4096, 11008)],
    "Q8_0": [(64, 32), (48, 1024), (4096, 4096)],
    "Q5_0": [(64, 32), (48, 1024), (4096, 4096)],
    "Q4_0": [(64, 32), (48, 1024)],
    "Q5_K": [(64, 256), (48, 1024)],
    "Q2_K": [(64, 256), (48, 1024)],
    "Q3_K": [(64, 256), (48, 1024)],
}
CASES = [(n, i) for n in NAMES for i in range(len(SHAPES[n]))]


@pytest.mark.parametrize("name,shape_i", CASES)
@pytest.mark.parametrize("ratio", RATIOS)
def test_gemv_outliers_decode(gpu, name, shape_i, ratio):
    rows, cols = SHAPES[name][shape_i]
    t = type_id(name)
    W, x = outlier_problem(name, rows, cols, ratio, 3100 + 7 * shape_i + int(np.log10(ratio)))
    y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what=f"{name} {rows}x{cols} outliers x{ratio:g}")


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("M", [2, 3, 8, 72])
@pytest.mark.parametrize("ratio", [1e4, 1e5])
def test_gemv_outliers_batched_tokens(gpu, name, M, ratio):
    rows, cols = SHAPES[name][1]
    t = type_id(name)
    W, x = outlier_problem(name, rows, cols, ratio, 3300 + M, M=M)
    y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(t, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what=f"{name} M={M} outliers x{ratio:g}")


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0"])
@pytest.mark.parametrize("ratio", RATIOS)
def test_gemv_batch_outliers(gpu, name, ratio):
    # Three matrices reading one x (a q/k/v-like group).
    t = type_id(name)
    cols = 1024
    x, pos = synth.activations_outliers(1, cols, 3500, ratio)
    rows = [64, 32, 48]
    Ws = [zero_weights_at(name, synth.random_blocks(name, r, cols, 3510 + i), r, cols, pos[0])
          for i, r in enumerate(rows)]
    ys = qk.gemv_batch(t, [dev_u8(W, gpu) for W in Ws], rows, cols, dev_f32(x[0], gpu))
    for W, r, y in zip(Ws, rows, ys):
        y_ref, S = oracle.gemv(t, W, r, cols, x)
        assert_gemv_close(y.cpu().numpy()[None, :], y_ref, S, what=f"{name} batch outliers x{ratio:g}")


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("ratio", RATIOS)
def test_swiglu_outliers(gpu, name, ratio):
    t = type_id(name)
    rows, cols = 64, 1024
    x, pos = synth.activations_outliers(1, cols, 3700, ratio)
    Wg = zero_weights_at(name, synth.random_blocks(name, rows, cols, 3701), rows, cols, pos[0])
    Wu = zero_weights_at(name, synth.random_blocks(name, rows, cols, 3702), rows, cols, pos[0])
    h = qk.gemv_swiglu(t, dev_u8(Wg, gpu), dev_u8(Wu, gpu), rows, cols, dev_f32(x[0], gpu)).cpu().numpy()
    h_ref, g, u, Sg, Su = oracle.swiglu(t, Wg, Wu, rows, cols, x[0])
    eg, eu = 1e-4 * Sg + 1e-6, 1e-4 * Su + 1e-6
    # |SiLU'| <= 1.1; the fp32 epilogue adds a few rounding steps of h.
    bound = 1.1 * eg * (np.abs(u) + eu) + np.abs(oracle.silu(g)) * eu + 1e-6 * np.abs(h_ref) + 1e-7
    err = np.abs(h - h_ref)
    assert (err <= bound).all(), f"{name} swiglu outliers x{ratio:g}: worst err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("name", ["Q8_0", "Q4_0", "Q5_0"])
@pytest.mark.parametrize("ratio", RATIOS)
def test_attn_query_outliers(gpu, name, ratio):
    # One outlier per 32 query elements; the cached keys hold the type's zero
    # code in those dimensions, so the scores stay in the usual range and only
    # the representation of the other query elements is tested.
    t = type_id(name)
    T, nh, nkv, d = 300, 8, 2, 128
    G = nh // nkv
    q, pos = synth.activations_outliers(nh, d, 3900, ratio)
    K = synth.random_blocks(name, T * nkv, d, 3901)
    V = synth.random_blocks(name, T * nkv, d, 3902)
    codes, sc, mins, _, _ = oracle.unpack(t, K, T * nkv * d // 32)
    codes = codes.reshape(T, nkv, d)
    for h in range(nh):
        dims = 32 * np.arange(d // 32) + pos[h]
        codes[:, h // G, dims] = ZERO_CODE[name]
    d_bits = _half_bits(K, name, T * nkv * d // 32, 0)
    K2 = oracle.pack(t, codes.reshape(-1, 32), sc, mins, d_bits)
    scale = 1.0 / np.sqrt(d)
    o = qk.attn_decode(t, dev_f32(q, gpu), dev_u8(K2, gpu), dev_u8(V, gpu), T, nh, nkv, d, scale).cpu().numpy()
    ref, Sv = oracle.attn_decode(t, q, K2, V, T, nh, nkv, d, scale)
    err = np.abs(o - ref)
    bound = 2e-4 * Sv + 1e-6
    assert (err <= bound).all(), f"{name} attention outliers x{ratio:g}: worst err/bound {np.max(err / bound):.3g}"
