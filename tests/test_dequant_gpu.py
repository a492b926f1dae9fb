"""Device unpackers and qk_dequant against the oracle: integer fields
bit-exact, fp32 weights bit-exact (the tolerance allows 1 ulp; the formulas
are exact in fp32 up to the last rounding, so 0 is expected), bf16 outputs
equal to round-to-nearest-even of the oracle's fp32 weights."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from golden_io import all_fixtures, load
from gpu_helpers import dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu
NAMES = ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"]


@pytest.mark.parametrize("name", NAMES)
def test_unpack_fields_bit_exact(gpu, name):
    t = type_id(name)
    nb = 777
    W = synth.random_blocks(name, 1, nb * synth.GEOMETRY[name][1], 100 + t)
    codes, sc, mins, d, dmin = (a.cpu().numpy() for a in qk.unpack(t, dev_u8(W, gpu), nb))
    rc, rsc, rmins, rd, rdmin = oracle.unpack(t, W, nb)
    assert np.array_equal(codes, rc)
    assert np.array_equal(sc, rsc)
    assert np.array_equal(mins, rmins)
    assert np.array_equal(d.view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(dmin.view(np.uint32), rdmin.view(np.uint32))


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("rows,nblk", [(1, 1), (3, 5), (67, 17)])
def test_dequant_fp32_bit_exact(gpu, name, rows, nblk):
    t = type_id(name)
    cols = nblk * synth.GEOMETRY[name][1]
    W = synth.random_blocks(name, rows, cols, 200 + rows + t)
    got = qk.dequant(t, dev_u8(W, gpu), rows, cols).cpu().numpy()
    ref = oracle.dequant(t, W, rows, cols)
    ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("name", NAMES)
def test_dequant_bf16_rounding(gpu, name):
    t = type_id(name)
    rows, cols = 9, 4 * synth.GEOMETRY[name][1]
    W = synth.random_blocks(name, rows, cols, 300 + t)
    got = qk.dequant(t, dev_u8(W, gpu), rows, cols, bf16=True).cpu().view(torch.int16).numpy()
    ref = torch.from_numpy(oracle.dequant(t, W, rows, cols)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("path", all_fixtures(), ids=lambda p: p.rsplit("/", 1)[-1])
def test_golden_blocks_on_device(gpu, path):
    name, blk, expect = load(path)
    t = type_id(name)
    w = qk.dequant(t, dev_u8(blk, gpu), 1, expect.size).cpu().numpy()[0]
    assert np.array_equal(w.astype(np.float64), expect)


def test_dequant_output_canaries(gpu):
    # Output surrounded by NaN sentinels: only the [rows, cols] window changes.
    t, rows, cols = qk.Q6_K, 5, 512
    W = synth.random_blocks("Q6_K", rows, cols, 400)
    buf = torch.full((rows * cols + 64,), float("nan"), device=gpu)
    out = buf[32:32 + rows * cols].view(rows, cols)
    qk.dequant(t, dev_u8(W, gpu), rows, cols, out=out)
    b = buf.cpu().numpy()
    assert np.isnan(b[:32]).all() and np.isnan(b[-32:]).all()
    assert np.array_equal(b[32:-32].reshape(rows, cols), oracle.dequant(t, W, rows, cols))
