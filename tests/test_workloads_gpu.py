"""Parity at the workloads' full sizes, in the launch configuration the bench
times: every output where the oracle finishes in seconds, sampled outputs
(computed one by one by the oracle) elsewhere."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import assert_gemv_close, dev_f32, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu


def test_tiny_q4k_all_outputs(gpu):
    # 256 x 1024 Q4_K, uniform codes and 6-bit scales/mins,
    # d = |N(0,1)|*1e-2, dmin = |N(0,1)|*5e-3, x ~ N(0,1).
    (_, name, rows, cols), = synth.TINY
    W = synth.random_blocks(name, rows, cols, 1001, d_scale=1e-2, dmin_scale=5e-3)
    x = synth.activations(1, cols, 1002)
    y = qk.gemv(qk.Q4_K, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
    y_ref, S = oracle.gemv(qk.Q4_K, W, rows, cols, x)
    assert_gemv_close(y, y_ref, S, what="tiny")


def test_llama7b_layer_all_outputs(gpu):
    # Codes from the plain quantizer applied to N(0, 0.02) weights.
    for i, (nm, name, rows, cols) in enumerate(synth.LLAMA7B_LAYER):
        t = type_id(name)
        W = oracle.quantize(t, synth.normal_weights(rows, cols, 1100 + i))
        x = synth.activations(1, cols, 1200 + i)
        y = qk.gemv(t, dev_u8(W, gpu), rows, cols, dev_f32(x, gpu)).cpu().numpy()
        y_ref, S = oracle.gemv(t, W, rows, cols, x)
        assert_gemv_close(y, y_ref, S, what=nm)


def _sampled_check(gpu, t, Wd, rows, cols, xd, y, nsamp, seed, what):
    g = synth.rng(seed)
    M = xd.shape[0]
    ni = np.sort(g.choice(rows, size=min(nsamp, rows), replace=False))
    mi = g.integers(0, M, ni.size)
    rb = qk.row_bytes(t, cols)
    # Only the sampled rows travel to the host.
    Wrows = torch.cat([Wd[n * rb:(n + 1) * rb] for n in ni]).cpu().numpy()
    x = xd.cpu().numpy()
    y_ref, S = oracle.entries(t, Wrows, ni.size, cols, mi, np.arange(ni.size), x=x)
    got = y[mi, ni]
    assert_gemv_close(got, y_ref, S, what=what)


def test_llama7b_stack_sampled(gpu):
    # The full 32-layer stack (3.87 GiB of packed weights) is run matrix by
    # matrix, exactly as the bench does; 4 outputs per matrix are checked.
    stack = synth.llama7b_stack()
    for i, (nm, name, rows, cols) in enumerate(stack):
        t = type_id(name)
        Wd = synth.random_blocks_torch(name, rows, cols, 5000 + i, gpu)
        g = torch.Generator(device=gpu)
        g.manual_seed(9000 + i)
        xd = torch.randn((1, cols), device=gpu, generator=g)
        y = qk.gemv(t, Wd, rows, cols, xd).cpu().numpy()
        _sampled_check(gpu, t, Wd, rows, cols, xd, y, 4, 7000 + i, nm)
        del Wd


@pytest.mark.parametrize("name", ["Q4_K", "Q5_0"])
@pytest.mark.parametrize("M", list(synth.FFN_BATCHES))
def test_llama3_ffn_batches(gpu, name, M):
    for i, (nm, tname, rows, cols) in enumerate(synth.llama3_ffn(name)):
        t = type_id(tname)
        Wd = synth.random_blocks_torch(tname, rows, cols, 6000 + 10 * i + M, gpu)
        g = torch.Generator(device=gpu)
        g.manual_seed(6100 + 10 * i + M)
        xd = torch.randn((M, cols), device=gpu, generator=g)
        y = qk.gemv(t, Wd, rows, cols, xd).cpu().numpy()
        _sampled_check(gpu, t, Wd, rows, cols, xd, y, 48, 6200 + i, f"{nm} M={M}")


def test_decode_large_rows_several_reduction_chunks(gpu):
    # 40000 x 16384 Q4_K at M = 1: eight K slices, so a CTA's 264 rows are
    # reduced in two chunks of partial sums; sampled outputs, with rows at
    # both ends of the matrix.
    name, rows, cols = "Q4_K", 40000, 16384
    t = type_id(name)
    Wd = synth.random_blocks_torch(name, rows, cols, 7100, gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(7101)
    xd = torch.randn((1, cols), device=gpu, generator=g)
    y = qk.gemv(t, Wd, rows, cols, xd).cpu().numpy()
    _sampled_check(gpu, t, Wd, rows, cols, xd, y, 48, 7102, "Q4_K 40000x16384")
    rb = qk.row_bytes(t, cols)
    ends = np.array([0, 255, 256, 263, 264, rows - 1])
    Wrows = torch.cat([Wd[n * rb:(n + 1) * rb] for n in ends]).cpu().numpy()
    y_ref, S = oracle.entries(t, Wrows, ends.size, cols, np.zeros(ends.size, dtype=np.int64),
                              np.arange(ends.size), x=xd.cpu().numpy())
    assert_gemv_close(y[0, ends], y_ref, S, what="chunk edges")


def test_llama7b_layer_in_bench_launch_configuration(gpu):
    # The bench's step: q/k/v in one batched launch, o alone, gate/up batched,
    # down alone; one activation vector per launch; every output checked.
    import bench
    layer, groups = synth.LLAMA7B_LAYER, synth.LLAMA7B_LAYER_GROUPS
    Wh = [synth.random_blocks(name, rows, cols, 7300 + i) for i, (_, name, rows, cols) in enumerate(layer)]
    xh = [synth.activations(1, layer[g[0]][3], 7400 + gi) for gi, g in enumerate(groups)]
    Wd = [dev_u8(W, gpu) for W in Wh]
    xd = [dev_f32(x, gpu)[0] for x in xh]
    ys = [torch.empty(rows, device=gpu) for (_, _, rows, _) in layer]
    for gi, grp in enumerate(groups):
        bench.run_group(layer, grp, Wd, xd[gi], ys)
    qk.device_status()
    for gi, grp in enumerate(groups):
        for i in grp:
            (nm, name, rows, cols) = layer[i]
            y_ref, S = oracle.gemv(type_id(name), Wh[i], rows, cols, xh[gi])
            assert_gemv_close(ys[i].cpu().numpy()[None, :], y_ref, S, what=f"bench layer {nm}")
