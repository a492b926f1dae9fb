"""qk_gemm (tcgen05 tensor-core dequant-GEMM) against the oracle fed the same
bf16 activations: |Y - Y_ref| <= 5e-3 * sum|w x| per output.  Shapes cover
one tile, ragged weight rows and token counts, a K whose last 64-block is
half empty (32-weight blocks), every quant type, M from 1 to 1100, token
tiles whose second 256-token accumulator is empty, partial or full, and the
skinny pipeline (M <= 64) with fewer k-blocks than it has stages."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import GEMM_RTOL, assert_gemv_close, dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

CASES = [
    ("Q4_K", 128, 256, 256),
    ("Q4_K", 200, 512, 300),
    ("Q6_K", 136, 768, 64),
    ("Q8_0", 130, 96, 17),
    ("Q5_0", 256, 160, 1),
    ("Q5_0", 64, 1024, 257),
    ("Q8_0", 384, 2048, 512),
    ("Q4_K", 256, 512, 600),     # two 512-token tiles, the second with one live accumulator
    ("Q6_K", 130, 512, 1100),    # three token tiles, ragged rows
    ("Q5_0", 128, 320, 513),     # second tile holds a single token
    ("Q4_0", 200, 1056, 77),
    ("Q5_K", 200, 512, 300),     # the wide kernel: ragged rows, a partial second token tile
    ("Q2_K", 200, 512, 300),
    ("Q3_K", 130, 768, 600),
    ("Q3_K", 130, 768, 40),      # rows of 330 bytes: the wide kernel at a small batch
    # Skinny pipeline (M <= 64): fewer k-blocks than operand stages, a half
    # k-block at the end, ragged rows, one token.
    ("Q4_K", 130, 256, 40),
    ("Q8_0", 200, 96, 64),
    ("Q5_0", 257, 2080, 48),
    ("Q6_K", 129, 1536, 2),
    ("Q4_0", 128, 64 * 32, 63),
    ("Q5_K", 130, 768, 40),
    ("Q2_K", 130, 1024, 40),
    ("Q3_K", 200, 2048, 16),
    ("Q2_K", 257, 2304, 16),     # the small-batch decoders: every k-block position, ragged rows
    ("Q3_K", 131, 1280, 5),
]


def run_gemm(gpu, name, rows, cols, M, seed):
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, seed)
    Xb = synth.activations_bf16_bits(M, cols, seed + 1)
    Xd = torch.from_numpy(Xb.view(np.int16)).to(gpu).view(torch.bfloat16)
    Y = qk.gemm(t, dev_u8(W, gpu), rows, cols, Xd).cpu().numpy()
    qk.device_status()
    Y_ref, S = oracle.gemm_bf16(t, W, rows, cols, Xb)
    return Y, Y_ref, S


@pytest.mark.parametrize("name,rows,cols,M", CASES)
def test_gemm_parity(gpu, name, rows, cols, M):
    Y, Y_ref, S = run_gemm(gpu, name, rows, cols, M, 3000 + rows + M)
    assert Y.shape == (M, rows)
    assert_gemv_close(Y, Y_ref, S, rtol=GEMM_RTOL, atol=0.0, what=f"gemm {name} {rows}x{cols} M={M}")


def test_gemm_matches_dequant_then_matmul(gpu):
    # Same bf16 weights, fp32 accumulation on both sides: agreement far
    # inside the GEMM tolerance.
    name, rows, cols, M = "Q4_K", 256, 1024, 256
    t = type_id(name)
    W = synth.random_blocks(name, rows, cols, 4000)
    Wd = dev_u8(W, gpu)
    Xb = synth.activations_bf16_bits(M, cols, 4001)
    Xd = torch.from_numpy(Xb.view(np.int16)).to(gpu).view(torch.bfloat16)
    Y = qk.gemm(t, Wd, rows, cols, Xd)
    Wbf = qk.dequant(t, Wd, rows, cols, bf16=True)
    ref = (Xd.float() @ Wbf.float().t())
    _, S = oracle.gemm_bf16(t, W, rows, cols, Xb)
    assert np.all(np.abs((Y - ref).cpu().numpy()) <= 1e-4 * S + 1e-5)


def test_gemm_empty_and_zero_k(gpu):
    t = qk.Q4_K
    Y = torch.full((4, 8), 3.0, device=gpu)
    qk.gemm(t, torch.zeros(16, dtype=torch.uint8, device=gpu), 8, 0,
            torch.zeros((4, 0), dtype=torch.bfloat16, device=gpu), Y=Y)
    assert (Y == 0).all()
    qk.gemm(t, torch.zeros(144, dtype=torch.uint8, device=gpu), 0, 256,
            torch.zeros((4, 256), dtype=torch.bfloat16, device=gpu), Y=torch.empty((4, 0), device=gpu))
    qk.device_status()


# Small token batches against long K: the plan splits K over CTAs (partials
# in the workspace, added in split order) and narrows the MMA to M rounded up
# to 16.
SPLIT_CASES = [
    ("Q4_K", 256, 8192, 4),
    ("Q6_K", 100, 14336, 16),
    ("Q8_0", 384, 4096, 64),
    ("Q5_0", 96, 5120, 9),
    ("Q4_K", 130, 2048, 1),
    ("Q4_0", 64, 8192, 5),
    ("Q5_K", 300, 8192, 16),
    ("Q3_K", 96, 8192, 4),
    ("Q2_K", 64, 8192, 9),
]


@pytest.mark.parametrize("name,rows,cols,M", SPLIT_CASES)
def test_gemm_split_k_parity(gpu, name, rows, cols, M):
    t = type_id(name)
    assert qk.gemm_workspace(t, rows, cols, M) > 0          # the split path is taken
    Y, Y_ref, S = run_gemm(gpu, name, rows, cols, M, 3500 + rows + M)
    assert_gemv_close(Y, Y_ref, S, rtol=GEMM_RTOL, atol=0.0, what=f"split gemm {name} {rows}x{cols} M={M}")


def test_gemm_split_k_is_deterministic_and_checks_workspace(gpu):
    name, rows, cols, M = "Q4_K", 256, 8192, 8
    t = type_id(name)
    W = dev_u8(synth.random_blocks(name, rows, cols, 3600), gpu)
    Xb = synth.activations_bf16_bits(M, cols, 3601)
    Xd = torch.from_numpy(Xb.view(np.int16)).to(gpu).view(torch.bfloat16)
    a = qk.gemm(t, W, rows, cols, Xd).cpu().numpy()
    b = qk.gemm(t, W, rows, cols, Xd).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    need = qk.gemm_workspace(t, rows, cols, M)
    small = torch.empty(need - 16, dtype=torch.uint8, device=gpu)
    with pytest.raises(qk.QKError) as e:
        qk.gemm(t, W, rows, cols, Xd, ws=small)
    assert e.value.status == 5



# Small batches at full size and with many row tiles: the Llama-3-8B FFN
# shapes (K split or not by the plan), sampled rows including both ends of
# row tiles, every token, against the oracle on those rows.
@pytest.mark.parametrize("rows,cols,M", [(14336, 4096, 16), (4096, 14336, 64), (14336, 4096, 1), (38400, 1024, 5)])
def test_gemm_small_batch_llama3_ffn_sampled(gpu, rows, cols, M):
    t = qk.Q4_K
    Wd = synth.random_blocks_torch("Q4_K", rows, cols, 3800 + M, gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(3801 + M)
    Xd = torch.randn((M, cols), device=gpu, generator=g).to(torch.bfloat16)
    Y = qk.gemm(t, Wd, rows, cols, Xd).cpu().numpy()
    qk.device_status()
    rng = synth.rng(3802 + M)
    ni = np.unique(np.concatenate([rng.choice(rows, 40, replace=False), [0, 127, 128, 255, rows - 1]]))
    rb = qk.row_bytes(t, cols)
    Wrows = torch.cat([Wd[n * rb:(n + 1) * rb] for n in ni]).cpu().numpy()
    Xb = Xd.view(torch.int16).cpu().numpy().view(np.uint16)
    Y_ref, S = oracle.gemm_bf16(t, Wrows, ni.size, cols, Xb)
    assert_gemv_close(Y[:, ni], Y_ref, S, rtol=GEMM_RTOL, atol=0.0, what=f"FFN gemm {rows}x{cols} M={M}")


# The prefill workload at full size in the bench's launch configuration:
# every matrix of the M = 2048 recipe (Q4_K / Q6_K / Q8_0 at 4096x4096,
# 14336x4096 and 4096x14336, and the 128256x4096 Q6_K vocabulary), all 2048
# tokens of sampled rows (both ends of row tiles among them) against the
# oracle on those rows.
@pytest.mark.parametrize("i", range(len(synth.PREFILL)), ids=[p[0] for p in synth.PREFILL])
def test_gemm_prefill_recipe_full_size_sampled(gpu, i):
    nm, name, rows, cols = synth.PREFILL[i]
    t = synth.TYPE_IDS[name]
    M = synth.PREFILL_M
    Wd = synth.random_blocks_torch(name, rows, cols, 4100 + i, gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(4200 + i)
    Xd = torch.randn((M, cols), device=gpu, generator=g).to(torch.bfloat16)
    Y = qk.gemm(t, Wd, rows, cols, Xd).cpu().numpy()   # as the bench calls it
    qk.device_status()
    rng = synth.rng(4300 + i)
    ni = np.unique(np.concatenate([rng.choice(rows, 12, replace=False), [0, 127, 128, rows - 129, rows - 1]]))
    rb = qk.row_bytes(t, cols)
    Wrows = torch.cat([Wd[n * rb:(n + 1) * rb] for n in ni]).cpu().numpy()
    Xb = Xd.view(torch.int16).cpu().numpy().view(np.uint16)
    Y_ref, S = oracle.gemm_bf16(t, Wrows, ni.size, cols, Xb)
    assert_gemv_close(Y[:, ni], Y_ref, S, rtol=GEMM_RTOL, atol=0.0, what=f"prefill {nm} {rows}x{cols} M={M}")
    del Wd, Xd
    torch.cuda.empty_cache()
