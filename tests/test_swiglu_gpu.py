"""qk_gemv_swiglu (decode SwiGLU gate, h = SiLU(Wg x) * (Wu x), one launch)
against the oracle's fp64 SwiGLU.  Tolerance per output, from the GEMV bound
eps = 1e-4 * sum|w x| + 1e-6 on each of g and u, |SiLU'| <= 1.1, and the fp32
epilogue (expf within 2 ulp, a division, a product):
    |h - h_ref| <= 1.1 * eps_g * (|u| + eps_u) + |SiLU(g)| * eps_u + 1e-6 |h| + 1e-7."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

CASES = [
    ("Q4_K", 96, 1024),
    ("Q4_K", 1, 4096),
    ("Q4_K", 14336, 4096),   # Llama-3-8B gate/up
    ("Q6_K", 33, 2048),
    ("Q8_0", 130, 512),
    ("Q5_0", 17, 256),
    ("Q4_0", 40, 4096),
    ("Q5_K", 96, 2048),
    ("Q2_K", 64, 1024),
    ("Q3_K", 50, 2048),
]


def check(h, h_ref, g, u, Sg, Su, what):
    eg, eu = 1e-4 * Sg + 1e-6, 1e-4 * Su + 1e-6
    tol = 1.1 * eg * (np.abs(u) + eu) + np.abs(oracle.silu(g)) * eu + 1e-6 * np.abs(h_ref) + 1e-7
    bad = np.abs(h - h_ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs out of tolerance, first at {int(np.argmax(bad))}"


@pytest.mark.parametrize("name,rows,cols", CASES)
def test_swiglu_parity(gpu, name, rows, cols):
    t = type_id(name)
    Wg = synth.random_blocks(name, rows, cols, 7100 + rows)
    Wu = synth.random_blocks(name, rows, cols, 7200 + rows)
    x = synth.activations(1, cols, 7300 + cols)[0]
    h = qk.gemv_swiglu(t, dev_u8(Wg, gpu), dev_u8(Wu, gpu), rows, cols, torch.from_numpy(x).to(gpu)).cpu().numpy()
    qk.device_status()
    h_ref, g, u, Sg, Su = oracle.swiglu(t, Wg, Wu, rows, cols, x)
    check(h, h_ref, g, u, Sg, Su, f"swiglu {name} {rows}x{cols}")


def test_swiglu_matches_the_unfused_pair(gpu):
    # The same g and u from qk_gemv_batch, then SiLU * up in torch: agreement
    # to a few fp32 ulps (the dot products are the same kernel's).
    t, rows, cols = qk.Q4_K, 2048, 4096
    Wg = dev_u8(synth.random_blocks("Q4_K", rows, cols, 7401), gpu)
    Wu = dev_u8(synth.random_blocks("Q4_K", rows, cols, 7402), gpu)
    x = torch.from_numpy(synth.activations(1, cols, 7403)[0]).to(gpu)
    h = qk.gemv_swiglu(t, Wg, Wu, rows, cols, x)
    g, u = qk.gemv_batch(t, [Wg, Wu], [rows, rows], cols, x)
    ref = torch.nn.functional.silu(g) * u
    assert torch.allclose(h, ref, rtol=2e-6, atol=1e-7)


def test_swiglu_edges(gpu):
    t = qk.Q8_0
    h = torch.full((5,), 7.0, device=gpu)
    z = torch.zeros(16, dtype=torch.uint8, device=gpu)
    qk.gemv_swiglu(t, z, z, 5, 0, torch.zeros(4, device=gpu), h=h)   # cols == 0: h = SiLU(0) * 0
    assert (h == 0).all()
    qk.gemv_swiglu(t, z, z, 0, 32, torch.zeros(32, device=gpu), h=torch.empty(0, device=gpu))   # rows == 0
    # Large |g|: e^-g overflows to inf (h -> -0 * u) or vanishes (h -> g * u).
    rows, cols = 4, 32
    blk = np.zeros((rows, 34), np.uint8)
    blk[:, 1] = 0x5C   # d = fp16 256.0
    blk[:, 2:] = np.array([[127], [-128], [64], [1]], np.int8).view(np.uint8)
    up = np.zeros((rows, 34), np.uint8)
    up[:, 1] = 0x3C    # d = 1
    up[:, 2:] = 1
    x = np.full(cols, 2.0, np.float32)
    hd = qk.gemv_swiglu(t, dev_u8(blk.reshape(-1), gpu), dev_u8(up.reshape(-1), gpu), rows, cols,
                        torch.from_numpy(x).to(gpu)).cpu().numpy()
    h_ref, g, u, Sg, Su = oracle.swiglu(t, blk.reshape(-1), up.reshape(-1), rows, cols, x)
    assert np.all(np.isfinite(hd))
    check(hd, h_ref, g, u, Sg, Su, "swiglu saturated")
    qk.device_status()
