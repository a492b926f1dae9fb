"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no dequantization or matmul arithmetic: it only draws
random numbers and places them.  Packed blocks are random bytes with the
binary16 scale fields overwritten by finite values of a chosen magnitude, so
every code, sub-block scale and min is uniform over its range.  Activations
are N(0, 1).  Workload shapes (the Llama-7B decoder layer, the Llama-3-8B FFN,
the prefill recipe) are listed here too, so that every user draws the same
inputs from the same seeds.

Block geometry (bytes, weights) and the byte offsets of the binary16 fields:
  Q4_K 144 B / 256 w, d at 0, dmin at 2     Q6_K 210 B / 256 w, d at 208
  Q8_0  34 B /  32 w, d at 0                Q5_0  22 B /  32 w, d at 0
  Q4_0  18 B /  32 w, d at 0                Q5_K 176 B / 256 w, d at 0, dmin at 2
  Q2_K  84 B / 256 w, d at 80, dmin at 82   Q3_K 110 B / 256 w, d at 108
"""
from __future__ import annotations

import numpy as np

TYPE_IDS = {"Q4_K": 1, "Q6_K": 2, "Q8_0": 3, "Q5_0": 4, "Q4_0": 5, "Q5_K": 6, "Q2_K": 7, "Q3_K": 8}
GEOMETRY = {  # name: (block bytes, weights per block, d offset, dmin offset or None)
    "Q4_K": (144, 256, 0, 2),
    "Q6_K": (210, 256, 208, None),
    "Q8_0": (34, 32, 0, None),
    "Q5_0": (22, 32, 0, None),
    "Q4_0": (18, 32, 0, None),
    "Q5_K": (176, 256, 0, 2),
    "Q2_K": (84, 256, 80, 82),
    "Q3_K": (110, 256, 108, None),
}


def type_name(t) -> str:
    if isinstance(t, str):
        return t
    for k, v in TYPE_IDS.items():
        if v == t:
            return k
    raise KeyError(t)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(t, cols: int) -> int:
    bb, be, _, _ = GEOMETRY[type_name(t)]
    assert cols % be == 0
    return cols // be * bb


def random_blocks(t, rows: int, cols: int, seed: int, d_scale: float = 1e-2,
                  dmin_scale: float = 5e-3) -> np.ndarray:
    """Packed [rows, cols] matrix of random blocks (uint8, flat).

    Codes, 6-bit scales / mins and int8 scales are uniform (random bytes);
    d = fp16(|N(0,1)| * d_scale), dmin = fp16(|N(0,1)| * dmin_scale)."""
    name = type_name(t)
    bb, be, d_off, dmin_off = GEOMETRY[name]
    nb = rows * (cols // be)
    g = rng(seed)
    W = g.integers(0, 256, size=(nb, bb), dtype=np.uint8)
    d = (np.abs(g.standard_normal(nb)) * d_scale).astype(np.float16)
    W[:, d_off:d_off + 2] = d.view(np.uint8).reshape(nb, 2)
    if dmin_off is not None:
        dm = (np.abs(g.standard_normal(nb)) * dmin_scale).astype(np.float16)
        W[:, dmin_off:dmin_off + 2] = dm.view(np.uint8).reshape(nb, 2)
    return W.reshape(-1)


def random_blocks_torch(t, rows: int, cols: int, seed: int, device, d_scale: float = 1e-2,
                        dmin_scale: float = 5e-3):
    """Same distribution as random_blocks, drawn with torch on `device`
    (used for the multi-GB stacks, where host generation would dominate).
    Returns a flat uint8 tensor.  Not bitwise equal to random_blocks."""
    import torch
    name = type_name(t)
    bb, be, d_off, dmin_off = GEOMETRY[name]
    nb = rows * (cols // be)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    W = torch.randint(0, 256, (nb, bb), dtype=torch.uint8, device=device, generator=g)
    d = (torch.randn(nb, device=device, generator=g).abs() * d_scale).to(torch.float16)
    W[:, d_off:d_off + 2] = d.view(torch.uint8).view(nb, 2)
    if dmin_off is not None:
        dm = (torch.randn(nb, device=device, generator=g).abs() * dmin_scale).to(torch.float16)
        W[:, dmin_off:dmin_off + 2] = dm.view(torch.uint8).view(nb, 2)
    return W.view(-1)


def normal_weights(rows: int, cols: int, seed: int, std: float = 0.02) -> np.ndarray:
    """fp32 weights ~ N(0, std^2), the input of the quantizer."""
    return (rng(seed).standard_normal((rows, cols)) * std).astype(np.float32)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """fp32 [M, K] ~ N(0, 1)."""
    return rng(seed).standard_normal((M, K)).astype(np.float32)


def activations_bf16_bits(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 [M, K] ~ N(0, 1), as raw uint16 bit patterns (drawn in fp32 and
    rounded by torch's fp32 -> bf16 conversion)."""
    import torch
    x = torch.from_numpy(activations(M, K, seed))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

# Tiny Q4_K GEMV: 256 x 1024 (4 super-blocks per row).
TINY = [("w", "Q4_K", 256, 1024)]

# One Llama-7B-shaped decoder layer at decode batch 1 (rows = out, cols = in).
LLAMA7B_LAYER = [
    ("q", "Q4_K", 4096, 4096), ("k", "Q4_K", 4096, 4096), ("v", "Q4_K", 4096, 4096),
    ("o", "Q4_K", 4096, 4096), ("gate", "Q4_K", 11008, 4096), ("up", "Q4_K", 11008, 4096),
    ("down", "Q6_K", 4096, 11008),
]


# The layer's matrices grouped by the activation vector they read: q/k/v
# project the same hidden state, gate/up the same one (one launch each).
LLAMA7B_LAYER_GROUPS = [(0, 1, 2), (3,), (4, 5), (6,)]


def llama7b_stack(n_layers: int = 32):
    """32 decoder layers + lm_head 32000 x 4096 Q6_K + two 4096^2 Q8_0 tensors."""
    out = []
    for layer in range(n_layers):
        out += [(f"l{layer}.{n}", t, r, c) for (n, t, r, c) in LLAMA7B_LAYER]
    out += [("lm_head", "Q6_K", 32000, 4096), ("q8a", "Q8_0", 4096, 4096), ("q8b", "Q8_0", 4096, 4096)]
    return out


# Llama-3-8B FFN (continuous-batching sweep), Q4_K and Q5_0 variants.
def llama3_ffn(t: str):
    return [("gate", t, 14336, 4096), ("up", t, 14336, 4096), ("down", t, 4096, 14336)]


FFN_BATCHES = (1, 4, 16, 64)

# Prefill dequant-GEMM: M = 2048 against every shape x type, plus the vocab.
PREFILL_M = 2048
PREFILL = ([(f"{s}_{t}", t, r, c) for t in ("Q4_K", "Q6_K", "Q8_0")
            for (s, r, c) in (("sq", 4096, 4096), ("up", 14336, 4096), ("down", 4096, 14336))]
           + [("vocab", "Q6_K", 128256, 4096)])


def activations_outliers(M: int, K: int, seed: int, ratio: float, block: int = 32):
    """fp32 [M, K] ~ N(0, 1) with one coordinate per `block` consecutive
    elements replaced by +-ratio (a massive activation, `ratio` times the
    typical magnitude).  Returns (x, pos) with pos int64 [M, K // block] the
    position of the outlier inside each block."""
    g = rng(seed)
    x = g.standard_normal((M, K)).astype(np.float32)
    nb = K // block
    pos = g.integers(0, block, size=(M, nb))
    sign = np.where(g.integers(0, 2, size=(M, nb)) == 0, -1.0, 1.0)
    cols = np.arange(nb)[None, :] * block + pos
    x[np.arange(M)[:, None], cols] = (sign * ratio).astype(np.float32)
    return x, pos
