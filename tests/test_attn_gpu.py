"""qk_attn_decode (decode attention over a Q8_0 / Q5_0 / Q4_0 KV cache)
against the oracle on the same blocks: |out - ref| <= 2e-4 * sum_t p_t |V| +
1e-6 per output.  Shapes cover one position, a ragged last chunk, several
chunks, grouped-query heads (1, 4 and 8 query heads per kv head) and head
dimensions 32 to 256; a long cache is checked on sampled heads."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import dev_u8, gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

RTOL = 2e-4


def run(gpu, name, Tn, nh, nkv, d, seed, scale=None):
    t = type_id(name)
    K = synth.random_blocks(name, Tn * nkv, d, seed)
    V = synth.random_blocks(name, Tn * nkv, d, seed + 1)
    q = synth.activations(nh, d, seed + 2)
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    out = qk.attn_decode(t, torch.from_numpy(q).to(gpu), dev_u8(K, gpu), dev_u8(V, gpu), Tn, nh, nkv, d, scale)
    qk.device_status()
    ref, Sv = oracle.attn_decode(t, q, K, V, Tn, nh, nkv, d, scale)
    return out.cpu().numpy(), ref, Sv


CASES = [
    ("Q8_0", 1, 4, 4, 128),
    ("Q8_0", 300, 32, 8, 128),     # a ragged last chunk, 4 heads per kv head
    ("Q8_0", 1000, 8, 1, 64),      # 8 heads per kv head
    ("Q4_0", 777, 16, 4, 128),
    ("Q5_0", 513, 8, 8, 32),
    ("Q8_0", 260, 4, 2, 256),
]


@pytest.mark.parametrize("name,Tn,nh,nkv,d", CASES)
def test_attn_decode_parity(gpu, name, Tn, nh, nkv, d):
    out, ref, Sv = run(gpu, name, Tn, nh, nkv, d, 800 + Tn + d)
    err = np.abs(out - ref) - (RTOL * Sv + 1e-6)
    assert (err <= 0).all(), f"{name} T={Tn}: worst excess {err.max():.3e}"


@pytest.mark.parametrize("name", ["Q8_0", "Q5_0", "Q4_0"])
@pytest.mark.parametrize("Tn", [191, 192, 193, 255, 256, 257, 385, 513])
def test_attn_decode_chunk_edges(gpu, name, Tn):
    # Position counts on both sides of one and two chunks of 192 and of 256
    # positions, and a single position left over in the last chunk.
    out, ref, Sv = run(gpu, name, Tn, 8, 2, 128, 1200 + Tn)
    err = np.abs(out - ref) - (RTOL * Sv + 1e-6)
    assert (err <= 0).all(), f"{name} T={Tn}: worst excess {err.max():.3e}"


def test_attn_decode_peaked_scores(gpu):
    # A large scale makes the softmax nearly one-hot: the chunk maxima and
    # the log-sum-exp combination carry the result.
    out, ref, Sv = run(gpu, "Q8_0", 1500, 8, 2, 128, 900, scale=3.0)
    assert (np.abs(out - ref) <= RTOL * Sv + 1e-6).all()


def test_attn_decode_long_cache_sampled_heads(gpu):
    # 32k positions, Llama-3-8B-like heads (32 query, 8 kv, d = 128): every
    # output of two sampled kv heads against the oracle on those heads' rows.
    t, Tn, nh, nkv, d = qk.Q8_0, 32768, 32, 8, 128
    K = synth.random_blocks_torch("Q8_0", Tn * nkv, d, 950, gpu)
    V = synth.random_blocks_torch("Q8_0", Tn * nkv, d, 951, gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(952)
    q = torch.randn((nh, d), device=gpu, generator=g)
    out = qk.attn_decode(t, q, K, V, Tn, nh, nkv, d, 1.0 / np.sqrt(d)).cpu().numpy()
    qk.device_status()
    rb = qk.row_bytes(t, d)
    grp = nh // nkv
    for kv in (0, 5):
        rows = torch.arange(Tn, device=gpu) * nkv + kv
        idx = (rows[:, None] * rb + torch.arange(rb, device=gpu)[None, :]).reshape(-1)
        Kh, Vh = K[idx].cpu().numpy(), V[idx].cpu().numpy()
        qh = q[kv * grp:(kv + 1) * grp].cpu().numpy()
        ref, Sv = oracle.attn_decode(t, qh, Kh, Vh, Tn, grp, 1, d, 1.0 / np.sqrt(d))
        got = out[kv * grp:(kv + 1) * grp]
        assert (np.abs(got - ref) <= RTOL * Sv + 1e-6).all(), f"kv head {kv}"


def test_attn_decode_deterministic(gpu):
    a, _, _ = run(gpu, "Q4_0", 2000, 16, 4, 128, 990)
    b, _, _ = run(gpu, "Q4_0", 2000, 16, 4, 128, 990)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name,Tn,nh,nkv,d", [
    ("Q4_0", 400, 8, 8, 128),    # one head per kv head
    ("Q5_0", 350, 16, 8, 64),    # two heads per kv head
    ("Q8_0", 290, 8, 1, 32),     # eight heads, d = 32 (whole blocks per lane)
    ("Q5_0", 700, 32, 4, 256),   # eight heads, d = 256: the runtime-group path
    ("Q4_0", 100, 2, 1, 32),     # two heads, d = 32: the runtime-group path
    ("Q8_0", 333, 8, 4, 128),    # two heads, d = 128: p V on the MMA, half its columns
    ("Q4_0", 257, 4, 2, 128),    # the same for Q4_0, a ragged last stage
])
def test_attn_decode_every_group_path(gpu, name, Tn, nh, nkv, d):
    out, ref, Sv = run(gpu, name, Tn, nh, nkv, d, 1100 + Tn + d)
    assert (np.abs(out - ref) <= RTOL * Sv + 1e-6).all()


def test_attn_decode_maximum_positions(gpu):
    # The largest cache the call accepts, T = 65535 * 256 positions (one kv
    # head, two query heads, d = 32, Q4_0: 2 x 302 MB), every output against
    # the oracle.
    t, Tn, nh, nkv, d = qk.Q4_0, 65535 * 256, 2, 1, 32
    K = synth.random_blocks_torch("Q4_0", Tn * nkv, d, 1300, gpu)
    V = synth.random_blocks_torch("Q4_0", Tn * nkv, d, 1301, gpu)
    g = torch.Generator(device=gpu)
    g.manual_seed(1302)
    q = torch.randn((nh, d), device=gpu, generator=g)
    out = qk.attn_decode(t, q, K, V, Tn, nh, nkv, d, 1.0 / np.sqrt(d)).cpu().numpy()
    qk.device_status()
    ref, Sv = oracle.attn_decode(t, q.cpu().numpy(), K.cpu().numpy(), V.cpu().numpy(), Tn, nh, nkv, d, 1.0 / np.sqrt(d))
    assert (np.abs(out - ref) <= RTOL * Sv + 1e-6).all()
    del K, V
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["Q8_0", "Q4_0"])
@pytest.mark.parametrize("v_scale", [1e-7, 1e-5, 1e-2, 50.0, "mixed"])
def test_attn_decode_v_scale_range(gpu, name, v_scale):
    # d = 128, four query heads per kv head (p V on the MMA with the stage's
    # power-of-two scale): V block scales from fp16 subnormals (1e-7) to
    # ~200, and a cache whose positions mix scales 2^30 apart inside every
    # stage.
    t, Tn, nh, nkv, d = type_id(name), 1000, 16, 4, 128
    K = synth.random_blocks(name, Tn * nkv, d, 1400)
    if v_scale == "mixed":
        V = synth.random_blocks(name, Tn * nkv, d, 1401).copy()
        blocks = V.reshape(-1, qk.block_bytes(t))
        dv = blocks[:, :2].copy().view(np.float16).astype(np.float32)
        pos = np.arange(blocks.shape[0]) // (nkv * d // 32)
        dv[pos % 3 == 1] *= 2.0 ** -20
        dv[pos % 7 == 2] *= 2.0 ** 10
        blocks[:, :2] = dv.astype(np.float16).view(np.uint8).reshape(-1, 2)
    else:
        V = synth.random_blocks(name, Tn * nkv, d, 1401, d_scale=v_scale)
    q = synth.activations(nh, d, 1402)
    out = qk.attn_decode(t, torch.from_numpy(q).to(gpu), dev_u8(K, gpu), dev_u8(V, gpu), Tn, nh, nkv, d,
                         1.0 / np.sqrt(d)).cpu().numpy()
    qk.device_status()
    ref, Sv = oracle.attn_decode(t, q, K, V, Tn, nh, nkv, d, 1.0 / np.sqrt(d))
    assert np.isfinite(out).all()
    err = np.abs(out - ref) - (RTOL * Sv + 1e-6)
    assert (err <= 0).all(), f"{name} V scale {v_scale}: worst excess {err.max():.3e}"
