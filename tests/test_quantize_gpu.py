"""qk_quantize (fp32 weights -> packed blocks) against the oracle's quantizer:
the bytes must be identical (codes, scales and fp16 fields are integer work,
and both sides take every rounding decision in the same fp32 operations).
Shapes cover one warp's 32 groups of 32 weights, several warps and a ragged
last warp; the special-value blocks cover the zero-divisor paths, fp16
subnormal and overflowing scales, exact rounding ties, NaN, infinities and
negative zero."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gpu_helpers import gpu, type_id  # noqa: F401

pytestmark = pytest.mark.gpu

CASES = [
    ("Q4_K", 3, 768),      # 72 groups: two warps + a ragged 8
    ("Q4_K", 37, 2048),
    ("Q6_K", 5, 256),
    ("Q6_K", 17, 4096),
    ("Q8_0", 5, 96),       # 15 groups: less than one warp
    ("Q8_0", 33, 1024),
    ("Q5_0", 33, 224),
    ("Q5_0", 8, 4096),
    ("Q4_0", 7, 4096),
    ("Q4_0", 3, 352),
    ("Q5_K", 3, 768),
    ("Q5_K", 37, 2048),
    ("Q2_K", 3, 768),
    ("Q2_K", 37, 2048),
    ("Q3_K", 3, 768),
    ("Q3_K", 37, 2048),
]


def run(gpu, t, w):
    got = qk.quantize(t, torch.from_numpy(np.ascontiguousarray(w)).to(gpu)).cpu().numpy()
    qk.device_status()
    return got


@pytest.mark.parametrize("name,rows,cols", CASES)
def test_quantize_matches_oracle(gpu, name, rows, cols):
    t = type_id(name)
    w = synth.normal_weights(rows, cols, 5000 + rows + cols)
    got = run(gpu, t, w)
    ref = oracle.quantize(t, w)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref), f"{name}: {int((got != ref).sum())} bytes differ"


def special_blocks(n):
    """Rows of n weights, each row one special pattern (n = 256 or 32)."""
    rng = np.random.default_rng(6060)
    base = rng.standard_normal(n).astype(np.float32) * 0.02
    rows = [
        np.zeros(n),
        np.full(n, 0.37),
        np.full(n, -0.37),
        np.where(np.arange(n) == 5, 3.0, 0.0),                 # one spike
        -np.abs(base),                                           # all negative
        np.abs(base) + 0.01,                                     # all positive, min > 0
        base * 1e-5,                                             # fp16-subnormal scales
        base * 1e-9,                                             # scales that round to 0
        base * 2e7,                                              # scales that overflow fp16
        np.where(np.arange(n) % 32 == 0, 127.0 / 128.0,
                 (np.arange(n) % 32 - 16 + 0.5) / 128.0),       # max 127/128: Q8_0 d = 1/128, exact .5 ties
        np.where(np.arange(n) == 7, np.nan, base),               # NaN inside a block
        np.where(np.arange(n) % 32 == 0, np.nan, base),          # NaN first in every 32-weight group
        np.where(np.arange(n) % 16 == 0, np.nan, -np.abs(base)),  # ... and every 16-weight group
        np.where(np.arange(n) == 9, np.inf, base),
        np.where(np.arange(n) == 9, -np.inf, base),
        np.where(np.arange(n) % 3 == 0, -0.0, base),
        np.concatenate([np.full(n // 2, -50.0), base[: n - n // 2]]),   # wide mins, tiny ranges
    ]
    return np.stack([np.asarray(r, np.float32) for r in rows])


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
def test_quantize_special_values(gpu, name):
    t = type_id(name)
    n = 256 if name in ("Q4_K", "Q6_K", "Q5_K", "Q2_K", "Q3_K") else 32
    w = special_blocks(n)
    # Repeat the patterns along each row so every lane position of a warp sees them.
    w = np.tile(w, (1, 8))
    with np.errstate(invalid="ignore", over="ignore"):
        ref = oracle.quantize(t, w)
    got = run(gpu, t, w)
    assert np.array_equal(got, ref), f"{name}: {int((got != ref).sum())} bytes differ"


@pytest.mark.parametrize("name,qmax", [("Q8_0", 100), ("Q5_0", 14), ("Q4_0", 6)])
def test_quantize_near_ties(gpu, name, qmax):
    # Weights whose quotient by the block scale lies just beside a half-integer
    # (offsets from 0 to +-1e-3 of a code step): the code decisions near the
    # rounding boundary.  The block's largest weight is kept from a first
    # quantization, so the fp16 scale d is known and stays the same.
    t = type_id(name)
    rng = np.random.default_rng(7070)
    nb = 512
    base = rng.standard_normal((nb, 32)).astype(np.float32)
    d = oracle.quantize(t, base).reshape(nb, -1)[:, :2].copy().view(np.float16).astype(np.float64)[:, 0]
    deltas = np.array([0.0, 1e-7, -1e-7, 1e-6, -1e-6, 1e-5, -1e-5, 5e-5, -5e-5,
                       1.2e-4, -1.2e-4, 2.4e-4, -2.4e-4, 2.6e-4, -2.6e-4, 1e-3, -1e-3])
    m = rng.integers(-qmax - 1, qmax + 1, size=(nb, 32))
    dl = deltas[rng.integers(0, deltas.size, size=(nb, 32))]
    w = ((m + 0.5 + dl) * d[:, None]).astype(np.float32)
    keep = np.argmax(np.abs(base), axis=1)
    w[np.arange(nb), keep] = base[np.arange(nb), keep]
    ref = oracle.quantize(t, w.reshape(16, -1))
    assert np.array_equal(ref.reshape(nb, -1)[:, :2], oracle.quantize(t, base).reshape(nb, -1)[:, :2])   # same scales
    got = run(gpu, t, w.reshape(16, -1))
    assert np.array_equal(got, ref), f"{name}: {int((got != ref).sum())} bytes differ"


def test_quantize_bench_size_sampled_rows(gpu):
    # The bench's launch: a 14336 x 4096 fp32 matrix (235 MB, beyond L2); the
    # oracle quantizes sampled rows (blocks never straddle rows).
    t, rows, cols = qk.Q4_K, 14336, 4096
    g = torch.Generator(device=gpu)
    g.manual_seed(31337)
    w = torch.randn((rows, cols), device=gpu, generator=g) * 0.02
    got = qk.quantize(t, w)
    rb = qk.row_bytes(t, cols)
    pick = np.random.default_rng(7).choice(rows, 48, replace=False)
    pick[:2] = (0, rows - 1)
    wsel = w[torch.from_numpy(pick).to(gpu)].cpu().numpy()
    ref = oracle.quantize(t, wsel).reshape(len(pick), rb)
    got_rows = got.view(rows, rb)[torch.from_numpy(pick).to(gpu)].cpu().numpy()
    assert np.array_equal(got_rows, ref)


def test_quantize_is_deterministic_and_takes_4_byte_aligned_output(gpu):
    t, rows, cols = qk.Q8_0, 9, 160     # 45 groups: the last warp writes 13 blocks = 442 bytes
    w = synth.normal_weights(rows, cols, 5151)
    wd = torch.from_numpy(w).to(gpu)
    a = qk.quantize(t, wd).cpu().numpy()
    nb = rows * qk.row_bytes(t, cols)
    buf = torch.full((nb + 8,), 0xAB, dtype=torch.uint8, device=gpu)
    qk.quantize(t, wd, out=buf[4:4 + nb])
    b = buf.cpu().numpy()
    assert np.array_equal(a, b[4:4 + nb])
    assert np.all(b[:4] == 0xAB) and np.all(b[4 + nb:] == 0xAB)   # nothing written outside
    assert np.array_equal(a, oracle.quantize(t, w))


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
@pytest.mark.parametrize("rows,cols", [(3, 512), (33, 2048)])
def test_quantize_imatrix_matches_oracle(gpu, name, rows, cols):
    # Bytes identical to the oracle's importance-weighted quantizer, with
    # heavy-tailed importances, a run of zero-importance columns and one
    # dominant column.
    t = type_id(name)
    w = synth.normal_weights(rows, cols, 610 + t)
    g = np.random.default_rng(611 + t)
    imp = (g.standard_normal(cols) ** 2 * np.exp(2.0 * g.standard_normal(cols))).astype(np.float32)
    imp[40:72] = 0.0
    imp[100] = 1e4
    ref = oracle.quantize_imatrix(t, w, imp)
    got = qk.quantize_imatrix(t, torch.from_numpy(w).to(gpu), torch.from_numpy(imp).to(gpu)).cpu().numpy()
    qk.device_status()
    assert np.array_equal(got, ref), f"{name}: {int((got != ref).sum())} bytes differ"
    # All-zero importances: the plain quantizer's bytes.
    z = qk.quantize_imatrix(t, torch.from_numpy(w).to(gpu), torch.zeros(cols, device=gpu)).cpu().numpy()
    assert np.array_equal(z, oracle.quantize(t, w))


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
def test_quantize_imatrix_special_values(gpu, name):
    # The special-value blocks (zero divisors, fp16 subnormal and overflowing
    # scales, exact ties, NaN, infinities, negative zero) through the
    # importance-weighted search, with positive importances.
    t = type_id(name)
    n = 256 if name in ("Q4_K", "Q6_K", "Q5_K", "Q2_K", "Q3_K") else 32
    w = np.tile(special_blocks(n), (1, 8))
    imp = np.random.default_rng(8181).uniform(0.1, 4.0, w.shape[1]).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        ref = oracle.quantize_imatrix(t, w, imp)
    got = qk.quantize_imatrix(t, torch.from_numpy(w).to(gpu), torch.from_numpy(imp).to(gpu)).cpu().numpy()
    qk.device_status()
    assert np.array_equal(got, ref), f"{name}: {int((got != ref).sum())} bytes differ"


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0"])
def test_quantize_imatrix_bench_size_sampled_rows(gpu, name):
    # The bench's importance-weighted launch (14336 x 4096, N(0, 0.02) weights,
    # log-normal importances); the oracle quantizes 24 sampled rows.
    t, rows, cols = type_id(name), 14336, 4096
    g = torch.Generator(device=gpu)
    g.manual_seed(4242)
    w = torch.randn((rows, cols), device=gpu, generator=g) * 0.02
    imp = torch.exp(torch.randn(cols, device=gpu, generator=g))
    got = qk.quantize_imatrix(t, w, imp)
    qk.device_status()
    rb = qk.row_bytes(t, cols)
    pick = np.random.default_rng(8).choice(rows, 24, replace=False)
    pick[:2] = (0, rows - 1)
    sel = torch.from_numpy(pick).to(gpu)
    ref = oracle.quantize_imatrix(t, w[sel].cpu().numpy(), imp.cpu().numpy()).reshape(len(pick), rb)
    assert np.array_equal(got.view(rows, rb)[sel].cpu().numpy(), ref)


@pytest.mark.parametrize("name", ["Q4_K", "Q8_0"])
def test_quantize_imatrix_takes_4_byte_aligned_importances(gpu, name):
    # imp one float past a 16-byte boundary (the contract asks 4 bytes): the
    # same bytes as the oracle.
    t, rows, cols = type_id(name), 5, 512
    w = synth.normal_weights(rows, cols, 9191)
    imp = np.random.default_rng(9192).uniform(0.05, 3.0, cols).astype(np.float32)
    buf = torch.zeros(cols + 4, device=gpu)
    buf[1:1 + cols] = torch.from_numpy(imp).to(gpu)
    got = qk.quantize_imatrix(t, torch.from_numpy(w).to(gpu), buf[1:1 + cols]).cpu().numpy()
    qk.device_status()
    assert np.array_equal(got, oracle.quantize_imatrix(t, w, imp))


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q3_K"])
def test_quantize_persistent_grid_ragged_tail(gpu, name):
    # 1201 x 2304: 86,472 groups = 2,702 tiles of 32 groups and a last tile of 8,
    # more tiles than the persistent grid's warps, so warps take several tiles
    # and one of them the ragged tail.
    t = type_id(name)
    w = synth.normal_weights(1201, 2304, 9393)
    got = run(gpu, t, w)
    assert np.array_equal(got, oracle.quantize(t, w))
