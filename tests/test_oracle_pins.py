"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one part of the oracle to something other than itself: a
size or a formula the pages print, a hand-packed block with hand-derived
weights (tests/golden/), a library routine (numpy / torch conversions,
numpy's float64 matmul), an exact-integer special case or a bijection.
"""
import numpy as np
import pytest
import torch

import synth
from golden_io import all_fixtures, load

pytestmark = pytest.mark.filterwarnings("ignore")

T = {"Q4_K": 1, "Q6_K": 2, "Q8_0": 3, "Q5_0": 4, "Q4_0": 5, "Q5_K": 6, "Q2_K": 7, "Q3_K": 8}


# ---------------------------------------------------------------- sizes --

def test_block_sizes_and_bits_per_weight(oracle_mod):
    o = oracle_mod
    # "Hitchhiker's Guide", 11.2 / "12 -- llama.cpp / GGUF", bit layout:
    # 256 weights -> 144 bytes = 4.5 bits per weight.
    assert o.block_bytes(T["Q4_K"]) == 144 and o.block_elems(T["Q4_K"]) == 256
    assert o.block_bytes(T["Q4_K"]) * 8 / 256 == 4.5
    # "Hitchhiker's Guide", 11.1: Q4_0, 32 weights -> 18 bytes = 4.5 bits/weight.
    assert o.block_bytes(T["Q4_0"]) == 18 and o.block_bytes(T["Q4_0"]) * 8 / 32 == 4.5
    # "12 -- llama.cpp / GGUF", k-quants table: Q6_K at 6.6 bits/weight.
    bpw6 = o.block_bytes(T["Q6_K"]) * 8 / o.block_elems(T["Q6_K"])
    assert bpw6 == 6.5625 and round(bpw6, 1) == 6.6
    # Q8_0: fp16 d + 32 int8 = 34 B; Q5_0: fp16 d + 4 B + 16 B = 22 B.
    assert o.block_bytes(T["Q8_0"]) == 34 and o.block_elems(T["Q8_0"]) == 32
    assert o.block_bytes(T["Q5_0"]) == 22 and o.block_elems(T["Q5_0"]) == 32
    # "12 -- llama.cpp / GGUF", k-quants table: Q5_K at 5.5-5.7 bits/weight on
    # 256-weight super-blocks; the reading's 176 bytes is the low end.
    assert o.block_bytes(T["Q5_K"]) == 176 and o.block_elems(T["Q5_K"]) == 256
    assert o.block_bytes(T["Q5_K"]) * 8 / 256 == 5.5
    # The same table: Q2_K at 2.5-2.6 and Q3_K at 3.4-4.0 bits/weight, both on
    # 256-weight super-blocks; the readings' 84 and 110 bytes.
    bpw2 = o.block_bytes(T["Q2_K"]) * 8 / o.block_elems(T["Q2_K"])
    bpw3 = o.block_bytes(T["Q3_K"]) * 8 / o.block_elems(T["Q3_K"])
    assert o.block_elems(T["Q2_K"]) == o.block_elems(T["Q3_K"]) == 256
    assert bpw2 == 2.625 and 2.5 <= round(bpw2, 1) <= 2.6
    assert bpw3 == 3.4375 and 3.4 <= bpw3 <= 4.0
    # Row bytes: cols / elems * block bytes (the workload's 9,030-byte rows).
    assert o.row_bytes(T["Q6_K"], 11008) == 9030
    assert o.row_bytes(T["Q4_K"], 1024) * 256 == 147456


# ---------------------------------------------------- number formats --

def test_half_decode_exhaustive(oracle_mod):
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle_mod.half_to_float(int(v)) for v in h], np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_half_encode_matches_numpy(oracle_mod):
    g = synth.rng(7)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 5, 4000),
        np.arange(-2048, 2049, dtype=np.float32) * np.float32(2.0 ** -25),  # subnormal ties
        np.array([65504, 65519.99, 65520, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.0, -0.0], np.float32)])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch(oracle_mod):
    g = synth.rng(8)
    bits = g.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # exact ties
    vals = np.concatenate([vals, ties, -ties, np.array([0.0, -0.0, 3.4e38, 1e-40], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.float_to_bf16_array(vals)
    assert np.array_equal(got, ref)
    back = np.array([oracle_mod.bf16_to_float(int(b)) for b in ref[:100]], np.float32)
    assert np.array_equal(back, torch.from_numpy(ref[:100].view(np.int16)).view(torch.bfloat16).float().numpy())


# -------------------------------------------------- golden fixtures --

@pytest.mark.parametrize("path", all_fixtures(), ids=lambda p: p.rsplit("/", 1)[-1])
def test_golden_block(oracle_mod, path):
    name, blk, expect = load(path)
    t = T[name]
    assert blk.size == oracle_mod.block_bytes(t)
    w = oracle_mod.dequant(t, blk, 1, oracle_mod.block_elems(t))[0]
    assert np.array_equal(w.astype(np.float64), expect), np.nonzero(w != expect)


# --------------------------------------- nibble order: the Q4_0 routine --

def _q4_0_as_printed(blocks: np.ndarray) -> np.ndarray:
    """Q4_0 dequantization as "How LLM Inference Engines Work" ("Loading GGUF
    Models") describes it: per 18-byte block an fp16 scale, then 16 bytes
    whose low nibbles, minus 8, are the first 16 values and whose high
    nibbles, minus 8, the last 16; everything times the scale."""
    b = blocks.reshape(-1, 18)
    scale = b[:, :2].copy().view(np.float16).astype(np.float32)
    nib = b[:, 2:]
    first = (nib & 15).astype(np.float32) - 8
    second = (nib >> 4).astype(np.float32) - 8
    return (np.concatenate([first, second], axis=1) * scale).reshape(-1)


def test_q4_0_nibble_order_matches_page_routine(oracle_mod):
    W = synth.rng(3).integers(0, 256, (64, 18), dtype=np.uint8)
    W[:, :2] = (np.abs(synth.rng(4).standard_normal(64)) * 0.01).astype(np.float16).view(np.uint8).reshape(64, 2)
    got = oracle_mod.dequant(T["Q4_0"], W.reshape(-1), 64, 32).reshape(-1)
    assert np.array_equal(got, _q4_0_as_printed(W.reshape(-1)))


def test_q5_0_low_nibbles_follow_q4_0_convention(oracle_mod):
    # With every fifth bit clear, Q5_0 codes equal the Q4_0 codes of the same
    # nibble bytes, so w_Q5_0 + 16d == w_Q4_0 + 8d element by element.
    g = synth.rng(5)
    nib = g.integers(0, 256, (32, 16), dtype=np.uint8)
    d = np.full((32, 2), [0, 0x3C], np.uint8)  # d = 1.0
    q5 = np.concatenate([d, np.zeros((32, 4), np.uint8), nib], axis=1).reshape(-1)
    q4 = np.concatenate([d, nib], axis=1).reshape(-1)
    w5 = oracle_mod.dequant(T["Q5_0"], q5, 32, 32)
    w4 = oracle_mod.dequant(T["Q4_0"], q4, 32, 32)
    assert np.array_equal(w5 + 16, w4 + 8)


# ------------------------------------------------------ round trips --

@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
def test_bytes_unpack_pack_bijection(oracle_mod, name):
    # Every byte of these blocks is used, so unpack followed by pack must give
    # back the same bytes (and unpack of that, the same fields).
    t = T[name]
    bb, nb = oracle_mod.block_bytes(t), 200
    W = synth.rng(11).integers(0, 256, nb * bb, dtype=np.uint8)
    codes, sc, mins, d, dmin = oracle_mod.unpack(t, W, nb)
    dbits = np.array([oracle_mod.float_to_half(float(v)) for v in d], np.uint16)
    dminbits = np.array([oracle_mod.float_to_half(float(v)) for v in dmin], np.uint16)
    # fp16 NaN payloads do not survive a float round trip; restore raw bits.
    off = {"Q4_K": 0, "Q6_K": 208, "Q8_0": 0, "Q5_0": 0, "Q4_0": 0, "Q5_K": 0, "Q2_K": 80, "Q3_K": 108}[name]
    raw_d = W.reshape(nb, bb)[:, off:off + 2].copy().view(np.uint16).reshape(nb)
    dbits = raw_d
    if name in ("Q4_K", "Q5_K"):
        dminbits = W.reshape(nb, bb)[:, 2:4].copy().view(np.uint16).reshape(nb)
    if name == "Q2_K":
        dminbits = W.reshape(nb, bb)[:, 82:84].copy().view(np.uint16).reshape(nb)
    again = oracle_mod.pack(t, codes, sc, mins, dbits, dminbits)
    assert np.array_equal(again, W)


def test_q4k_every_6bit_value_in_every_slot(oracle_mod):
    # 64 values x 8 scale slots and 64 x 8 min slots, others random.
    g = synth.rng(12)
    nb = 64 * 8
    sc = np.zeros((nb, 16), np.int16)
    mn = np.zeros((nb, 16), np.uint8)   # 8 used
    sc[:, :8] = g.integers(0, 64, (nb, 8))
    mn[:, :8] = g.integers(0, 64, (nb, 8))
    for i in range(nb):
        v, slot = i % 64, i // 64
        sc[i, slot] = v
        mn[i, 7 - slot] = 63 - v
    codes = g.integers(0, 16, (nb, 256)).astype(np.int16)
    W = oracle_mod.pack(1, codes, sc, mn, np.full(nb, 0x3C00, np.uint16), np.full(nb, 0x3C00, np.uint16))
    c2, sc2, mn2, d, dmin = oracle_mod.unpack(1, W, nb)
    assert np.array_equal(c2, codes) and np.array_equal(sc2, sc) and np.array_equal(mn2, mn)
    assert np.all(d == 1.0) and np.all(dmin == 1.0)


def test_q6k_q8_q5_code_ranges_round_trip(oracle_mod):
    g = synth.rng(13)
    for name, lo, hi, be in (("Q6_K", 0, 64, 256), ("Q8_0", -128, 128, 32), ("Q5_0", 0, 32, 32)):
        nb = 128
        codes = g.integers(lo, hi, (nb, be)).astype(np.int16)
        codes[0, :hi - lo if hi - lo <= be else be] = np.arange(lo, lo + min(hi - lo, be))
        sc = np.zeros((nb, 16), np.int16)
        if name == "Q6_K":
            sc[:] = g.integers(-128, 128, (nb, 16))
            sc[1, :] = [-128, 127] * 8
        W = oracle_mod.pack(T[name], codes, sc, None, np.full(nb, 0x3800, np.uint16))
        c2, sc2, _, d, _ = oracle_mod.unpack(T[name], W, nb)
        assert np.array_equal(c2, codes)
        if name == "Q6_K":
            assert np.array_equal(sc2, sc)
        assert np.all(d == 0.5)


def test_q5k_is_q4k_plus_a_fifth_bit(oracle_mod):
    # Q5_K (a reading of the GGUF layout; the pages give only its size) is
    # Q4_K's super-block with a 32-byte high-bit plane inserted after the
    # scales.  With every high bit clear it must decode exactly as the Q4_K
    # block holding the same d, dmin, scale bytes and code bytes (a path
    # pinned by the pages' Q4_K figures), and with every high bit set each
    # code grows by exactly 16.  A wrong offset of qs, of the scales or of the
    # plane, or a high bit added at the wrong weight, breaks one of the two.
    nb = 64
    W4 = synth.random_blocks("Q4_K", 1, 256 * nb, 31).reshape(nb, 144)
    for fill, shift in ((0x00, 0), (0xFF, 16)):
        W5 = np.zeros((nb, 176), np.uint8)
        W5[:, :16] = W4[:, :16]
        W5[:, 16:48] = fill
        W5[:, 48:] = W4[:, 16:]
        c4, sc4, m4, d4, dm4 = oracle_mod.unpack(1, W4.reshape(-1), nb)
        c5, sc5, m5, d5, dm5 = oracle_mod.unpack(6, W5.reshape(-1), nb)
        assert np.array_equal(c5, c4 + shift)
        assert np.array_equal(sc5, sc4) and np.array_equal(m5, m4)
        assert np.array_equal(d5, d4) and np.array_equal(dm5, dm4)
        if shift == 0:
            assert np.array_equal(oracle_mod.dequant(6, W5.reshape(-1), 1, 256 * nb),
                                  oracle_mod.dequant(1, W4.reshape(-1), 1, 256 * nb))


def test_q5k_high_bit_planes_select_their_weights(oracle_mod):
    # One high bit at a time: bit b of qh[l] must raise exactly one code by
    # 16 (and no other), and over all 256 (byte, bit) pairs each code is
    # raised exactly once -- the plane is a bijection onto the weights, in
    # the same low-half / high-half order as the nibbles of each 64-weight
    # group (bit 2c + h of qh[l] belongs to the weight whose low nibble is
    # half h of qs[32c + l]).
    base = np.zeros((256, 176), np.uint8)
    base[:, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    hit = np.zeros(256, int)
    for k in range(256):
        l, b = k // 8, k % 8
        base[k, 16 + l] = 1 << b
    codes, _, _, _, _ = oracle_mod.unpack(6, base.reshape(-1), 256)
    for k in range(256):
        l, b = k // 8, k % 8
        (raised,) = np.nonzero(codes[k])
        assert raised.size == 1 and codes[k, raised[0]] == 16
        n = raised[0]
        hit[n] += 1
        # its low nibble lives in qs[32 (n // 64) + n % 32], half (n // 32) % 2
        assert n % 32 == l and 2 * (n // 64) + (n // 32) % 2 == b
    assert np.all(hit == 1)


def _one_bit_blocks(nbytes_total, plane_off, plane_len, bits):
    """Blocks with a single set bit each: one per (byte of the plane, bit)."""
    blocks = np.zeros((plane_len * len(bits), nbytes_total), np.uint8)
    for k in range(plane_len):
        for i, b in enumerate(bits):
            blocks[k * len(bits) + i, plane_off + k] = 1 << b
    return blocks


def test_q2k_code_pairs_are_a_bijection_onto_the_weights(oracle_mod):
    # Q2_K (a reading; the pages give only its size): every 2-bit field of the
    # 64 code bytes must be the code of exactly one weight, all 256 covered.
    # A field set to 1 in an otherwise zero block raises exactly one code to 1.
    B = np.zeros((256, 84), np.uint8)
    for k in range(64):
        for j in range(4):
            B[4 * k + j, 16 + k] = 1 << (2 * j)
    codes, _, _, _, _ = oracle_mod.unpack(7, B.reshape(-1), 256)
    hit = np.zeros(256, int)
    for e in range(256):
        (n,) = np.nonzero(codes[e])
        assert n.size == 1 and codes[e, n[0]] == 1
        hit[n[0]] += 1
        k, j = e // 4, e % 4
        # byte 32t + l, field j: weight 128t + 32j + l
        assert n[0] == 128 * (k // 32) + 32 * j + k % 32
    assert np.all(hit == 1)


def test_q3k_mask_and_code_planes(oracle_mod):
    # Q3_K (a reading): with every mask bit clear a code is its 2-bit field
    # minus 4 (all codes -4 on a zero block); each of the 256 mask bits lifts
    # exactly one weight by 4, and each 2-bit field set to 1 raises exactly
    # one code by 1 -- both bijections onto the weights, matching each other.
    zero = np.zeros(110, np.uint8)
    c0, _, _, _, _ = oracle_mod.unpack(8, zero, 1)
    assert np.all(c0 == -4)
    M = _one_bit_blocks(110, 0, 32, range(8))
    cm, _, _, _, _ = oracle_mod.unpack(8, M.reshape(-1), 256)
    Q = np.zeros((256, 110), np.uint8)
    for k in range(64):
        for j in range(4):
            Q[4 * k + j, 32 + k] = 1 << (2 * j)
    cq, _, _, _, _ = oracle_mod.unpack(8, Q.reshape(-1), 256)
    hm = np.zeros(256, int)
    hq = np.zeros(256, int)
    for e in range(256):
        (nm,) = np.nonzero(cm[e] + 4)
        (nq,) = np.nonzero(cq[e] + 4)
        assert nm.size == 1 and cm[e, nm[0]] == 0
        assert nq.size == 1 and cq[e, nq[0]] == -3
        hm[nm[0]] += 1
        hq[nq[0]] += 1
        # mask byte l, bit 4t + j and code byte 32t + l, field j: weight 128t + 32j + l
        l, bit = e // 8, e % 8
        assert nm[0] == 128 * (bit // 4) + 32 * (bit % 4) + l
    assert np.all(hm == 1) and np.all(hq == 1)


@pytest.mark.parametrize("name", ["Q2_K", "Q3_K"])
def test_group_scales_follow_weight_order(oracle_mod, name):
    # Sixteen distinct scales and all codes equal: the weights step through
    # the scales in group order, 16 weights each (pairs each scale field with
    # its 16 weights: a wrong group index or a wrong scale unpacking moves a
    # weight to another scale).
    t = T[name]
    sc = np.arange(16, dtype=np.int16)[None, :] + (0 if name == "Q2_K" else -8)
    codes = np.full((1, 256), 1, np.int16)
    W = oracle_mod.pack(t, codes, sc, None, np.array([0x3C00], np.uint16), np.array([0], np.uint16))
    w = oracle_mod.dequant(t, W, 1, 256)[0]
    assert np.array_equal(w, np.repeat(sc[0].astype(np.float32), 16))


# --------------------------------------------- dequant formula checks --

def test_q4k_formula_exact_in_fp32(oracle_mod):
    # d*sc and dmin*m are exact products in fp32 (11 + 6 significant bits), so
    # is (d*sc)*q (+ 4 bits); only the final subtraction rounds.  Hence the
    # oracle's weight equals fl(fl64((d*sc)*q) - fl64(dmin*m)) computed in fp64.
    W = synth.random_blocks("Q4_K", 8, 2048, 21)
    codes, sc, mins, d, dmin = oracle_mod.unpack(1, W, 64)
    ds = d[:, None].astype(np.float64) * sc[:, :8].astype(np.float64)
    dm = dmin[:, None].astype(np.float64) * mins.astype(np.float64)
    sub = np.repeat(np.arange(8), 32)
    exact = ds[:, sub] * codes.astype(np.float64) - dm[:, sub]
    got = oracle_mod.dequant(1, W, 8, 2048).reshape(64, 256)
    assert np.array_equal(got, exact.astype(np.float32))


def test_q5k_formula_exact_in_fp32(oracle_mod):
    # As for Q4_K: d*sc (11 + 6 bits) times a 5-bit code stays within 24 bits,
    # so only the final subtraction rounds.
    W = synth.random_blocks("Q5_K", 8, 2048, 22)
    codes, sc, mins, d, dmin = oracle_mod.unpack(6, W, 64)
    ds = d[:, None].astype(np.float64) * sc[:, :8].astype(np.float64)
    dm = dmin[:, None].astype(np.float64) * mins.astype(np.float64)
    sub = np.repeat(np.arange(8), 32)
    exact = ds[:, sub] * codes.astype(np.float64) - dm[:, sub]
    got = oracle_mod.dequant(6, W, 8, 2048).reshape(64, 256)
    assert np.array_equal(got, exact.astype(np.float32))
    assert codes.min() == 0 and codes.max() == 31


@pytest.mark.parametrize("name", ["Q2_K", "Q3_K"])
def test_q2k_q3k_formula_exact_in_fp32(oracle_mod, name):
    # d*sc (11 + 6 bits) times a code of at most 3 bits and dmin*m stay
    # within 24 bits: only Q2_K's final subtraction rounds.
    t = T[name]
    W = synth.random_blocks(name, 8, 2048, 23)
    codes, sc, mins, d, dmin = oracle_mod.unpack(t, W, 64)
    grp = np.repeat(np.arange(16), 16)
    ds = d[:, None].astype(np.float64) * sc.astype(np.float64)
    dm = dmin[:, None].astype(np.float64) * mins.astype(np.float64)
    exact = ds[:, grp] * codes.astype(np.float64) - dm[:, grp]
    got = oracle_mod.dequant(t, W, 8, 2048).reshape(64, 256)
    assert np.array_equal(got, exact.astype(np.float32))


def test_zero_scale_block_is_zero(oracle_mod):
    for name in ("Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q5_K", "Q2_K", "Q3_K"):
        W = synth.random_blocks(name, 2, 512, 22)
        bb, be, doff, dmoff = synth.GEOMETRY[name]
        B = W.reshape(-1, bb)
        B[:, doff:doff + 2] = 0
        if dmoff is not None:
            B[:, dmoff:dmoff + 2] = 0
        w = oracle_mod.dequant(T[name], W, 2, 512)
        assert np.all(w == 0)


# ------------------------------------------------------ dot products --

@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
@pytest.mark.parametrize("rows,cols,M", [(1, 256, 1), (3, 512, 2), (4, 1024, 3)])
def test_gemv_matches_numpy_float64_matmul(oracle_mod, name, rows, cols, M):
    t = T[name]
    W = synth.random_blocks(name, rows, cols, 30 + rows)
    x = synth.activations(M, cols, 31)
    y, S = oracle_mod.gemv(t, W, rows, cols, x)
    w = oracle_mod.dequant(t, W, rows, cols).astype(np.float64)
    ref = x.astype(np.float64) @ w.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(S, np.abs(x.astype(np.float64)) @ np.abs(w).T, rtol=1e-12)
    assert np.all(S >= np.abs(y) - 1e-12)


def test_gemv_exact_integer_case(oracle_mod):
    # Q8_0 with d = 2^-3 and small-integer x: every product and partial sum is
    # an exact binary fraction, so y equals (codes . x) * 2^-3 exactly, with
    # the codes taken from the generator, not from the unpacker.
    g = synth.rng(40)
    rows, cols = 5, 256
    codes = g.integers(-128, 128, (rows * cols // 32, 32)).astype(np.int16)
    W = oracle_mod.pack(3, codes, None, None, np.full(rows * cols // 32, 0x3000, np.uint16))
    x = g.integers(-8, 9, (2, cols)).astype(np.float32)
    y, _ = oracle_mod.gemv(3, W, rows, cols, x)
    expect = (x.astype(np.int64) @ codes.reshape(rows, cols).astype(np.int64).T) * 0.125
    assert np.array_equal(y, expect)


def test_gemm_bf16_is_gemv_on_rounded_activations(oracle_mod):
    name, rows, cols, M = "Q4_K", 6, 512, 3
    W = synth.random_blocks(name, rows, cols, 50)
    Xb = synth.activations_bf16_bits(M, cols, 51)
    Y, S = oracle_mod.gemm_bf16(1, W, rows, cols, Xb)
    xf = torch.from_numpy(Xb.view(np.int16)).view(torch.bfloat16).float().numpy()
    y2, S2 = oracle_mod.gemv(1, W, rows, cols, xf)
    assert np.array_equal(Y, y2) and np.array_equal(S, S2)


def test_entries_equal_full_products(oracle_mod):
    name, rows, cols, M = "Q6_K", 9, 768, 4
    W = synth.random_blocks(name, rows, cols, 60)
    x = synth.activations(M, cols, 61)
    Xb = synth.activations_bf16_bits(M, cols, 62)
    y, S = oracle_mod.gemv(2, W, rows, cols, x)
    Y, SY = oracle_mod.gemm_bf16(2, W, rows, cols, Xb)
    mi = np.array([0, 3, 2, 1, 3]); ni = np.array([8, 0, 4, 4, 7])
    ye, Se = oracle_mod.entries(2, W, rows, cols, mi, ni, x=x)
    Ye, SYe = oracle_mod.entries(2, W, rows, cols, mi, ni, X_bits=Xb)
    assert np.array_equal(ye, y[mi, ni]) and np.array_equal(Se, S[mi, ni])
    assert np.array_equal(Ye, Y[mi, ni]) and np.array_equal(SYe, SY[mi, ni])


# -------------------------------------------------------- quantizer --

def test_quantizer_error_bounds(oracle_mod):
    w = synth.normal_weights(16, 1024, 70)
    # Q8_0: |w - wq| <= d/2 per block (the max element maps to +-127 exactly
    # up to the fp16 rounding of d, which moves it by less than half a step).
    W = oracle_mod.quantize(3, w)
    dq = oracle_mod.dequant(3, W, 16, 1024)
    _, _, _, d, _ = oracle_mod.unpack(3, W, 16 * 32)
    err = np.abs(dq - w).reshape(-1, 32).max(axis=1)
    assert np.all(err <= 0.5 * d * 1.01 + 1e-9)
    # Q4_K: every weight within one code step (d*sc) of the input plus the
    # min's rounding (dmin/2).
    W = oracle_mod.quantize(1, w)
    dq = oracle_mod.dequant(1, W, 16, 1024)
    codes, sc, mins, d, dmin = oracle_mod.unpack(1, W, 64)
    step = (d[:, None] * sc[:, :8]).repeat(32, axis=1).reshape(-1)
    bound = step + np.repeat(dmin, 256) * 0.5 + 1e-6
    assert np.all(np.abs(dq.reshape(-1) - w.reshape(-1)) <= bound)


def _codes(oracle_mod, t, W, nblocks):
    return oracle_mod.unpack(t, W, nblocks)


def test_quantizer_exact_codes_on_dyadic_grids(oracle_mod):
    # Values on the grid d*(q - off) with the extreme code present give a
    # scale d = max|w| / (top code) that is exact in fp16, so every code is
    # recovered exactly: pins the divisor, the offset and the sign.
    rng = np.random.default_rng(91)
    for t, top, off, d_true, lo_q, hi_q in ((3, 127, 0, 2.0 ** -7, -127, 127),   # Q8_0
                                            (4, 15, 16, 2.0 ** -4, 1, 31),       # Q5_0
                                            (5, 7, 8, 2.0 ** -3, 1, 15)):        # Q4_0
        q = rng.integers(lo_q, hi_q + 1, size=(4, 32))
        q[:, 0] = hi_q
        q[:, 1] = lo_q
        w = ((q - off) * d_true).astype(np.float32)
        W = oracle_mod.quantize(t, w.reshape(1, -1))
        codes, _, _, d, _ = _codes(oracle_mod, t, W, 4)
        assert np.all(d == d_true)
        assert np.array_equal(codes[:, :32], q)


def test_quantizer_exact_codes_k_quants(oracle_mod):
    # Q4_K: every sub-block spans [lo, hi] with lo < 0 in 15 equal steps, so
    # sc = m = 63 and the code is the step count (the fp16 rounding of d and
    # dmin moves (w + dmin*m) / (d*sc) by < 0.01).  Pins the sign of the min
    # term, the 6-bit scale packing and the nibble order.
    rng = np.random.default_rng(92)
    lo, hi = -0.37, 0.81
    k = rng.integers(0, 16, size=256)
    k[::32] = 0
    k[1::32] = 15
    w = (lo + k * (hi - lo) / 15.0).astype(np.float32)
    W = oracle_mod.quantize(1, w.reshape(1, -1))
    codes, sc, mins, d, dmin = _codes(oracle_mod, 1, W, 1)
    assert np.array_equal(codes[0], k)
    assert np.all(sc[0, :8] == 63) and np.all(mins[0, :8] == 63)
    # Q6_K: each 16-group has max |w| = A, values A*k/32 for k in -32..31:
    # sc = 127 and the code is k + 32.
    A = 0.23
    k6 = rng.integers(-32, 32, size=256)
    k6[::16] = -32
    w6 = (A * k6 / 32.0).astype(np.float32)
    W6 = oracle_mod.quantize(2, w6.reshape(1, -1))
    c6, s6, _, _, _ = _codes(oracle_mod, 2, W6, 1)
    assert np.array_equal(c6[0], k6 + 32)
    assert np.all(s6[0, :16] == 127)
    # Q5_K: the Q4_K construction with 31 steps; codes 0..31 come back.
    k5 = rng.integers(0, 32, size=256)
    k5[::32] = 0
    k5[1::32] = 31
    w5 = (lo + k5 * (hi - lo) / 31.0).astype(np.float32)
    W5 = oracle_mod.quantize(6, w5.reshape(1, -1))
    c5, s5, m5, _, _ = _codes(oracle_mod, 6, W5, 1)
    assert np.array_equal(c5[0], k5)
    assert np.all(s5[0, :8] == 63) and np.all(m5[0, :8] == 63)
    # Q2_K: each 16-group spans [lo, hi] in 3 steps: sc = m = 15, code = step.
    k2 = rng.integers(0, 4, size=256)
    k2[::16] = 0
    k2[1::16] = 3
    w2 = (lo + k2 * (hi - lo) / 3.0).astype(np.float32)
    c2, s2, m2, _, _ = _codes(oracle_mod, 7, oracle_mod.quantize(7, w2.reshape(1, -1)), 1)
    assert np.array_equal(c2[0], k2)
    assert np.all(s2[0] == 15) and np.all(m2[0] == 15)
    # Q3_K: each 16-group has max |w| = A at code -4, values A*k/4 for k in
    # -4..3: sc = 31 and the code is k.
    k3 = rng.integers(-4, 4, size=256)
    k3[::16] = -4
    w3 = (A * k3 / 4.0).astype(np.float32)
    c3, s3, _, _, _ = _codes(oracle_mod, 8, oracle_mod.quantize(8, w3.reshape(1, -1)), 1)
    assert np.array_equal(c3[0], k3)
    assert np.all(s3[0] == 31)


def test_quantizer_zero_blocks(oracle_mod):
    # An all-zero block takes the zero-divisor path: d = 0 and the offset code.
    for t, n, code in ((1, 256, 0), (2, 256, 32), (3, 32, 0), (4, 32, 16), (5, 32, 8), (6, 256, 0), (7, 256, 0),
                       (8, 256, 0)):
        W = oracle_mod.quantize(t, np.zeros((1, n), np.float32))
        codes, sc, mins, d, dmin = _codes(oracle_mod, t, W, 1)
        assert np.all(codes[0, :n] == code) and d[0] == 0.0
        if t == 1:
            assert dmin[0] == 0.0 and not sc.any() and not mins.any()


# ------------------------------------------------------------ SwiGLU --

def test_silu_against_the_logistic_function(oracle_mod):
    # SiLU(z) = z * sigmoid(z); sigmoid from scipy's expit (a library routine).
    special = pytest.importorskip("scipy.special")
    z = np.concatenate([np.linspace(-40.0, 40.0, 4001), [-1e3, -745.5, 0.0, 1e-300, 745.5, 1e3]])
    s = oracle_mod.silu(z)
    ref = z * special.expit(z)
    assert np.allclose(s, ref, rtol=4e-16, atol=1e-300)
    assert s[z == 0.0][0] == 0.0 and s[-1] == 1e3 and s[z == -1e3][0] == 0.0   # e^1000 overflows: -0


def test_silu_reflection_identity(oracle_mod):
    # SiLU(-z) = -z (1 - sigmoid(z)) = SiLU(z) - z.
    z = np.linspace(-30.0, 30.0, 601)
    assert np.allclose(oracle_mod.silu(-z), oracle_mod.silu(z) - z, rtol=1e-14, atol=1e-13)


def test_swiglu_on_an_exact_block(oracle_mod):
    # Q8_0 with d = 1 (fp16 0x3C00): w = q exactly, so g and u are exact
    # integer dot products; h = SiLU(g) * u from the closed form.
    rng = np.random.default_rng(93)
    rows, cols = 3, 64
    def mat(seed):
        q = np.random.default_rng(seed).integers(-5, 6, size=(rows, cols))
        blk = np.zeros((rows, cols // 32, 34), np.uint8)
        blk[:, :, 0], blk[:, :, 1] = 0x00, 0x3C
        blk[:, :, 2:] = q.reshape(rows, cols // 32, 32).astype(np.int8).view(np.uint8)
        return blk.reshape(-1), q
    (Wg, qg), (Wu, qu) = mat(1), mat(2)
    x = rng.integers(-3, 4, size=cols).astype(np.float32)
    h, g, u, _, _ = oracle_mod.swiglu(3, Wg, Wu, rows, cols, x)
    ge, ue = qg @ x.astype(np.float64), qu @ x.astype(np.float64)
    assert np.array_equal(g, ge) and np.array_equal(u, ue)
    assert np.allclose(h, ge / (1.0 + np.exp(-ge)) * ue, rtol=0, atol=0)


# ------------------------------------------- importance-weighted quantizer --
# "Hitchhiker's Guide -- Lab 01", 11.3: minimise sum_i E[x_i^2] (w_i - w^_i)^2.

def _heavy_importances(cols, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal(cols) ** 2 * np.exp(2.0 * g.standard_normal(cols))).astype(np.float32)


def _block_errors(oracle_mod, t, W, w, imp):
    rows, cols = w.shape
    be = oracle_mod.block_elems(t)
    dq = oracle_mod.dequant(t, W, rows, cols).astype(np.float64)
    e = (dq - w.astype(np.float64)) ** 2 * imp.astype(np.float64)[None, :]
    return e.reshape(rows, cols // be, be).sum(axis=2)


@pytest.mark.parametrize("name", ["Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"])
def test_imatrix_never_worse_and_clearly_better(oracle_mod, name):
    # Per block, the weighted error never exceeds the plain quantizer's (the
    # plain block is the fall-back); over the matrix, with heavy-tailed
    # importances, it is clearly lower (a no-op search would fail this).
    t = T[name]
    w = synth.normal_weights(12, 1024, 501)
    imp = _heavy_importances(1024, 502)
    Wp = oracle_mod.quantize(t, w)
    Wi = oracle_mod.quantize_imatrix(t, w, imp)
    ep = _block_errors(oracle_mod, t, Wp, w, imp)
    ei = _block_errors(oracle_mod, t, Wi, w, imp)
    assert np.all(ei <= ep * (1 + 1e-5) + 1e-30)
    assert ei.sum() < 0.8 * ep.sum()


def test_imatrix_degenerate_importances(oracle_mod):
    w = synth.normal_weights(4, 512, 503)
    for name, t in T.items():
        # All-zero importance: no refit is possible, the plain bytes come back.
        assert np.array_equal(oracle_mod.quantize_imatrix(t, w, np.zeros(512, np.float32)), oracle_mod.quantize(t, w))
        # Only relative importances matter: a power-of-two factor scales every
        # sum exactly, so the bytes cannot change.
        imp = _heavy_importances(512, 504)
        a = oracle_mod.quantize_imatrix(t, w, imp)
        b = oracle_mod.quantize_imatrix(t, w, imp * np.float32(8.0))
        assert np.array_equal(a, b), name


def test_imatrix_protects_the_important_column(oracle_mod):
    # One dominant column per 32-block: the symmetric 32-weight types refit
    # their scale on it, so its reconstruction error falls well below the
    # plain quantizer's on every block.
    rows, cols = 16, 1024
    w = synth.normal_weights(rows, cols, 505)
    imp = np.full(cols, 1e-6, np.float32)
    imp[5::32] = 1.0
    for t in (T["Q8_0"], T["Q5_0"], T["Q4_0"]):
        dp = oracle_mod.dequant(t, oracle_mod.quantize(t, w), rows, cols)
        di = oracle_mod.dequant(t, oracle_mod.quantize_imatrix(t, w, imp), rows, cols)
        ep = np.abs(dp - w)[:, 5::32]
        ei = np.abs(di - w)[:, 5::32]
        assert ei.mean() < 0.25 * ep.mean()


# ------------------------------------------- attention over a quantized KV cache --
# "Hitchhiker's Guide -- Lab 01", 13.2: q8_0 / q4_0 K and V read inside attention.

def _kv(name, T, nkv, d, seed):
    return (synth.random_blocks(name, T * nkv, d, seed), synth.random_blocks(name, T * nkv, d, seed + 1))


@pytest.mark.parametrize("name", ["Q8_0", "Q4_0", "Q5_0"])
def test_attn_matches_torch_sdpa(oracle_mod, name):
    # torch's scaled_dot_product_attention in fp64 on the dequantized caches
    # (an independent library routine), grouped-query heads expanded by hand.
    t = T[name]
    Tn, nh, nkv, d = 37, 8, 2, 64
    K, V = _kv(name, Tn, nkv, d, 700)
    q = synth.activations(nh, d, 702)
    out, _ = oracle_mod.attn_decode(t, q, K, V, Tn, nh, nkv, d, 0.125)
    Kd = torch.from_numpy(oracle_mod.dequant(t, K, Tn * nkv, d).reshape(Tn, nkv, d)).double()
    Vd = torch.from_numpy(oracle_mod.dequant(t, V, Tn * nkv, d).reshape(Tn, nkv, d)).double()
    grp = nh // nkv
    k = Kd.permute(1, 0, 2).repeat_interleave(grp, dim=0)     # [nh, T, d]
    v = Vd.permute(1, 0, 2).repeat_interleave(grp, dim=0)
    qq = torch.from_numpy(q).double().unsqueeze(1)             # [nh, 1, d]
    ref = torch.nn.functional.scaled_dot_product_attention(qq, k, v, scale=0.125).squeeze(1).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_attn_special_cases(oracle_mod):
    t, d, nkv = T["Q8_0"], 32, 1
    # One position: the output is that position's value row, exactly.
    K, V = _kv("Q8_0", 1, nkv, d, 710)
    q = synth.activations(2, d, 711)
    out, Sv = oracle_mod.attn_decode(t, q, K, V, 1, 2, nkv, d, 1.0)
    v0 = oracle_mod.dequant(t, V, 1, d)[0].astype(np.float64)
    assert np.array_equal(out[0], v0) and np.array_equal(out[1], v0)
    assert np.array_equal(Sv[0], np.abs(v0))
    # Identical keys: uniform attention, the output is the mean value row.
    Tn = 9
    K1, V9 = _kv("Q8_0", Tn, nkv, d, 712)
    K9 = np.tile(K1.reshape(Tn, -1)[:1], (Tn, 1)).reshape(-1)
    out, _ = oracle_mod.attn_decode(t, q, K9, V9, Tn, 2, nkv, d, 0.5)
    mean = oracle_mod.dequant(t, V9, Tn, d).astype(np.float64).mean(axis=0)
    assert np.allclose(out, mean[None, :], rtol=1e-13, atol=1e-13)
    # Grouped heads: equal queries in one group give equal outputs; the
    # other group reads other rows.
    Tn, nh, nkv = 11, 4, 2
    K, V = _kv("Q8_0", Tn, nkv, d, 713)
    q = np.tile(synth.activations(1, d, 714), (nh, 1))
    out, _ = oracle_mod.attn_decode(t, q, K, V, Tn, nh, nkv, d, 0.3)
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[2], out[3])
    assert not np.array_equal(out[0], out[2])
