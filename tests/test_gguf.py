"""GGUF container reader (qk_gguf_*, host code, no GPU) against the plain
oracle reader (oracle/gguf.py) and a hand-assembled golden file: header,
metadata of every value type, tensor infos, alignment, tensor data pointers;
malformed and truncated images must give QK_ERR_FORMAT, never a crash."""
import os
import struct

import numpy as np
import pytest

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gguf_writer import write
from oracle import gguf as og

HERE = os.path.dirname(os.path.abspath(__file__))
FORMAT, IO = 9, 10


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gguf_quant_dequant_gb300 import build
    build.build()
    return qk.load()


def load_fixture(path):
    hexs, exp = [], {"kv": {}, "expect": []}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, *toks = line.split()
        if key == "hex":
            for tok in toks:
                if "*" in tok:
                    b, k = tok.split("*")
                    hexs.append(b * int(k))
                else:
                    hexs.append(tok)
        elif key in ("version", "alignment", "data_offset"):
            exp[key] = int(toks[0])
        elif key == "kv":
            exp["kv"][toks[0]] = (toks[1], toks[2])
        elif key == "tensor":
            exp["tensor"] = (toks[0], [int(v) for v in toks[1].split(",")], int(toks[2]), int(toks[3]), int(toks[4]))
        elif key == "expect":
            exp["expect"] += [float(v) for v in toks]
    return bytes.fromhex("".join(hexs)), exp


def test_golden_minimal_file():
    data, exp = load_fixture(os.path.join(HERE, "golden", "gguf_minimal.gguf.hex"))
    assert len(data) == exp["data_offset"] + exp["tensor"][4]
    # The oracle reader ...
    o = og.read(data)
    assert o["version"] == exp["version"] and o["alignment"] == exp["alignment"]
    assert o["data_offset"] == exp["data_offset"]
    assert o["kv"]["general.architecture"] == (8, b"llama") and o["kv"]["general.alignment"] == (4, 32)
    name, dims, gtype, off, nbytes = exp["tensor"]
    assert o["tensors"] == [(name, dims, gtype, off)]
    # ... the library's reader ...
    with qk.GGUF(data=data) as g:
        assert (g.version, g.alignment, g.data_offset) == (3, 32, 160)
        assert g.keys() == ["general.architecture", "general.alignment"]
        assert g.kv("general.architecture") == "llama" and g.kv("general.alignment") == 32
        t = g.tensor("w")
        assert t["dims"] == dims and t["ggml_type"] == gtype and t["qk_type"] == qk.Q8_0
        assert t["offset"] == 160 and t["nbytes"] == nbytes
        blob = np.frombuffer(g.tensor_bytes("w"), np.uint8)
    # ... and the weights the blocks hold.
    w = oracle.dequant(oracle.Q8_0, blob, dims[1], dims[0])
    assert np.array_equal(w.reshape(-1), np.array(exp["expect"], np.float32))


KVS = [
    ("general.architecture", "str", "llama"),
    ("general.name", "str", "tiny ünïcode model"),
    ("llama.context_length", "u32", 131072),
    ("llama.embedding_length", "u64", 4096),
    ("x.i8", "i8", -5), ("x.u8", "u8", 250), ("x.i16", "i16", -30000), ("x.u16", "u16", 65000),
    ("x.i32", "i32", -2 ** 31), ("x.i64", "i64", -2 ** 63), ("x.f32", "f32", 1.5), ("x.f64", "f64", -2.25e-300),
    ("x.bool", "bool", True),
    ("tokenizer.ggml.tokens", ("arr", "str"), ["<s>", "</s>", "hello", ""]),
    ("tokenizer.ggml.scores", ("arr", "f32"), [0.0, -1.5, 2.25]),
    ("x.ints", ("arr", "i32"), [1, -2, 3]),
    ("x.flags", ("arr", "bool"), [True, False]),
    ("x.nested", ("arr", ("arr", "u8")), [[1, 2], [3]]),
    ("x.empty", ("arr", "u64"), []),
    ("x.big", "u64", 2 ** 64 - 1),
]


def rich_tensors():
    rng = np.random.default_rng(42)
    ts = [("unsized.q41", [32, 1], "Q4_1", rng.integers(0, 256, 20, dtype=np.uint8).tobytes())]
    for name, gt, rows, cols in (("blk.0.ffn_up.weight", "Q4_K", 8, 1024), ("blk.0.attn_v.weight", "Q6_K", 3, 256),
                                 ("blk.0.attn_q.weight", "Q8_0", 5, 64), ("blk.0.ffn_gate.weight", "Q5_0", 2, 32),
                                 ("blk.0.attn_k.weight", "Q4_0", 1, 96), ("blk.1.attn_q.weight", "Q5_K", 2, 512),
                                 ("blk.1.ffn_up.weight", "Q2_K", 3, 256), ("blk.1.ffn_down.weight", "Q3_K", 2, 768)):
        ts.append((name, [cols, rows], gt, synth.random_blocks(gt, rows, cols, 300 + rows).tobytes()))
    ts.append(("norm.weight", [7], "F32", rng.standard_normal(7).astype(np.float32).tobytes()))
    ts.append(("emb.f16", [4, 2], "F16", rng.standard_normal(8).astype(np.float16).tobytes()))
    ts.append(("emb.bf16", [3], "BF16", rng.integers(0, 2 ** 16, 3, dtype=np.uint16).tobytes()))
    return ts


def test_rich_file_matches_the_oracle_reader(tmp_path):
    ts = rich_tensors()
    data = write(KVS, ts, alignment=64)
    o = og.read(data)
    path = tmp_path / "rich.gguf"
    path.write_bytes(data)
    for g in (qk.GGUF(data=data), qk.GGUF(path=str(path))):
        with g:
            assert g.version == 3 and g.alignment == 64 and g.data_offset == o["data_offset"]
            assert g.keys() == list(o["kv"])
            for key, (vt, val) in o["kv"].items():
                if key in ("x.nested", "x.big"):
                    with pytest.raises(qk.QKError):
                        g.kv(key)
                    continue
                got = g.kv(key)
                if vt == 8:
                    assert got == val.decode()
                elif vt == 9:
                    et, items = val
                    assert got == [v.decode() if et == 8 else v for v in items]
                else:
                    assert got == val
            assert g.kv_type("x.nested") == 9
            tens = g.tensors()
            assert [(t["name"], t["dims"], t["ggml_type"], t["offset"] - o["data_offset"]) for t in tens] == \
                [(n, d, gt, off) for (n, d, gt, off) in o["tensors"]]
            for (name, dims, gt, blob), t in zip(ts, tens):
                if gt == "Q4_1":
                    assert t["nbytes"] == 0 and t["qk_type"] == -1   # not sized by this library
                    continue
                assert t["nbytes"] == len(blob) and g.tensor_bytes(name) == blob
                assert t["offset"] % 64 == 0
            assert g.tensor("blk.0.attn_v.weight")["qk_type"] == qk.Q6_K
            with pytest.raises(KeyError):
                g.tensor("missing")
            with pytest.raises(KeyError):
                g.kv("missing")


def _status(data):
    try:
        qk.GGUF(data=data).close()
        return 0
    except qk.QKError as e:
        return e.status


def test_every_truncation_is_rejected():
    ts = rich_tensors()
    data = write(KVS, ts, alignment=32)
    o = og.read(data)
    # The last sized tensor's data ends here; the unsized one comes first.
    last = max(off + len(blob) for (_, _, _, off), (_, _, gt, blob) in zip(o["tensors"], ts) if gt != "Q4_1")
    end = o["data_offset"] + last
    for n in range(len(data) + 1):
        st = _status(data[:n])
        assert st == (0 if n >= end else FORMAT), (n, st)


def test_corrupted_images_never_crash():
    data = bytearray(write(KVS, rich_tensors(), alignment=32))
    meta_end = og.read(bytes(data))["data_offset"]
    rng = np.random.default_rng(77)
    seen = set()
    for _ in range(400):
        d = bytearray(data)
        for _ in range(int(rng.integers(1, 5))):
            d[int(rng.integers(0, meta_end))] = int(rng.integers(0, 256))
        st = _status(bytes(d))
        assert st in (0, FORMAT)
        seen.add(st)
    assert FORMAT in seen


def header(nt, nkv, version=3):
    return b"GGUF" + struct.pack("<IQQ", version, nt, nkv)


@pytest.mark.parametrize("case", [
    "magic", "version1", "version4", "huge_tensor_count", "huge_kv_count", "alignment_48",
    "alignment_u64", "unaligned_offset", "n_dims_0", "n_dims_5", "partial_block", "shape_overflow",
    "data_past_end", "bad_value_type", "bad_array_type", "deep_array",
])
def test_malformed_images(case):
    ok_t = [("w", [32, 1], "Q8_0", bytes(34))]
    if case == "magic":
        data = b"GGUX" + write([], ok_t)[4:]
    elif case == "version1":
        data = write([], ok_t, version=1)
    elif case == "version4":
        data = write([], ok_t, version=4)
    elif case == "huge_tensor_count":
        data = header(2 ** 63, 0) + bytes(64)
    elif case == "huge_kv_count":
        data = header(0, 2 ** 62) + bytes(64)
    elif case == "alignment_48":
        data = write([], ok_t, alignment=48)
    elif case == "alignment_u64":
        data = write([("general.alignment", "u64", 32)], ok_t)
    elif case == "unaligned_offset":
        data = bytearray(write([], [("a", [32, 1], "Q8_0", bytes(34)), ("b", [32, 1], "Q8_0", bytes(34))]))
        o = og.read(bytes(data))
        # Patch tensor b's offset (its last 8 info bytes) to 1 byte past its start.
        pos = data.find(b"\x01\x00\x00\x00\x00\x00\x00\x00b") + 9 + 4 + 16 + 4
        struct.pack_into("<Q", data, pos, o["tensors"][1][3] + 1)
        data = bytes(data)
    elif case == "n_dims_0":
        data = write([], [("w", [], "F32", b"")])
    elif case == "n_dims_5":
        data = write([], [("w", [1, 1, 1, 1, 1], "F32", bytes(4))])
    elif case == "partial_block":
        data = write([], [("w", [100, 1], "Q4_K", bytes(144))])
    elif case == "shape_overflow":
        data = write([], [("w", [2 ** 40, 2 ** 40], "F32", b"")])
    elif case == "data_past_end":
        data = write([], [("w", [256, 2], "Q4_K", bytes(144))])   # two rows declared, one written
    elif case == "bad_value_type":
        data = header(0, 1) + struct.pack("<Q", 1) + b"k" + struct.pack("<I", 13) + bytes(8)
    elif case == "bad_array_type":
        data = header(0, 1) + struct.pack("<Q", 1) + b"k" + struct.pack("<IIQ", 9, 13, 1) + bytes(8)
    else:   # nine levels of nested arrays
        v = b""
        for _ in range(9):
            v = struct.pack("<IQ", 9, 1) + v
        data = header(0, 1) + struct.pack("<Q", 1) + b"k" + struct.pack("<I", 9) + v + struct.pack("<IQ", 0, 0)
    assert _status(data) == FORMAT, case


def test_open_errors(tmp_path):
    with pytest.raises(qk.QKError) as e:
        qk.GGUF(path=str(tmp_path / "missing.gguf"))
    assert e.value.status == IO
    (tmp_path / "empty.gguf").write_bytes(b"")
    with pytest.raises(qk.QKError) as e:
        qk.GGUF(path=str(tmp_path / "empty.gguf"))
    assert e.value.status == IO
    with pytest.raises(qk.QKError) as e:
        qk.GGUF(path=str(tmp_path))   # a directory
    assert e.value.status == IO
    (tmp_path / "junk.gguf").write_bytes(b"not a gguf file at all, just text")
    with pytest.raises(qk.QKError) as e:
        qk.GGUF(path=str(tmp_path / "junk.gguf"))
    assert e.value.status == FORMAT


def test_null_arguments_are_rejected(lib):
    import ctypes
    h = ctypes.c_void_p()
    assert lib.qk_gguf_open(None, ctypes.byref(h)) == 4
    assert lib.qk_gguf_parse(None, 10, ctypes.byref(h)) == 4
    assert lib.qk_gguf_n_kv(None) == -1 and lib.qk_gguf_find_tensor(None, b"x") == -1
    lib.qk_gguf_close(None)
