"""End to end from a GGUF file: tensors of every supported type are written
to a file, opened through the library's reader (memory-mapped), their blocks
copied to the device and run through qk_dequant and qk_gemv; the results are
checked against the oracle on the same bytes (dequant bit-exact, GEMV within
1e-4 * sum|w x| + 1e-6)."""
import numpy as np
import pytest
import torch

import gguf_quant_dequant_gb300 as qk
import oracle
import synth
from gguf_writer import write
from gpu_helpers import assert_gemv_close, gpu  # noqa: F401

pytestmark = pytest.mark.gpu

SHAPES = [("blk.0.attn_q.weight", "Q4_K", 96, 1024), ("blk.0.attn_v.weight", "Q6_K", 40, 512),
          ("blk.0.ffn_down.weight", "Q8_0", 33, 1024), ("blk.0.ffn_gate.weight", "Q5_0", 17, 256),
          ("blk.0.ffn_up.weight", "Q4_0", 64, 2048), ("blk.0.attn_k.weight", "Q5_K", 40, 1024),
          ("blk.1.ffn_up.weight", "Q2_K", 24, 1024), ("blk.1.ffn_down.weight", "Q3_K", 16, 768)]


def test_gemv_from_a_gguf_file(gpu, tmp_path):
    blobs = {name: synth.random_blocks(t, rows, cols, 900 + rows) for name, t, rows, cols in SHAPES}
    tensors = [(name, [cols, rows], t, blobs[name].tobytes()) for name, t, rows, cols in SHAPES]
    tensors.append(("output_norm.weight", [4096], "F32", np.ones(4096, np.float32).tobytes()))
    path = tmp_path / "layer.gguf"
    path.write_bytes(write([("general.architecture", "str", "llama")], tensors))
    with qk.GGUF(path=str(path)) as g:
        assert g.kv("general.architecture") == "llama"
        for name, t, rows, cols in SHAPES:
            info = g.tensor(name)
            assert info["dims"] == [cols, rows] and info["qk_type"] == synth.TYPE_IDS[t]
            W = np.frombuffer(g.tensor_bytes(name), np.uint8).copy()
            assert np.array_equal(W, blobs[name])
            Wd = torch.from_numpy(W).to(gpu)
            qt = info["qk_type"]
            w = qk.dequant(qt, Wd, rows, cols).cpu().numpy()
            assert np.array_equal(w, oracle.dequant(qt, W, rows, cols))
            x = synth.activations(1, cols, 950 + rows)
            y = qk.gemv(qt, Wd, rows, cols, torch.from_numpy(x).to(gpu)).cpu().numpy()
            y_ref, S = oracle.gemv(qt, W, rows, cols, x)
            assert_gemv_close(y, y_ref, S, what=f"gemv from file: {name}")
    qk.device_status()
