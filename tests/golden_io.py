"""Reader for the hand-packed block fixtures under tests/golden/.

Format: '#' comments; 'type NAME'; 'hex ...' tokens (hex digits, or 'XX*k'
for a byte repeated k times) concatenated in order; optional 'scale S' (a
power of two multiplying every expected value); 'expect ...' tokens (a
number, or 'v*k' for v repeated k times)."""
from __future__ import annotations

import glob
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand(tok: str):
    if "*" in tok:
        v, k = tok.split("*")
        return [v] * int(k)
    return [tok]


def load(path: str):
    t, hexs, expect, scale = None, [], [], 1.0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *toks = line.split()
            if key == "type":
                t = toks[0]
            elif key == "hex":
                for tok in toks:
                    for piece in _expand(tok):
                        hexs.append(piece)
            elif key == "scale":
                scale = float(toks[0])
            elif key == "expect":
                for tok in toks:
                    expect += [float(v) for v in _expand(tok)]
    raw = bytes.fromhex("".join(hexs))
    return t, np.frombuffer(raw, np.uint8).copy(), np.array(expect, np.float64) * scale


def all_fixtures():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))
