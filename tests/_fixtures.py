"""Readers for the text fixtures under tests/golden/ (test plumbing only)."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def code_map():
    """[(doubled_magnitude, code, magnitude)] from e2m1_code_map.txt."""
    return [(int(a), int(b), float(c)) for a, b, c in _lines("e2m1_code_map.txt")]


def packing():
    """[(value_even, value_odd, byte)] from packing.txt."""
    return [(float(a), float(b), int(c, 16)) for a, b, c in _lines("packing.txt")]


def _bf16_bits(tok: str) -> int:
    v = np.float32(float(tok))
    bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
    assert bits & 0xFFFF == 0, f"{tok} is not exact in bf16"
    return bits >> 16


def hand_blocks():
    """(W bf16 bits [R, K], global, scales [R, K/16], packed [R, K/2])."""
    rows, scales, packed, g = {}, {}, {}, None
    for tok in _lines("hand_blocks.txt"):
        if tok[0] == "global":
            g = float(tok[1])
        elif tok[0] == "row":
            rows[int(tok[1])] = [_bf16_bits(t) for t in tok[2:]]
        elif tok[0] == "scales":
            scales[int(tok[1])] = [int(t, 16) for t in tok[2:]]
        elif tok[0] == "packed":
            packed[int(tok[1])] = [int(t, 16) for t in tok[2:]]
    R = len(rows)
    W = np.array([rows[i] for i in range(R)], dtype=np.uint16)
    S = np.array([scales[i] for i in range(R)], dtype=np.uint8)
    P = np.array([packed[i] for i in range(R)], dtype=np.uint8)
    return W, g, S, P
