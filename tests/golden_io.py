"""Readers for the small text fixtures under tests/golden/ (each fixture cites
the passage of the source page its values come from)."""
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    """Non-comment, non-empty lines of a fixture, split on whitespace."""
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def bits_to_f32(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b))[0]


def f32_to_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", np.float32(v)))[0]


def parse_value(tok: str) -> float:
    """'nan', a decimal, or '<decimal>p<exp>' meaning decimal * 2**exp."""
    if tok == "nan":
        return float("nan")
    if "p" in tok:
        m, e = tok.split("p")
        return float(m) * 2.0 ** int(e)
    return float(tok)
