"""An independent MXFP4 encoder for tests: the inverse of the layout, written
from the page's statement of it rather than from the oracle's decoder.

Layout ("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs", PEROP kernel mxfp4_mv and
fn mx_scale): element c of row r is nibble j of little-endian word k of group
g (c = 32g + 8k + j).  Little-endian words make nibble j land in byte j // 2
of the word, low half when j is even, so the code plane is simply the row-major
element sequence packed two nibbles per byte, low nibble first.  The scale
plane (one byte per group, row-major) follows the code plane.
"""
import numpy as np

# E2M1 value table taken from the page-derived fixture tests/golden/e2m1_codes.txt.
from golden_io import rows, bits_to_f32

E2M1_VALUES = np.array([bits_to_f32(int(b, 16)) for _, b, _ in rows("e2m1_codes.txt")],
                       dtype=np.float32)


def encode(codes: np.ndarray, scales: np.ndarray, pad16: bool = True) -> np.ndarray:
    """codes: int [rows, cols] in 0..15; scales: int [rows, cols/32] in 0..255."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows_, cols = codes.shape
    assert cols % 32 == 0 and scales.shape == (rows_, cols // 32)
    plane = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8).reshape(-1)
    body = np.concatenate([plane, scales.reshape(-1)])
    if pad16:
        n = (body.size + 15) // 16 * 16
        body = np.concatenate([body, np.zeros(n - body.size, dtype=np.uint8)])
    return body


def dense(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The matrix the encoded buffer stands for, built with numpy's ldexp from
    the fixture's value table (float32; NaN where the scale byte is 255)."""
    codes = np.asarray(codes)
    scales = np.asarray(scales, dtype=np.int64)
    v = E2M1_VALUES[codes]
    s = np.ldexp(np.float32(1.0), (scales - 127).astype(np.int32)).astype(np.float32)
    s = np.where(scales == 255, np.float32(np.nan), s)
    with np.errstate(over="ignore", invalid="ignore"):
        return (v * np.repeat(s, 32, axis=1)).astype(np.float32)


def random_case(rng: np.random.Generator, rows_: int, cols: int, lo: int = 118, hi: int = 136):
    codes = rng.integers(0, 16, size=(rows_, cols))
    scales = rng.integers(lo, hi + 1, size=(rows_, cols // 32))
    return codes, scales
