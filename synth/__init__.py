"""Seeded synthetic inputs shared by the oracle tests, the parity tests and the
benchmark.

This module only draws numbers and lays raw bytes out; it holds none of the
method's arithmetic (no decode, no dot product, no SiLU).  Every draw comes from
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): output i of a stream with seed s is the finaliser
applied to s + (i+1) * 0x9E3779B97F4A7C15, so any range of a stream can be
produced independently (counter-based), vectorised here with numpy.

Buffers follow the MXFP4 tensor layout of "cortiq-engine 0.8.40
src/gpu_wgpu/mxfp4.rs": rows*cols/2 code bytes, then rows*cols/32 E8M0 scale
bytes, then zero padding up to a multiple of 16 bytes (the GPU library's
buffer rule).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream `seed` (uint64)."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & _MASK64) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def substream(seed: int, name: str) -> int:
    """A stream seed derived from a config seed and a purpose name."""
    h = 0xCBF29CE484222325
    for ch in name.encode():
        h = ((h ^ ch) * 0x100000001B3) & _MASK64
    mixed = splitmix64((seed * 0x2545F4914F6CDD1D + h) & _MASK64, 1)[0]
    return int(mixed)


def random_bytes(seed: int, n: int, chunk: int = 1 << 24) -> np.ndarray:
    """n uniform bytes (8 per SplitMix64 output, little-endian)."""
    out = np.empty(n, dtype=np.uint8)
    words = (n + 7) // 8
    pos = 0
    for w0 in range(0, words, chunk):
        w = splitmix64(seed, min(chunk, words - w0), w0)
        b = w.view(np.uint8)
        take = min(b.size, n - pos)
        out[pos:pos + take] = b[:take]
        pos += take
    return out


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive), int64."""
    span = np.uint64(hi - lo + 1)
    return (splitmix64(seed, n) % span).astype(np.int64) + lo


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """n doubles uniform in (0, 1]: (top 53 bits + 1) * 2^-53."""
    w = splitmix64(seed, n, start)
    return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal_f32(seed: int, n: int) -> np.ndarray:
    """n N(0,1) draws (Box-Muller in double, rounded to float32)."""
    m = (n + 1) // 2
    u1 = uniform01(seed, m, 0)
    u2 = uniform01(seed, m, m)
    rad = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m)
    z[0::2] = rad * np.cos(2.0 * math.pi * u2)
    z[1::2] = rad * np.sin(2.0 * math.pi * u2)
    return z[:n].astype(np.float32)


# --- MXFP4 buffers -----------------------------------------------------------

def code_bytes(rows: int, cols: int) -> int:
    return rows * cols // 2


def scale_bytes(rows: int, cols: int) -> int:
    return rows * (cols // 32)


def padded_nbytes(rows: int, cols: int) -> int:
    n = code_bytes(rows, cols) + scale_bytes(rows, cols)
    return (n + 15) // 16 * 16


def assemble(codes: np.ndarray, scales: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Concatenate a code plane and a scale plane into one padded buffer."""
    assert codes.size == code_bytes(rows, cols) and scales.size == scale_bytes(rows, cols)
    buf = np.zeros(padded_nbytes(rows, cols), dtype=np.uint8)
    buf[:codes.size] = codes
    buf[codes.size:codes.size + scales.size] = scales
    return buf


def mxfp4_matrix(rows: int, cols: int, seed: int, scale_lo: int, scale_hi: int,
                 special: dict | None = None, scale_pattern: str = "uniform") -> np.ndarray:
    """A random [rows, cols] MXFP4 buffer.

    Code nibbles are uniform over 0..15.  Scales are uniform in
    [scale_lo, scale_hi] ("uniform"), or follow lo + (3*i + seed) mod 5 over
    the flat group index i ("adjacent_distinct": neighbouring groups, also
    across a row boundary, always get different scales, so reading another
    group's scale byte cannot go unnoticed).  `special` maps (row, group) to a
    forced scale byte (e.g. 0 for the subnormal scale, 255 for NaN).
    """
    assert cols % 32 == 0 and rows > 0
    codes = random_bytes(substream(seed, "codes"), code_bytes(rows, cols))
    n_s = scale_bytes(rows, cols)
    if scale_pattern == "uniform":
        scales = uniform_int(substream(seed, "scales"), n_s, scale_lo, scale_hi).astype(np.uint8)
    elif scale_pattern == "adjacent_distinct":
        i = np.arange(n_s, dtype=np.int64)
        scales = (scale_lo + (3 * i + seed) % 5).astype(np.uint8)
    else:
        raise ValueError(scale_pattern)
    for (r, g), k in (special or {}).items():
        scales[r * (cols // 32) + g] = k
    return assemble(codes, scales, rows, cols)


def expert_bank(n_experts: int, rows: int, cols: int, seed: int, scale_lo: int,
                scale_hi: int, role: str) -> np.ndarray:
    """n_experts MXFP4 [rows, cols] buffers back to back, each padded; every
    expert and role gets its own code and scale streams (no two experts share
    a scale plane)."""
    stride = padded_nbytes(rows, cols)
    bank = np.empty(n_experts * stride, dtype=np.uint8)
    for e in range(n_experts):
        bank[e * stride:(e + 1) * stride] = mxfp4_matrix(
            rows, cols, substream(seed, f"{role}/{e}"), scale_lo, scale_hi)
    return bank


def int_activations(seed: int, n: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Small-integer activations (exact in every float format used)."""
    return uniform_int(seed, n, lo, hi).astype(np.float32)


def routes(seed: int, n_tokens: int, top_k: int, n_experts: int):
    """Per token: top_k distinct experts drawn uniformly (partial Fisher-Yates)
    and route weights = softmax of top_k N(0,1) logits (computed in double,
    stored as float32).  Returns (ids int32 [T, k], weights float32 [T, k])."""
    draws = splitmix64(substream(seed, "route-ids"), n_tokens * top_k)
    ids = np.empty((n_tokens, top_k), dtype=np.int32)
    for t in range(n_tokens):
        perm = list(range(n_experts))
        for j in range(top_k):
            pick = j + int(draws[t * top_k + j] % np.uint64(n_experts - j))
            perm[j], perm[pick] = perm[pick], perm[j]
            ids[t, j] = perm[j]
    logits = normal_f32(substream(seed, "route-logits"), n_tokens * top_k)
    logits = logits.astype(np.float64).reshape(n_tokens, top_k)
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    weights = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, weights


# --- GGUF Q4_K buffers (the second codec) ---------------------------------------

Q4K_BLOCK_BYTES = 144   # one 256-element super-block (layout: the library's q4k.h)


def q4k_nbytes(rows: int, cols: int) -> int:
    return rows * (cols // 256) * Q4K_BLOCK_BYTES


def q4k_matrix(rows: int, cols: int, seed: int, d_lo: int = -12, d_hi: int = -9) -> np.ndarray:
    """rows x cols/256 Q4_K super-blocks of seeded bytes.  Bytes 0-1 (d) and 2-3
    (dmin) of each block are positive binary16 values 2^e (1 + f/1024), e uniform
    in [d_lo, d_hi] and f in [0, 1023]; every other byte is uniform (any byte
    pattern of the scales and codes is a valid encoding)."""
    assert cols % 256 == 0
    n_blk = rows * (cols // 256)
    buf = uniform_int(substream(seed, "q4k/bytes"), n_blk * Q4K_BLOCK_BYTES, 0, 255).astype(
        np.uint8).reshape(n_blk, Q4K_BLOCK_BYTES)
    for k, tag in ((0, "q4k/d"), (2, "q4k/dmin")):
        e = uniform_int(substream(seed, tag + "/e"), n_blk, d_lo, d_hi)
        f = uniform_int(substream(seed, tag + "/f"), n_blk, 0, 1023)
        bits = ((e + 15) << 10) | f
        buf[:, k] = (bits & 0xFF).astype(np.uint8)
        buf[:, k + 1] = (bits >> 8).astype(np.uint8)
    return buf.reshape(-1)


@dataclass(frozen=True)
class Q4kConfig:
    name: str
    rows: int
    cols: int
    nb: int
    seed: int

    def weights(self) -> np.ndarray:
        return q4k_matrix(self.rows, self.cols, self.seed)

    def activations(self) -> np.ndarray:
        return normal_f32(substream(self.seed, "x"), self.nb * self.cols).reshape(
            self.nb, self.cols)


# --- the workloads -----------------------------------------------------------

@dataclass(frozen=True)
class MatConfig:
    name: str
    rows: int
    cols: int
    nb: int
    seed: int
    scale_lo: int = 118
    scale_hi: int = 130
    special: dict = field(default_factory=dict)

    def weights(self) -> np.ndarray:
        return mxfp4_matrix(self.rows, self.cols, self.seed, self.scale_lo, self.scale_hi,
                            self.special)

    def activations(self) -> np.ndarray:
        return normal_f32(substream(self.seed, "x"), self.nb * self.cols).reshape(
            self.nb, self.cols)


@dataclass(frozen=True)
class MoeConfig:
    name: str
    n_experts: int
    hidden: int
    inter: int
    n_tokens: int
    top_k: int
    seed: int
    scale_lo: int = 118
    scale_hi: int = 130

    @property
    def gu_stride(self) -> int:
        return padded_nbytes(self.inter, self.hidden)

    @property
    def down_stride(self) -> int:
        return padded_nbytes(self.hidden, self.inter)

    def banks(self):
        gate = expert_bank(self.n_experts, self.inter, self.hidden, self.seed,
                           self.scale_lo, self.scale_hi, "gate")
        up = expert_bank(self.n_experts, self.inter, self.hidden, self.seed,
                         self.scale_lo, self.scale_hi, "up")
        down = expert_bank(self.n_experts, self.hidden, self.inter, self.seed,
                           self.scale_lo, self.scale_hi, "down")
        return gate, up, down

    def activations(self) -> np.ndarray:
        return normal_f32(substream(self.seed, "x"), self.n_tokens * self.hidden).reshape(
            self.n_tokens, self.hidden)

    def routes(self):
        return routes(self.seed, self.n_tokens, self.top_k, self.n_experts)


# The five workloads (sizes, distributions and seeds of the method's
# configurations).  tiny: one k=0 (subnormal) group at (row 3, group 5) and one
# k=255 (NaN) group at (row 250, group 11).
TINY = MatConfig("mxfp4_mv tiny 256x512", 256, 512, 1, seed=0, scale_lo=118, scale_hi=136,
                 special={(3, 5): 0, (250, 11): 255})
DECODE = MatConfig("mxfp4_mv decode GEMV 14336x4096", 14336, 4096, 1, seed=1)
MM8 = MatConfig("mxfp4_mm small batch 4096x14336 nb=8", 4096, 14336, 8, seed=2)
MOE = MoeConfig("MoE 64 experts 2880x2880 top-4, 32 tokens", 64, 2880, 2880, 32, 4, seed=3)
PREFILL = MatConfig("mxfp4_mm prefill 4096x4096 nb=2048", 4096, 4096, 2048, seed=4)
# the second codec: the same decode GEMV shape in GGUF Q4_K, f32 activations
Q4K_DECODE = Q4kConfig("q4k_mv decode GEMV 14336x4096 (GGUF Q4_K)", 14336, 4096, 1, seed=5)
CONFIGS = {"tiny": TINY, "decode": DECODE, "mm8": MM8, "moe": MOE, "prefill": PREFILL}
