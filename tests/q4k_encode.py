"""An independent encoder of GGUF Q4_K super-blocks for the tests: it packs
given scales, mins and codes the way the page's decode unpacks them ("rlx-cpu
0.2.17 src/gguf_matmul.rs", q4k_scale_min_x86 and q4k_dot_q8_block_avx2), so
that the oracle's decode can be pinned against values chosen by hand."""
import numpy as np


def pack_scales(sc, m) -> np.ndarray:
    """Eight 6-bit scales and mins -> the 12 packed bytes.  Sub-blocks 0-3: low
    six bits of bytes j (scale) and j + 4 (min).  Sub-blocks 4-7: low four bits
    in the low / high nibble of byte j + 4 (= 8 + (j - 4)), high two bits in the
    top of byte j - 4 (scale) and byte j (min)."""
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert all(0 <= v < 64 for v in sc + m)
    q = [0] * 12
    for j in range(4):
        q[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        q[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        q[j + 8] = (sc[j + 4] & 0x0F) | ((m[j + 4] & 0x0F) << 4)
    return np.array(q, dtype=np.uint8)


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def block(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """One 144-byte block from d, dmin (exact binary16 values), the sub-blocks'
    scales and mins and the 256 codes q (0..15) in element order."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 15
    out = np.zeros(144, dtype=np.uint8)
    db, mb = f16_bits(d), f16_bits(dmin)
    out[0], out[1], out[2], out[3] = db & 0xFF, db >> 8, mb & 0xFF, mb >> 8
    out[4:16] = pack_scales(sc, m)
    for s in range(4):   # 64 elements per 32 code bytes: low nibbles first
        lo = q[64 * s: 64 * s + 32]
        hi = q[64 * s + 32: 64 * s + 64]
        out[16 + 32 * s: 16 + 32 * s + 32] = (lo | (hi << 4)).astype(np.uint8)
    return out


def block_values(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """The 256 element values in float32: d*sc*q and dmin*m (exact) and one
    float32 rounding of their difference, sub-block j = element // 32."""
    q = np.asarray(q, dtype=np.float32)
    j = np.arange(256) // 32
    scv = np.asarray(sc, dtype=np.float32)[j]
    mv = np.asarray(m, dtype=np.float32)[j]
    scaled = (np.float32(d) * scv) * q
    mins = np.float32(dmin) * mv
    return (scaled - mins).astype(np.float32)


def random_components(rng, n_blocks: int):
    """Per block: d, dmin (exact binary16), scales, mins, codes."""
    out = []
    for _ in range(n_blocks):
        d = float(np.float16(rng.uniform(2.0 ** -12, 2.0 ** -6)))
        dmin = float(np.float16(rng.uniform(2.0 ** -12, 2.0 ** -6)))
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        out.append((d, dmin, sc, m, q))
    return out
