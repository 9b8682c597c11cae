"""Pins for the oracle's second codec (GGUF Q4_K): its binary16 decode against
numpy's, its scale/min unpacking and element placement against an independent
encoder, its block dot against the page's own loop form, and its products
against dense numpy.  CPU only."""
import numpy as np
import pytest

from q4k_encode import block, block_values, pack_scales, random_components


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def test_f16_every_bit_pattern_matches_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([orc.f16(int(b)) for b in bits], dtype=np.float32)
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    assert np.array_equal(nan_w, nan_g)
    assert np.array_equal(got[~nan_g].view(np.uint32), want[~nan_w].view(np.uint32))


def test_f16_closed_forms(orc):
    assert orc.f16(0x3C00) == 1.0 and orc.f16(0xC000) == -2.0
    assert orc.f16(0x0001) == 2.0 ** -24 and orc.f16(0x0400) == 2.0 ** -14
    assert orc.f16(0x7BFF) == 65504.0 and orc.f16(0x7C00) == float("inf")


def test_scale_min_roundtrip_and_hand_example(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        sc, m = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
        q = pack_scales(sc, m)
        for j in range(8):
            assert orc.q4k_scale_min(q, j) == (sc[j], m[j])
    # sub-block 5 by hand: scale 0b101101 = 45, min 0b010110 = 22 -> byte 9 =
    # 0x6D (min low nibble 6, scale low nibble 13), byte 1 top bits 0b10 (scale),
    # byte 5 top bits 0b01 (min)
    q = np.zeros(12, dtype=np.uint8)
    q[9], q[1], q[5] = 0x6D, 0b10 << 6, 0b01 << 6
    assert orc.q4k_scale_min(q, 5) == (45, 22)
    assert orc.q4k_scale_min(q, 1) == (0, 0)   # the borrowed top bits are not sub-block 1's


def test_dequant_against_hand_chosen_components(orc):
    rng = np.random.default_rng(7)
    rows, nblk = 3, 2
    comps = random_components(rng, rows * nblk)
    buf = np.concatenate([block(*c) for c in comps])
    want = np.concatenate([block_values(*c) for c in comps]).reshape(rows, nblk * 256)
    got = orc.q4k_dequant(buf, rows, nblk * 256)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_one_element_by_hand(orc):
    # d = 0.5, dmin = 0.25, sub-block 3 (elements 96..127: the high nibbles of
    # bytes 48..79): scale 7, min 5; element 100 has code 9
    sc, m = [0] * 8, [0] * 8
    sc[3], m[3] = 7, 5
    q = np.zeros(256, dtype=np.int64)
    q[100] = 9
    buf = block(0.5, 0.25, sc, m, q)
    assert buf[16 + 32 + 4] == 9 << 4          # element 100 = 64 + 32 + 4
    w = orc.q4k_dequant(buf, 1, 256)[0]
    assert w[100] == 0.5 * 7 * 9 - 0.25 * 5     # 30.25
    assert w[101] == -1.25 and w[95] == 0.0   # code 0 in sub-block 3; sub-block 2 all zero


def test_block_dot_in_the_pages_loop_form(orc):
    # the page's block dot walks the 128 code bytes 32 at a time: the low
    # nibbles of bytes is..is+31 against x[yi..yi+31] (sub-block j), the high
    # nibbles against x[yi+32..yi+63] (sub-block j+1), and subtracts dmin*m_j
    # times the sum of each sub-block's x; written here from the raw bytes
    rng = np.random.default_rng(11)
    for c in random_components(rng, 6):
        buf = block(*c)
        x = rng.standard_normal(256).astype(np.float32)
        d = float(np.float16(c[0]))
        dmin = float(np.float16(c[1]))
        scal = [orc.q4k_scale_min(buf[4:16], j) for j in range(8)]
        qs = buf[16:].astype(np.int64)
        xd = x.astype(np.float64)
        total, is_, yi = 0.0, 0, 0
        for j in range(0, 8, 2):
            lo = qs[is_:is_ + 32] & 0x0F
            hi = qs[is_:is_ + 32] >> 4
            total += d * scal[j][0] * np.dot(lo, xd[yi:yi + 32])
            total += d * scal[j + 1][0] * np.dot(hi, xd[yi + 32:yi + 64])
            total -= dmin * scal[j][1] * xd[yi:yi + 32].sum()
            total -= dmin * scal[j + 1][1] * xd[yi + 32:yi + 64].sum()
            yi += 64
            is_ += 32
        y, l1 = orc.q4k_matmat(buf, 1, 256, x, 1)
        # the oracle's elements are float-rounded: within a float spacing each
        assert abs(y[0, 0] - total) <= 2.0 ** -23 * l1[0, 0] + 1e-30


@pytest.mark.parametrize("rows,cols,nb", [(3, 256, 1), (5, 512, 3), (2, 1024, 2)])
def test_matmat_against_dense_numpy(orc, rows, cols, nb):
    import synth
    w = synth.q4k_matrix(rows, cols, rows + cols + nb)
    x = synth.normal_f32(nb + 3, nb * cols).reshape(nb, cols)
    y, l1 = orc.q4k_matmat(w, rows, cols, x, nb)
    W = orc.q4k_dequant(w, rows, cols).astype(np.float64)
    X = x.astype(np.float64)
    np.testing.assert_allclose(y, X @ W.T, rtol=0, atol=1e-12 * (np.abs(X) @ np.abs(W).T).max())
    np.testing.assert_allclose(l1, np.abs(X) @ np.abs(W).T, rtol=1e-12)
    y2, _ = orc.q4k_matmat(w, rows, cols, x, nb, 1, rows)   # a row window
    assert np.array_equal(y2, y[:, 1:])


def test_nbytes_closed_form_and_refusals(orc):
    assert orc.q4k_nbytes(14336, 4096) == 14336 * 16 * 144
    assert orc.q4k_nbytes(1, 256) == 144
    assert orc.q4k_nbytes(4, 320) == 0 and orc.q4k_nbytes(0, 256) == 0
