"""GPU parity of the second codec (GGUF Q4_K, f32 activations) against the
oracle: the dequantisation bit for bit, products within 1e-5 of their L1 norm,
exact inputs exactly, the batch equal to the matvec per token bit for bit,
special block factors, the decode GEMV shape."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import REL_FP32, assert_within, cuda, empty, host, to_dev
from q4k_encode import block, random_components

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    return cuda()


def same_bits(a, b):
    a = np.asarray(a, dtype=np.float32).reshape(-1)
    b = np.asarray(b, dtype=np.float32).reshape(-1)
    na, nb_ = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb_), "NaN positions differ"
    assert np.array_equal(a[~na].view(np.uint32), b[~nb_].view(np.uint32))


@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (77, 1024), (130, 4096)])
def test_dequant_bit_for_bit(mx, rows, cols):
    w = synth.q4k_matrix(rows, cols, rows * 7 + cols)
    out = empty(rows * cols)
    mx.q4k_dequant(to_dev(w), rows, cols, out)
    same_bits(host(out), oracle.q4k_dequant(w, rows, cols))


@pytest.mark.parametrize("rows,cols", [(1, 256), (5, 512), (257, 4096), (64, 14336),
                                       (40, 7168)])
def test_mv_against_oracle(mx, rows, cols):
    w = synth.q4k_matrix(rows, cols, rows + 3 * cols)
    x = synth.normal_f32(rows + cols, cols)
    y = empty(rows)
    mx.q4k_mv(to_dev(w), rows, cols, to_dev(x), y)
    ref, l1 = oracle.q4k_matmat(w, rows, cols, x, 1)
    assert_within(host(y), ref[0], l1[0], REL_FP32, "q4k_mv")


@pytest.mark.parametrize("nb", [2, 3, 5, 8, 9, 17])
def test_mm_equals_mv_per_token(mx, nb):
    rows, cols = 96, 1536
    w = synth.q4k_matrix(rows, cols, 40 + nb)
    X = synth.normal_f32(nb, nb * cols).reshape(nb, cols)
    wd = to_dev(w)
    Y = empty(nb * rows)
    mx.q4k_mm(wd, rows, cols, to_dev(X), nb, Y)
    got = host(Y).reshape(nb, rows)
    for t in range(nb):
        y = empty(rows)
        mx.q4k_mv(wd, rows, cols, to_dev(X[t]), y)
        same_bits(got[t], host(y))
    ref, l1 = oracle.q4k_matmat(w, rows, cols, X, nb)
    assert_within(got, ref, l1, REL_FP32, "q4k_mm")


def test_exact_inputs_exactly(mx):
    # d, dmin powers of two, x small integers: every value and sum is exact
    rng = np.random.default_rng(3)
    rows, nblk = 6, 3
    blocks = []
    for _ in range(rows * nblk):
        d = float(2.0 ** rng.integers(-4, 0))
        dmin = float(2.0 ** rng.integers(-4, 0))
        blocks.append(block(d, dmin, rng.integers(0, 64, 8), rng.integers(0, 64, 8),
                            rng.integers(0, 16, 256)))
    w = np.concatenate(blocks)
    cols = nblk * 256
    x = rng.integers(-3, 4, cols).astype(np.float32)
    y = empty(rows)
    mx.q4k_mv(to_dev(w), rows, cols, to_dev(x), y)
    ref, _ = oracle.q4k_matmat(w, rows, cols, x, 1)
    assert np.array_equal(host(y).astype(np.float64), ref[0])


def test_special_block_factors(mx):
    # infinite, NaN and subnormal d / dmin, zero dmin: element values as the
    # definition gives them (NaN compared by class), products NaN exactly where
    # the oracle's are
    rng = np.random.default_rng(9)
    comps = random_components(rng, 8)
    w = np.concatenate([block(*c) for c in comps])
    hdr = w.reshape(8, 144)
    for i, (db, mb) in enumerate([(0x7C00, 0x2000), (0x2000, 0x7E00), (0x0001, 0x0003),
                                  (0x3C00, 0x0000), (0xFC00, 0x2000), (0x0000, 0x0000)]):
        hdr[i, 0], hdr[i, 1], hdr[i, 2], hdr[i, 3] = db & 0xFF, db >> 8, mb & 0xFF, mb >> 8
    rows, cols = 2, 1024
    out = empty(rows * cols)
    mx.q4k_dequant(to_dev(w), rows, cols, out)
    same_bits(host(out), oracle.q4k_dequant(w, rows, cols))
    x = synth.normal_f32(5, cols)
    y = empty(rows)
    mx.q4k_mv(to_dev(w), rows, cols, to_dev(x), y)
    ref, l1 = oracle.q4k_matmat(w, rows, cols, x, 1)
    got = host(y)
    assert np.array_equal(np.isnan(got), np.isnan(ref[0]))


def test_decode_config_row_windows_and_rerun(mx):
    cfg = synth.Q4K_DECODE
    w, x = cfg.weights(), cfg.activations()[0]
    wd, xd = to_dev(w), to_dev(x)
    y = empty(cfg.rows)
    mx.q4k_mv(wd, cfg.rows, cfg.cols, xd, y)
    got = host(y)
    for r0, r1 in ((0, 512), (7000, 7300), (cfg.rows - 300, cfg.rows)):
        ref, l1 = oracle.q4k_matmat(w, cfg.rows, cfg.cols, x, 1, r0, r1)
        assert_within(got[r0:r1], ref[0], l1[0], REL_FP32, f"rows {r0}..{r1}")
    y2 = empty(cfg.rows)
    mx.q4k_mv(wd, cfg.rows, cfg.cols, xd, y2)
    same_bits(host(y2), got)
