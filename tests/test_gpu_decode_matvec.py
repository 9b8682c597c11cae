"""GPU parity: standalone decode (bit-exact) and the FP32 matvec / small-batch
product (within 1e-5 of the L1 bound) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (REL_FP32, assert_bits_equal, assert_within, cuda, empty, host, to_dev)
from mx_encode import encode, random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    return cuda()


def run_mv(mx, w_h, rows, cols, x_h):
    y = empty(rows)
    mx.mxfp4_mv(to_dev(w_h), rows, cols, to_dev(x_h), y)
    return host(y)


def run_mm(mx, w_h, rows, cols, X_h, nb, fn="mxfp4_mm"):
    Y = empty(nb * rows)
    getattr(mx, fn)(to_dev(w_h), rows, cols, to_dev(X_h), nb, Y)
    return host(Y).reshape(nb, rows)


# --- decode ------------------------------------------------------------------

def test_decode_tiny_config_bit_exact(mx):
    cfg = synth.TINY
    w_h = cfg.weights()
    out = empty(cfg.rows * cfg.cols)
    mx.mxfp4_dequant(to_dev(w_h), cfg.rows, cfg.cols, out)
    assert_bits_equal(host(out), oracle.dequant(w_h, cfg.rows, cfg.cols), "tiny decode")


def test_decode_exhaustive_code_by_scale(mx):
    codes = np.tile(np.concatenate([np.arange(16), np.arange(16)]), (256, 1))
    scales = np.arange(256).reshape(256, 1)
    buf = encode(codes, scales)
    out = empty(256 * 32)
    mx.mxfp4_dequant(to_dev(buf), 256, 32, out)
    got = host(out)
    assert_bits_equal(got, oracle.dequant(buf, 256, 32), "16x256 table")
    assert np.signbit(got[127 * 32 + 8]) and got[127 * 32 + 8] == 0.0  # code 8 -> -0.0


@pytest.mark.parametrize("name", ["decode", "mm8", "prefill"])
def test_decode_full_size_planes_bit_exact(mx, name):
    cfg = synth.CONFIGS[name]
    w_h = cfg.weights()
    out = empty(cfg.rows * cfg.cols)
    mx.mxfp4_dequant(to_dev(w_h), cfg.rows, cfg.cols, out)
    assert_bits_equal(host(out), oracle.dequant(w_h, cfg.rows, cfg.cols), name)


def test_decode_moe_expert_bit_exact(mx):
    cfg = synth.MOE
    w_h = synth.mxfp4_matrix(cfg.inter, cfg.hidden, synth.substream(cfg.seed, "gate/7"),
                             cfg.scale_lo, cfg.scale_hi)
    out = empty(cfg.inter * cfg.hidden)
    mx.mxfp4_dequant(to_dev(w_h), cfg.inter, cfg.hidden, out)
    assert_bits_equal(host(out), oracle.dequant(w_h, cfg.inter, cfg.hidden), "expert")


# --- matvec ------------------------------------------------------------------

def test_mv_tiny_config_with_subnormal_and_nan_groups(mx):
    cfg = synth.TINY
    w_h, x_h = cfg.weights(), cfg.activations()
    got = run_mv(mx, w_h, cfg.rows, cfg.cols, x_h)
    ref, l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, x_h, 1)
    assert np.isnan(got[250]) and not np.isnan(np.delete(got, 250)).any()
    assert_within(got, ref, l1, REL_FP32, "tiny mv")


def test_mv_decode_config_every_row(mx):
    cfg = synth.DECODE
    w_h, x_h = cfg.weights(), cfg.activations()
    got = run_mv(mx, w_h, cfg.rows, cfg.cols, x_h)
    ref, l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, x_h, 1)
    worst = assert_within(got, ref, l1, REL_FP32, "decode GEMV")
    print(f"decode GEMV worst err/tol {worst:.3g}")


@pytest.mark.parametrize("rows,cols", [(40, 256), (300, 2304), (5, 5120), (33, 64)])
def test_mv_exact_inputs_bit_for_bit(mx, rows, cols):
    # integer x in [-4, 4], scales 126..128: every FP32 partial sum is exact, so
    # any summation order gives exactly the oracle's double result.
    rng = np.random.default_rng(rows + cols)
    codes, scales = random_case(rng, rows, cols, lo=126, hi=128)
    buf = encode(codes, scales)
    x = synth.int_activations(rows * 7 + cols, cols)
    got = run_mv(mx, buf, rows, cols, x)
    ref, _ = oracle.matmat(buf, rows, cols, x, 1)
    assert np.array_equal(got.astype(np.float64), ref[0])


def test_mv_one_hot_sweep_pins_every_nibble_and_scale(mx):
    rows, cols = 64, 256
    rng = np.random.default_rng(1)
    codes, scales = random_case(rng, rows, cols, lo=100, hi=150)
    buf = encode(codes, scales)
    dense = oracle.dequant(buf, rows, cols)
    w = to_dev(buf)
    X = np.eye(cols, dtype=np.float32)
    Y = empty(cols * rows)
    mx.mxfp4_mm_fp32(w, rows, cols, to_dev(X), cols, Y)   # token c = unit vector e_c
    got = host(Y).reshape(cols, rows)
    # one non-zero product per output: exact, but a sum that starts at +0
    # returns +0 for a -0 weight (code 8), so compare values, not sign bits
    assert np.array_equal(got, dense.T), "one-hot sweep"


@pytest.mark.parametrize("rows,cols", [(300, 2304), (70000, 64), (5, 5120)])
def test_page_shapes_mv_and_batches_equal_per_token(mx, rows, cols):
    seed = rows + cols
    w_h = synth.mxfp4_matrix(rows, cols, seed, 119, 123, scale_pattern="adjacent_distinct")
    x1 = synth.normal_f32(seed, cols)
    got = run_mv(mx, w_h, rows, cols, x1)
    ref, l1 = oracle.matmat(w_h, rows, cols, x1, 1)
    assert_within(got, ref, l1, REL_FP32, f"{rows}x{cols} mv")
    if rows > 1000 and cols < 128:
        batches = [9]
    else:
        batches = [2, 8, 9, 19]
    for b in batches:
        X = synth.normal_f32(seed * 31 + b, b * cols).reshape(b, cols)
        Y = run_mm(mx, w_h, rows, cols, X, b)
        Y32 = run_mm(mx, w_h, rows, cols, X, b, "mxfp4_mm_fp32")
        ref, l1 = oracle.matmat(w_h, rows, cols, X, b)
        assert_within(Y, ref, l1, REL_FP32, f"{rows}x{cols} batch {b}")
        assert_within(Y32, ref, l1, REL_FP32, f"{rows}x{cols} batch {b} (FP32 path)")
        for t in range(b):
            # per token, each batch path equals its own matvec bit for bit: the
            # FP32 path with nb = 1, and mxfp4_mm (whatever the rest of its
            # batch) equals mxfp4_mv
            one32 = run_mm(mx, w_h, rows, cols, X[t:t + 1], 1, "mxfp4_mm_fp32")
            assert_bits_equal(Y32[t], one32[0], f"FP32 batch {b} token {t} vs its matvec")
            one = run_mv(mx, w_h, rows, cols, X[t])
            assert_bits_equal(Y[t], one, f"batch {b} token {t} vs its matvec")


def test_mm8_config_every_output(mx):
    cfg = synth.MM8
    w_h, X = cfg.weights(), cfg.activations()
    Y = run_mm(mx, w_h, cfg.rows, cfg.cols, X, cfg.nb)
    ref, l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, X, cfg.nb)
    worst = assert_within(Y, ref, l1, REL_FP32, "mm nb=8")
    print(f"mm nb=8 worst err/tol {worst:.3g}")
    # one pass decodes each group once for all eight tokens; per token the
    # result is still the matvec's, bit for bit
    for t in range(cfg.nb):
        assert_bits_equal(Y[t], run_mv(mx, w_h, cfg.rows, cfg.cols, X[t]), f"mm8 token {t}")


@pytest.mark.parametrize("nb", [5, 6, 7, 8, 16, 21])
def test_eight_token_passes_equal_the_matvec(mx, nb):
    # five to eight tokens share one pass; more tokens take passes of eight
    rows, cols = 160, 4096
    w_h = synth.mxfp4_matrix(rows, cols, 800 + nb, 118, 130)
    X = synth.normal_f32(810 + nb, nb * cols).reshape(nb, cols)
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    assert_within(Y, ref, l1, REL_FP32, f"nb={nb}")
    for t in range(nb):
        assert_bits_equal(Y[t], run_mv(mx, w_h, rows, cols, X[t]), f"nb={nb} token {t}")


@pytest.mark.parametrize("nb", [1, 3, 5, 8, 13])
def test_mm_wide_dynamic_range_activations(mx, nb):
    # activations spanning ~2^-60 .. 2^60 inside every group, plus an all-zero
    # group: the per-(token, group) prescale of the tensor-core path must keep
    # every group's small elements
    rows, cols = 200, 1024
    w_h = synth.mxfp4_matrix(rows, cols, 40 + nb, 118, 130)
    base = synth.normal_f32(70 + nb, nb * cols).astype(np.float64)
    expo = synth.uniform_int(80 + nb, nb * cols, -60, 60)
    X = (base * np.exp2(expo)).astype(np.float32).reshape(nb, cols)
    X[:, 64:96] = 0.0
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    assert_within(Y, ref, l1, REL_FP32, f"wide range nb={nb}")


@pytest.mark.parametrize("nb", [1, 8])
def test_mm_error_floor_of_an_outlier_activation(mx, nb):
    # one element of 2^60 among N(0, 1) values: x * 2^p puts the N(0, 1) part
    # below the f16 subnormal spacing, so rows whose weight is zero where x
    # peaks lose it and exceed 1e-5 * L1; the stated bound adds 2^-39 * max|x|
    # * sum_c |w[r][c]| and holds everywhere
    rows, cols = 256, 512
    w_h = synth.mxfp4_matrix(rows, cols, 90 + nb, 118, 130)
    X = synth.normal_f32(91 + nb, nb * cols).reshape(nb, cols)
    X[:, 17] = np.float32(2.0 ** 60)
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    ref, l1 = ref.reshape(nb, rows), l1.reshape(nb, rows)
    wsum = np.abs(oracle.dequant(w_h, rows, cols)).sum(axis=1)
    floor = 2.0 ** -39 * np.abs(X).max(axis=1, keepdims=True) * wsum[None, :]
    err = np.abs(Y.astype(np.float64) - ref)
    assert (err <= REL_FP32 * l1 + floor).all(), f"worst {np.max(err / (REL_FP32 * l1 + floor)):.3g}"
    assert (err > REL_FP32 * l1).any()


@pytest.mark.parametrize("nb", [1, 8, 11])
def test_mm_wide_weight_scales(mx, nb):
    # scale bytes over 0..240 inside every row, rows whose largest-scale group
    # holds only zero codes, and rows with one NaN group: the tensor-core path
    # folds each group's scale into its f16 weights relative to the row's
    # largest scale byte, so groups far below it must still count in full
    rows, cols = 300, 2048
    rng = np.random.default_rng(500 + nb)
    codes, scales = random_case(rng, rows, cols, lo=0, hi=240)
    scales[:60] = rng.integers(90, 110, size=(60, cols // 32))
    scales[:60, 5] = 240
    codes[:60, 160:192] = rng.choice([0, 8], size=(60, 32))   # zero codes in group 5
    scales[100, 17] = 255
    buf = encode(codes, scales)
    X = synth.normal_f32(600 + nb, nb * cols).reshape(nb, cols)
    ref, l1 = oracle.matmat(buf, rows, cols, X, nb)
    for fn in ("mxfp4_mm", "mxfp4_mm_fp32"):
        Y = run_mm(mx, buf, rows, cols, X, nb, fn)
        assert np.isnan(Y[:, 100]).all()
        assert_within(Y, ref, l1, REL_FP32, f"wide weight scales nb={nb} {fn}")


@pytest.mark.parametrize("rows,cols,nb", [(50, 544, 3), (33, 32, 8), (17, 160, 2), (131, 2880, 8),
                                          (64, 96, 1)])
def test_mm_ragged_shapes(mx, rows, cols, nb):
    # group counts that do not split evenly over the CTAs of a cluster (or are
    # fewer than its CTAs), and row counts that are not multiples of 16
    w_h = synth.mxfp4_matrix(rows, cols, rows + cols + nb, 118, 130)
    X = synth.normal_f32(rows * 3 + nb, nb * cols).reshape(nb, cols)
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    assert_within(Y, ref, l1, REL_FP32, f"{rows}x{cols} nb={nb}")


def test_mm_exact_inputs_bit_for_bit(mx):
    rows, cols, nb = 96, 1024, 8
    rng = np.random.default_rng(5)
    codes, scales = random_case(rng, rows, cols, lo=126, hi=128)
    buf = encode(codes, scales)
    X = synth.int_activations(17, nb * cols).reshape(nb, cols)
    Y = run_mm(mx, buf, rows, cols, X, nb)
    ref, _ = oracle.matmat(buf, rows, cols, X, nb)
    assert np.array_equal(Y.astype(np.float64), ref)


def test_zero_activation_gives_zero_except_nan_rows(mx):
    cfg = synth.TINY
    w_h = cfg.weights()
    got = run_mv(mx, w_h, cfg.rows, cfg.cols, np.zeros(cfg.cols, np.float32))
    assert np.isnan(got[250])
    assert not np.delete(got, 250).any()


def test_results_are_deterministic(mx):
    cfg = synth.DECODE
    w, x = to_dev(cfg.weights()), to_dev(cfg.activations())
    outs = []
    for _ in range(3):
        y = empty(cfg.rows)
        mx.mxfp4_mv(w, cfg.rows, cfg.cols, x, y)
        outs.append(host(y))
    assert_bits_equal(outs[0], outs[1]) and assert_bits_equal(outs[0], outs[2])


def test_refusals_launch_nothing(mx):
    import torch
    w = to_dev(synth.TINY.weights())
    x = to_dev(np.ones(2304, np.float32))
    y = torch.full((300,), 7.0, device="cuda:0")
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_mv(w, 300, 2270, x, y)      # cols not a multiple of 32
    assert e.value.status == 1
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_mv(w, 300, 2304, x[1:], y)  # misaligned x
    assert e.value.status == 2
    assert (host(y) == 7.0).all()


def test_host_buffer_entry_matches_device_entry(mx):
    import torch
    cfg = synth.TINY
    w_h, x_h = cfg.weights(), cfg.activations()
    w = to_dev(w_h)
    y_dev_ref = empty(cfg.rows)
    mx.mxfp4_mv(w, cfg.rows, cfg.cols, to_dev(x_h), y_dev_ref)
    X_host = torch.from_numpy(x_h.copy()).pin_memory()
    Y_host = torch.empty(cfg.rows, dtype=torch.float32).pin_memory()
    mx.mxfp4_matmat_host(w, cfg.rows, cfg.cols, X_host, 1, Y_host, empty(cfg.cols),
                         empty(cfg.rows))
    assert_bits_equal(Y_host.numpy(), host(y_dev_ref), "host entry")


@pytest.mark.parametrize("nb", [1, 3, 8])
def test_launch_overlap_chain_is_bit_identical(mx, nb):
    # four layers, each reading the previous one's output: with programmatic
    # dependent launch a kernel starts early but must read its x only after the
    # previous kernel has written it, so the chain's results are the same bits
    n = 1024
    ws = [to_dev(synth.mxfp4_matrix(n, n, 900 + i, 118, 130)) for i in range(4)]
    x0 = to_dev(synth.normal_f32(950 + nb, nb * n))

    def chain():
        import torch
        outs, x = [], x0
        for w in ws:
            y = empty(nb * n)
            if nb == 1:
                mx.mxfp4_mv(w, n, n, x, y)
            else:
                mx.mxfp4_mm(w, n, n, x, nb, y)
            # keep magnitudes moderate between layers (a kernel of our own
            # would do; torch's scale runs between the launches anyway)
            x = y * (1.0 / 64.0)
            outs.append(y)
        torch.cuda.synchronize()
        return [host(o) for o in outs]

    mx.mxfp4_set_launch_overlap(False)
    want = chain()
    try:
        mx.mxfp4_set_launch_overlap(True)
        got = chain()
    finally:
        mx.mxfp4_set_launch_overlap(False)
    for i, (g, w_) in enumerate(zip(got, want)):
        assert_bits_equal(g, w_, f"layer {i} with launch overlap, nb={nb}")


def test_launch_overlap_back_to_back_matvecs(mx):
    # layers launched directly one after another (no other kernel in between):
    # each reads the previous layer's output as its x
    n = 1024
    ws = [to_dev(synth.mxfp4_matrix(n, n, 960 + i, 100, 104)) for i in range(6)]
    x0 = to_dev(synth.normal_f32(970, n))

    def chain():
        ys = [empty(n) for _ in ws]
        x = x0
        for w, y in zip(ws, ys):
            mx.mxfp4_mv(w, n, n, x, y)
            x = y
        return [host(y) for y in ys]

    mx.mxfp4_set_launch_overlap(False)
    want = chain()
    try:
        mx.mxfp4_set_launch_overlap(True)
        got = chain()
    finally:
        mx.mxfp4_set_launch_overlap(False)
    for i, (g, w_) in enumerate(zip(got, want)):
        assert_bits_equal(g, w_, f"back-to-back layer {i} with launch overlap")


@pytest.mark.parametrize("nb", [1, 2, 8])
def test_rows_too_wide_for_the_matvec_kernel(mx, nb):
    # 1152 groups per row: more than a cluster of eight k_mv_tc CTAs stages, so
    # mxfp4_mv and mxfp4_mm run the cluster split-K kernel k_mma_small
    rows, cols = 64, 36864
    w_h = synth.mxfp4_matrix(rows, cols, 700 + nb, 118, 130)
    X = synth.normal_f32(710 + nb, nb * cols).reshape(nb, cols)
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    assert_within(Y, ref, l1, REL_FP32, f"{rows}x{cols} nb={nb}")
    for t in range(nb):
        assert_bits_equal(Y[t], run_mv(mx, w_h, rows, cols, X[t]), f"token {t} vs its matvec")


def test_rows_too_wide_for_both_tensor_kernels(mx):
    # 1728 groups per row: neither tensor-core kernel stages the row's
    # activations, so mxfp4_mv and mxfp4_mm take the FP32 path
    rows, cols, nb = 40, 55296, 3
    w_h = synth.mxfp4_matrix(rows, cols, 720, 118, 130)
    X = synth.normal_f32(721, nb * cols).reshape(nb, cols)
    Y = run_mm(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, X, nb)
    assert_within(Y, ref, l1, REL_FP32, f"{rows}x{cols} nb={nb}")
    for t in range(nb):
        y = run_mv(mx, w_h, rows, cols, X[t])
        assert_within(y, ref[t], l1[t], REL_FP32, f"{rows}x{cols} mv token {t}")
        assert_bits_equal(Y[t], y, f"token {t} vs its matvec")
