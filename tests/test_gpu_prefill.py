"""GPU parity of the large-batch (prefill) product: W decoded exactly, X rounded
to nearest-even bfloat16, FP32 accumulation, against the oracle on bf16(X)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import REL_BF16, REL_FP32, assert_within, cuda, empty, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    return cuda()


def run(mx, fn, w_h, rows, cols, X, nb):
    Y = empty(nb * rows)
    getattr(mx, fn)(to_dev(w_h), rows, cols, to_dev(X), nb, Y)
    return host(Y).reshape(nb, rows)


@pytest.mark.parametrize("rows,cols,nb", [(256, 512, 100), (300, 2304, 77), (64, 64, 129),
                                          (130, 4096, 65), (96, 160, 1)])
def test_bf16_path_small_shapes(mx, rows, cols, nb):
    seed = rows * 3 + cols + nb
    w_h = synth.mxfp4_matrix(rows, cols, seed, 118, 130)
    X = synth.normal_f32(seed, nb * cols).reshape(nb, cols)
    Y = run(mx, "mxfp4_mm_bf16", w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, oracle.round_bf16(X), nb)
    assert_within(Y, ref, l1, REL_BF16, "bf16 path")
    # the products are exact and only the FP32 sums round: the FP32 bound holds too
    assert_within(Y, ref, l1, REL_FP32, "bf16 path, FP32 bound")


def test_mm_dispatches_large_batches_to_the_bf16_path(mx):
    rows, cols, nb = 128, 1024, 96
    w_h = synth.mxfp4_matrix(rows, cols, 3, 118, 130)
    X = synth.normal_f32(8, nb * cols).reshape(nb, cols)
    a = run(mx, "mxfp4_mm", w_h, rows, cols, X, nb)
    b = run(mx, "mxfp4_mm_bf16", w_h, rows, cols, X, nb)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_bf16_path_tiny_config_nan_and_subnormal_groups(mx):
    cfg = synth.TINY
    w_h = cfg.weights()
    nb = 80
    X = synth.normal_f32(12, nb * cfg.cols).reshape(nb, cfg.cols)
    Y = run(mx, "mxfp4_mm_bf16", w_h, cfg.rows, cfg.cols, X, nb)
    ref, l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, oracle.round_bf16(X), nb)
    assert np.isnan(Y[:, 250]).all()
    assert_within(Y, ref, l1, REL_BF16, "tiny bf16")


def test_bf16_path_exact_inputs_bit_for_bit(mx):
    rows, cols, nb = 256, 1024, 192
    w_h = synth.mxfp4_matrix(rows, cols, 21, 126, 128)
    X = synth.int_activations(4, nb * cols).reshape(nb, cols)    # exact in bf16
    Y = run(mx, "mxfp4_mm_bf16", w_h, rows, cols, X, nb)
    ref, _ = oracle.matmat(w_h, rows, cols, X, nb)
    assert np.array_equal(Y.astype(np.float64), ref)


def test_prefill_config_sampled_outputs(mx):
    cfg = synth.PREFILL
    w_h, X = cfg.weights(), cfg.activations()
    Y = run(mx, "mxfp4_mm", w_h, cfg.rows, cfg.cols, X, cfg.nb)
    rng = np.random.default_rng(0)
    n = 3000
    tok = np.concatenate([rng.integers(0, cfg.nb, n - 2), [0, cfg.nb - 1]]).astype(np.int32)
    row = np.concatenate([rng.integers(0, cfg.rows, n - 2), [0, cfg.rows - 1]]).astype(np.int32)
    ref, l1 = oracle.matmat_samples(w_h, cfg.rows, cfg.cols, oracle.round_bf16(X), tok, row)
    assert_within(Y[tok, row], ref, l1, REL_BF16, "prefill samples")
    worst = assert_within(Y[tok, row], ref, l1, REL_FP32, "prefill samples, FP32 bound")
    # against the unrounded activations: the bf16 rounding of X is the only gap
    ref32, _ = oracle.matmat_samples(w_h, cfg.rows, cfg.cols, X, tok, row)
    nrmse = np.sqrt(((Y[tok, row] - ref32) ** 2).sum() / (ref32 ** 2).sum())
    print(f"prefill worst err/tol {worst:.3g}; nrmse vs f32-X oracle {nrmse:.3e}")
    assert nrmse < 1e-2


def run_ws(mx, w_h, rows, cols, X, nb):
    import torch
    Y = empty(nb * rows)
    nbytes = mx.mxfp4_mm_bf16_workspace_bytes(rows, cols, nb)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    mx.mxfp4_mm_bf16_ws(to_dev(w_h), rows, cols, to_dev(X), nb, Y, ws)
    return host(Y).reshape(nb, rows)


@pytest.mark.parametrize("rows,cols,nb", [(256, 512, 100), (300, 2304, 77), (64, 64, 129),
                                          (130, 4096, 65), (96, 160, 1)])
def test_dense_after_dequant_small_shapes(mx, rows, cols, nb):
    seed = rows * 5 + cols + nb
    w_h = synth.mxfp4_matrix(rows, cols, seed, 118, 130)
    X = synth.normal_f32(seed, nb * cols).reshape(nb, cols)
    Y = run_ws(mx, w_h, rows, cols, X, nb)
    ref, l1 = oracle.matmat(w_h, rows, cols, oracle.round_bf16(X), nb)
    assert_within(Y, ref, l1, REL_BF16, "dense after dequant")
    assert_within(Y, ref, l1, REL_FP32, "dense after dequant, FP32 bound")


def test_dense_after_dequant_nan_subnormal_and_exact_inputs(mx):
    cfg = synth.TINY
    w_h = cfg.weights()
    X = synth.normal_f32(13, 80 * cfg.cols).reshape(80, cfg.cols)
    Y = run_ws(mx, w_h, cfg.rows, cfg.cols, X, 80)
    ref, l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, oracle.round_bf16(X), 80)
    assert np.isnan(Y[:, 250]).all()
    assert_within(Y, ref, l1, REL_BF16, "tiny dense")
    rows, cols, nb = 256, 1024, 192
    w_h = synth.mxfp4_matrix(rows, cols, 22, 126, 128)
    X = synth.int_activations(5, nb * cols).reshape(nb, cols)    # exact in bf16
    Y = run_ws(mx, w_h, rows, cols, X, nb)
    ref, _ = oracle.matmat(w_h, rows, cols, X, nb)
    assert np.array_equal(Y.astype(np.float64), ref)


def test_dense_after_dequant_prefill_config_samples_and_short_workspace(mx):
    import torch
    cfg = synth.PREFILL
    w_h, X = cfg.weights(), cfg.activations()
    Y = run_ws(mx, w_h, cfg.rows, cfg.cols, X, cfg.nb)
    rng = np.random.default_rng(1)
    n = 2000
    tok = np.concatenate([rng.integers(0, cfg.nb, n - 2), [0, cfg.nb - 1]]).astype(np.int32)
    row = np.concatenate([rng.integers(0, cfg.rows, n - 2), [0, cfg.rows - 1]]).astype(np.int32)
    ref, l1 = oracle.matmat_samples(w_h, cfg.rows, cfg.cols, oracle.round_bf16(X), tok, row)
    assert_within(Y[tok, row], ref, l1, REL_FP32, "prefill dense samples")
    # a workspace one byte short is refused and nothing runs
    nbytes = mx.mxfp4_mm_bf16_workspace_bytes(64, 512, 8)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    w_small = to_dev(synth.mxfp4_matrix(64, 512, 3, 118, 130))
    x_small = to_dev(synth.normal_f32(3, 8 * 512))
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_mm_bf16_ws(w_small, 64, 512, x_small, 8, empty(8 * 64), ws, nbytes - 1)


@pytest.mark.parametrize("fn", ["mxfp4_mm", "mxfp4_mm_bf16_ws"])
def test_prefill_config_full_token_bands(mx, fn):
    # every output of the first and the last 128-token band (one tile row of
    # the tensor-core kernels) over all 4096 rows: every epilogue position of
    # every weight tile.  The reference is the oracle's exact decode followed
    # by a float64 matrix product (numpy standing for the oracle's double dot
    # products, checked against oracle.matmat on a row window below).
    cfg = synth.PREFILL
    w_h, X = cfg.weights(), cfg.activations()
    if fn == "mxfp4_mm":
        Y = run(mx, fn, w_h, cfg.rows, cfg.cols, X, cfg.nb)
    else:
        Y = run_ws(mx, w_h, cfg.rows, cfg.cols, X, cfg.nb)
    Wd = oracle.dequant(w_h, cfg.rows, cfg.cols).astype(np.float64)
    for t0 in (0, cfg.nb - 128):
        Xb = oracle.round_bf16(X[t0:t0 + 128])
        ref = Xb.astype(np.float64) @ Wd.T
        l1 = np.abs(Xb.astype(np.float64)) @ np.abs(Wd).T
        win, win_l1 = oracle.matmat(w_h, cfg.rows, cfg.cols, Xb, 128, 1000, 1004)
        np.testing.assert_allclose(ref[:, 1000:1004], win, rtol=0, atol=1e-12 * win_l1.max())
        assert_within(Y[t0:t0 + 128], ref, l1, REL_BF16, f"{fn} band {t0}")
        assert_within(Y[t0:t0 + 128], ref, l1, REL_FP32, f"{fn} band {t0}, FP32 bound")


def test_mm_large_batches_workspace_per_stream_and_under_capture(mx):
    # mxfp4_mm's large batches convert W and X to bf16 once into a workspace
    # the library keeps per stream; where none can be had (a stream captured
    # before any eager call) the conversion runs inside the GEMM.  Every way
    # gives the same bits as mxfp4_mm_bf16.
    import torch
    rows, cols = 256, 1024
    w_h = synth.mxfp4_matrix(rows, cols, 11, 118, 130)
    wd = to_dev(w_h)
    for nb in (70, 100):   # the second size grows the workspaces made by the first
        X = synth.normal_f32(12 + nb, nb * cols).reshape(nb, cols)
        xd = to_dev(X)
        ref = run(mx, "mxfp4_mm_bf16", w_h, rows, cols, X, nb)
        fresh = torch.cuda.Stream()
        Y_cap = empty(nb * rows)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=fresh):
            mx.mxfp4_mm(wd, rows, cols, xd, nb, Y_cap)
        g.replay()
        outs = [Y_cap]
        for st in (torch.cuda.Stream(), torch.cuda.current_stream()):
            Y = empty(nb * rows)
            with torch.cuda.stream(st):
                mx.mxfp4_mm(wd, rows, cols, xd, nb, Y)
            outs.append(Y)
        torch.cuda.synchronize()
        for Y in outs:
            got = host(Y).reshape(nb, rows)
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
