"""Helpers for the GPU parity tests: device transfer and the comparison rules
(bit-exact for decode with NaN compared by class; |got - ref| <= rel * L1 for
the floating-point products, a NaN reference requiring a NaN result)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

REL_FP32 = 1e-5      # FP32 paths: error relative to sum |w x|
REL_BF16 = 2e-2      # tensor-core path with bf16 activations


def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_dequant_matmul_gb300 as mx
    mx.lib()
    return mx


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def empty(n, dtype=torch.float32):
    return torch.empty(int(n), dtype=dtype, device="cuda:0")


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_bits_equal(got, want, what=""):
    got = np.asarray(got, dtype=np.float32).reshape(-1)
    want = np.asarray(want, dtype=np.float32).reshape(-1)
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    diff = np.flatnonzero(got[~gn].view(np.uint32) != want[~wn].view(np.uint32))
    assert diff.size == 0, f"{what}: {diff.size} elements differ, first at {diff[:5]}"


def assert_within(got, ref, l1, rel, what=""):
    """|got - ref| <= rel * l1 (+1e-30), NaN where ref is NaN."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    l1 = np.asarray(l1, dtype=np.float64).reshape(-1)
    rn = np.isnan(ref)
    assert np.array_equal(np.isnan(got), rn), f"{what}: NaN positions differ"
    err = np.abs(got[~rn] - ref[~rn])
    tol = rel * l1[~rn] + 1e-30
    bad = np.flatnonzero(err > tol)
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert bad.size == 0, (f"{what}: {bad.size} of {err.size} over tolerance; worst "
                           f"err/tol {worst:.3g}")
    return worst
