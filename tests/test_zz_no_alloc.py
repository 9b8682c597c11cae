"""The routed-expert layer entry point that allocates nothing
(mxfp4_moe_layer_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory when they run the layer
(all of their device memory belongs to their own pool allocator, or they must
not call cudaMalloc once running because it can block the device).  Its
scratch is a fixed array inside the library, shared by every call and keeping
the previous call's contents.  So this test runs a large problem and then a
small one -- the small call finds the large call's plan, activations and
per-pair outputs in the array past its own -- and checks every call against
the CPU oracle within the suite's FP32 tolerance, and that the small call
changes neither the device's free memory nor torch's allocations.  The file
is named to run last: it must pass alone in a fresh process and after every
other test.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import REL_FP32, assert_within, cuda, host, to_dev

pytestmark = pytest.mark.gpu

SMALL = dict(E=4, hidden=256, inter=128, T=3, K=2)
LARGE = dict(E=64, hidden=512, inter=384, T=32, K=4)
# the bench's MoE layer: its plan, fragment blocks, per-pair outputs and act take 4.8 MB
LAYER = dict(E=64, hidden=2880, inter=2880, T=32, K=4)


def _case(seed, E, hidden, inter, T, K):
    cfg = synth.MoeConfig("noalloc case", E, hidden, inter, T, K, seed)
    gate, up, down = cfg.banks()
    ids, wts = cfg.routes()
    return cfg, gate, up, down, cfg.activations(), ids.astype(np.int32), wts


def _call_and_check(mx, seed, shape, check_memory=False):
    import torch
    cfg, gate, up, down, x, ids, wts = _case(seed, **shape)
    d = {"gate": to_dev(gate), "up": to_dev(up), "down": to_dev(down), "x": to_dev(x),
         "ids": to_dev(ids), "wts": to_dev(wts)}
    y = torch.full((cfg.n_tokens * cfg.hidden,), float("nan"), device="cuda:0")
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    status = mx.lib().mxfp4_moe_layer_noalloc(
        d["gate"].data_ptr(), d["up"].data_ptr(), d["down"].data_ptr(), cfg.n_experts,
        cfg.hidden, cfg.inter, d["x"].data_ptr(), cfg.n_tokens, cfg.top_k,
        d["ids"].data_ptr(), d["wts"].data_ptr(), y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert status == 0, mx.mxfp4_status_string(status)
    if check_memory:
        assert free1 == free0, f"device free memory changed by {free1 - free0} bytes"
        assert alloc1 == alloc0, f"torch allocations changed by {alloc1 - alloc0} bytes"
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, cfg.n_experts,
                             cfg.hidden, cfg.inter, x, cfg.n_tokens, cfg.top_k, ids, wts)
    assert_within(host(y), ref["out"], ref["bound_l1"] + ref["bound_prop"], REL_FP32,
                  f"no-alloc layer (seed {seed}, {cfg.n_experts} experts, {cfg.n_tokens} tokens)")


def test_noalloc_layer_matches_the_oracle_large_then_small():
    mx = cuda()
    # the first call on the device looks up the array's address and loads the
    # kernels; the large call then fills more of the array than the small one
    # reads, and the second small call must neither see those leftovers nor
    # allocate anything
    _call_and_check(mx, 31, SMALL)
    _call_and_check(mx, 32, LARGE)
    _call_and_check(mx, 33, SMALL, check_memory=True)


def test_noalloc_layer_takes_the_bench_moe_shape():
    mx = cuda()
    assert (mx.mxfp4_moe_workspace_bytes(64, 32, 4, 2880, 2880) + 255) // 256 * 256 + \
        32 * 4 * 2880 * 4 <= mx.NOALLOC_SCRATCH_BYTES
    _call_and_check(mx, 3, LAYER, check_memory=True)


def test_noalloc_layer_refuses_problems_larger_than_its_array():
    mx = cuda()
    A = 1 << 20   # never dereferenced: the size check comes first
    # 64 tokens x top-4 x inter 32768 floats of act alone is 32 MiB > 16 MiB
    status = mx.lib().mxfp4_moe_layer_noalloc(A, A, A, 8, 256, 32768, A, 64, 4, A, A, A, None)
    assert status == 4, mx.mxfp4_status_string(status)
