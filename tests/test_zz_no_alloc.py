"""The routed-expert layer entry point that allocates nothing
(mxfp4_moe_layer_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory when they run the layer
(all of their device memory belongs to their own pool allocator, or they must
not call cudaMalloc once running because it can block the device).  Its
scratch is a fixed array inside the library, shared by every call, so this
test makes two calls in a row with different inputs -- the second one finds
the first one's leftovers in the array -- and checks each against the
workspace entry points (mxfp4_moe_gate_up + mxfp4_moe_down) within the suite's
FP32 tolerance.  The file is named to run last: it must pass alone in a fresh
process and after every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import REL_FP32, assert_within, cuda, empty, host, to_dev

pytestmark = pytest.mark.gpu


def _case(seed, E=8, hidden=256, inter=192, T=12, K=3):
    cfg = synth.MoeConfig("noalloc case", E, hidden, inter, T, K, seed)
    gate, up, down = cfg.banks()
    ids, wts = cfg.routes()
    return cfg, gate, up, down, cfg.activations(), ids.astype(np.int32), wts


def _with_workspace(mx, cfg, d):
    P = cfg.n_tokens * cfg.top_k
    nbytes = mx.mxfp4_moe_workspace_bytes(cfg.n_experts, cfg.n_tokens, cfg.top_k, cfg.hidden,
                                          cfg.inter)
    ws = empty(nbytes // 4 + 4)
    act = empty(P * cfg.inter)
    y = empty(cfg.n_tokens * cfg.hidden)
    mx.mxfp4_moe_gate_up(d["gate"], d["up"], cfg.n_experts, cfg.hidden, cfg.inter, d["x"],
                         cfg.n_tokens, cfg.top_k, d["ids"], act, ws)
    mx.mxfp4_moe_down(d["down"], cfg.n_experts, cfg.hidden, cfg.inter, act, cfg.n_tokens,
                      cfg.top_k, d["ids"], d["wts"], y, ws)
    return host(y)


def test_noalloc_layer_matches_the_workspace_entry_points_on_two_calls():
    import torch
    mx = cuda()
    for seed in (31, 32):          # two calls in a row, different inputs
        cfg, gate, up, down, x, ids, wts = _case(seed)
        d = {"gate": to_dev(gate), "up": to_dev(up), "down": to_dev(down), "x": to_dev(x),
             "ids": to_dev(ids), "wts": to_dev(wts)}
        want = _with_workspace(mx, cfg, d)
        y = torch.full((cfg.n_tokens * cfg.hidden,), float("nan"), device="cuda:0")
        status = mx.lib().mxfp4_moe_layer_noalloc(
            d["gate"].data_ptr(), d["up"].data_ptr(), d["down"].data_ptr(), cfg.n_experts,
            cfg.hidden, cfg.inter, d["x"].data_ptr(), cfg.n_tokens, cfg.top_k,
            d["ids"].data_ptr(), d["wts"].data_ptr(), y.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert status == 0, mx.mxfp4_status_string(status)
        got = host(y)
        ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, cfg.n_experts,
                                 cfg.hidden, cfg.inter, x, cfg.n_tokens, cfg.top_k, ids, wts)
        bound = ref["bound_l1"] + ref["bound_prop"]
        assert_within(got, want, bound, REL_FP32, f"no-alloc call (seed {seed}) vs workspace")


def test_noalloc_layer_refuses_problems_larger_than_its_array():
    mx = cuda()
    A = 1 << 20   # never dereferenced: the size check comes first
    # 64 tokens x top-4 x inter 8192 floats of act alone is 8 MiB > 4 MiB
    status = mx.lib().mxfp4_moe_layer_noalloc(A, A, A, 8, 256, 8192, A, 64, 4, A, A, A, None)
    assert status == 4, mx.mxfp4_status_string(status)
