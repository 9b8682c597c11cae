"""GPU parity of the general routed-expert passes (mxfp4_moe_gate_up_ex /
mxfp4_moe_down_ex) against the oracle's global-bank layer: the DeepSeek-V4.1
mode of "cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs" (GLOBAL kernels with their
bf16 flag: gate, up, act and output rounded to bfloat16, the route weight
folded into the act), the SwiGLU limit, the expert -> slot table with cold
experts, and the page's global-bank MoE test case: four routed experts plus a
shared one, three routes, the last with a cold winner."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_within, cuda, empty, host, to_dev

pytestmark = pytest.mark.gpu

V41 = 1
F32 = 0


@pytest.fixture(scope="module")
def mx():
    return cuda()


def run_ex(mx, cfg, gate, up, down, x, ids, wts, mode, limit, slot_of=None, n_experts=None,
           n_slots=None):
    T, K = ids.shape
    n_slots = cfg.n_experts if n_slots is None else n_slots
    n_experts = n_slots if n_experts is None else n_experts
    nbytes = mx.mxfp4_moe_workspace_bytes(n_slots, T, K, cfg.hidden, cfg.inter)
    ws = empty(nbytes // 4 + 4)
    act = empty(T * K * cfg.inter)
    y = empty(T * cfg.hidden)
    w_d = to_dev(wts)
    mx.mxfp4_moe_gate_up_ex(to_dev(gate), to_dev(up), n_slots, cfg.hidden, cfg.inter, to_dev(x),
                            T, K, to_dev(ids), act, ws,
                            slot_of=None if slot_of is None else to_dev(slot_of),
                            n_experts=n_experts, route_w=w_d, mode=mode, swiglu_limit=limit)
    mx.mxfp4_moe_down_ex(to_dev(down), n_slots, cfg.hidden, cfg.inter, act, T, K, y, ws,
                         route_w=w_d, mode=mode)
    cold = mx.mxfp4_moe_cold_pairs(ws, n_slots, T, K)
    return host(y).reshape(T, cfg.hidden), cold, ws


def check(y, ref, what, max_nrmse, bf16):
    assert_within(y, ref["out"], ref["bound"], 1.0, what)
    want = ref["out"]
    diff = y - want
    nrmse = np.sqrt((diff ** 2).sum() / (want ** 2).sum())
    cos = (y * want).sum() / np.sqrt((y ** 2).sum() * (want ** 2).sum())
    assert nrmse < max_nrmse and cos > 0.999, (what, nrmse, cos)
    if bf16:
        # the outputs are bfloat16 values, and almost all equal the oracle's
        assert (y.view(np.uint32) & 0xFFFF == 0).all(), what
        assert (y == want).mean() > 0.9, (what, (y == want).mean())
    return nrmse


@pytest.mark.parametrize("E,hidden,inter,T,K,seed,mode,limit", [
    (8, 256, 128, 12, 3, 41, V41, 0.0),
    (8, 256, 128, 12, 3, 42, V41, 0.5),
    (8, 256, 128, 12, 3, 43, F32, 0.5),
    (6, 4608, 64, 5, 2, 44, V41, 0.5),      # 144 groups per gate/up row: the FP32 passes
    (64, 2880, 2880, 32, 4, 3, V41, 10.0),  # the MoE layer's workload in the V4.1 mode
])
def test_layer_modes_against_the_oracle(mx, E, hidden, inter, T, K, seed, mode, limit):
    cfg = synth.MoeConfig("ex", E, hidden, inter, T, K, seed, scale_lo=113, scale_hi=121)
    gate, up, down = cfg.banks()
    x = cfg.activations()
    ids, wts = cfg.routes()
    y, cold, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, mode, limit)
    ref = oracle.moe_forward_ex(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                                x, T, K, ids, wts, bf16_mode=mode == V41, limit=limit)
    assert cold == []
    check(y, ref, f"mode {mode} limit {limit} {E}x{hidden}x{inter}", 0.02, mode == V41)


def test_f32_mode_without_limit_is_the_plain_layer(mx):
    cfg = synth.MoeConfig("ex", 8, 256, 128, 12, 3, 45)
    gate, up, down = cfg.banks()
    x = cfg.activations()
    ids, wts = cfg.routes()
    y, _, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, F32, 0.0)
    nbytes = mx.mxfp4_moe_workspace_bytes(8, 12, 3, 256, 128)
    ws = empty(nbytes // 4 + 4)
    act = empty(12 * 3 * 128)
    y0 = empty(12 * 256)
    mx.mxfp4_moe_gate_up(to_dev(gate), to_dev(up), 8, 256, 128, to_dev(x), 12, 3, to_dev(ids),
                         act, ws)
    mx.mxfp4_moe_down(to_dev(down), 8, 256, 128, act, 12, 3, to_dev(ids), to_dev(wts), y0, ws)
    assert np.array_equal(y.reshape(-1).view(np.uint32), host(y0).view(np.uint32))


def test_slot_table_permuted_bank_and_invalid_slots(mx):
    cfg = synth.MoeConfig("ex", 6, 256, 128, 10, 2, 46, scale_lo=113, scale_hi=121)
    gate, up, down = cfg.banks()
    x = cfg.activations()
    ids, wts = cfg.routes()
    y_id, _, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, V41, 0.5)
    perm = np.array([3, 0, 5, 1, 4, 2], dtype=np.int32)   # expert e in slot perm[e]
    inv = np.argsort(perm)

    def permute(bank, stride):
        return np.ascontiguousarray(bank.reshape(6, stride)[inv]).reshape(-1)

    pg, pu = permute(gate, cfg.gu_stride), permute(up, cfg.gu_stride)
    pd = permute(down, cfg.down_stride)
    y_p, cold, _ = run_ex(mx, cfg, pg, pu, pd, x, ids, wts, V41, 0.5, slot_of=perm)
    assert cold == [] and np.array_equal(y_p.view(np.uint32), y_id.view(np.uint32))
    # an entry pointing past the bank: those pairs are invalid (counted, not cold)
    bad = perm.copy()
    bad[ids[0, 0]] = 6
    y_b, cold, ws = run_ex(mx, cfg, pg, pu, pd, x, ids, wts, V41, 0.5, slot_of=bad)
    assert cold == [] and mx.mxfp4_moe_plan_errors(ws) == int((ids == ids[0, 0]).sum())
    ref = oracle.moe_forward_ex(pg, pu, pd, cfg.gu_stride, cfg.down_stride, 6, 256, 128, x, 10, 2,
                                ids, wts, slot_of=bad, n_experts=6, bf16_mode=True, limit=0.5)
    check(y_b, ref, "invalid slot", 0.02, True)


@pytest.mark.parametrize("dim,inter,limit,max_nrmse", [(128, 64, 0.5, 0.02),
                                                       (5120, 2304, 10.0, 0.01)])
def test_global_bank_frame_three_routes_with_a_cold_winner(mx, dim, inter, limit, max_nrmse):
    # four routed experts and a shared one (bank slot 4, routed to every token
    # with weight 1), top-2 routes: (0, 1), (2, 3), and (3, 0) with expert 0
    # cold -- its pair is listed and left out, the rest still computed
    cfg = synth.MoeConfig("frame", 5, dim, inter, 1, 3, 47, scale_lo=113, scale_hi=121)
    gate, up, down = cfg.banks()
    cases = [((0, 1), (0.25, 0.75), False), ((2, 3), (0.9, 0.1), False),
             ((3, 0), (0.6, 0.4), True)]
    for case, (picks, w2, cold_winner) in enumerate(cases):
        x = oracle.round_bf16(2.0 * synth.normal_f32(500 + case, dim)).reshape(1, dim)
        ids = np.array([[picks[0], picks[1], 4]], dtype=np.int32)
        wts = np.array([[w2[0], w2[1], 1.0]], dtype=np.float32)
        slot_of = np.arange(5, dtype=np.int32)
        if cold_winner:
            slot_of[picks[1]] = -1
        y, cold, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, V41, limit, slot_of=slot_of)
        ref = oracle.moe_forward_ex(gate, up, down, cfg.gu_stride, cfg.down_stride, 5, dim, inter,
                                    x, 1, 3, ids, wts, slot_of=slot_of, n_experts=5,
                                    bf16_mode=True, limit=limit)
        assert cold == ref["cold"].tolist() == ([1] if cold_winner else [])
        nrmse = check(y, ref, f"frame case {case}", max_nrmse, True)
        print(f"frame {dim}x{inter} case {case}: nrmse {nrmse:.3e}")


def test_many_cold_pairs_are_listed_in_order(mx):
    cfg = synth.MoeConfig("ex", 16, 64, 64, 40, 4, 48)
    gate, up, down = cfg.banks()
    x = cfg.activations()
    ids, wts = cfg.routes()
    slot_of = np.arange(16, dtype=np.int32)
    slot_of[[2, 5, 7, 11, 13]] = -1
    y, cold, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, F32, 0.0, slot_of=slot_of)
    want = np.flatnonzero(np.isin(ids.reshape(-1), [2, 5, 7, 11, 13])).tolist()
    assert cold == want and len(want) > 32     # more than one ballot round
    ref = oracle.moe_forward_ex(gate, up, down, cfg.gu_stride, cfg.down_stride, 16, 64, 64, x,
                                40, 4, ids, wts, slot_of=slot_of, n_experts=16)
    check(y, ref, "cold pairs", 1e-4, False)


def test_ex_refusals(mx):
    A = 1 << 20   # never dereferenced: the checks come first
    lib = mx.lib()
    # mode out of range, NaN limit, a table missing while ids and slots differ
    assert lib.mxfp4_moe_gate_up_ex(A, A, 8, 64, 64, A, 2, 2, A, None, 8, A, 2, 0.0, A, A,
                                    1 << 20, None) == 1
    assert lib.mxfp4_moe_gate_up_ex(A, A, 8, 64, 64, A, 2, 2, A, None, 8, A, 1, float("nan"), A,
                                    A, 1 << 20, None) == 1
    assert lib.mxfp4_moe_gate_up_ex(A, A, 8, 64, 64, A, 2, 2, A, None, 9, A, 1, 0.0, A, A,
                                    1 << 20, None) == 1
    # the V4.1 mode needs the route weights in the gate/up pass
    assert lib.mxfp4_moe_gate_up_ex(A, A, 8, 64, 64, A, 2, 2, A, None, 8, None, 1, 0.0, A, A,
                                    1 << 20, None) == 2


@pytest.mark.parametrize("n_seg,seg_slots,where", [
    (3, 2, [0, 1, 2, 3, 4]),            # five experts over segments 0, 0, 1, 1, 2
    (16, 2, [1, 3, 5, 7, 31]),          # sixteen segments, local index 1 of each
    (4, 3, [11, 2, 6, 9, 0]),           # any slot order
])
def test_segmented_bank_equals_the_one_buffer_bank(mx, n_seg, seg_slots, where):
    # each segment its own device buffer; expert e in slot where[e] (slot_of):
    # the result is the one-buffer bank's, bit for bit, in both passes and both
    # kernel families (128 groups per row: tensor cores; 144: the FP32 passes)
    import torch
    for hidden in (256, 4608):
        cfg = synth.MoeConfig("seg", 5, hidden, 64, 6, 3, 49, scale_lo=113, scale_hi=121)
        gate, up, down = cfg.banks()
        x = cfg.activations()
        ids, wts = cfg.routes()
        y_ref, _, _ = run_ex(mx, cfg, gate, up, down, x, ids, wts, V41, 0.5)
        n_slots = n_seg * seg_slots
        slot_of = np.array(where, dtype=np.int32)

        def segments(bank, stride):
            out = [torch.zeros(seg_slots * stride, dtype=torch.uint8, device="cuda:0")
                   for _ in range(n_seg)]
            for e, s in enumerate(where):
                out[s // seg_slots][(s % seg_slots) * stride:(s % seg_slots + 1) * stride] = \
                    to_dev(bank[e * stride:(e + 1) * stride])
            return out

        gs, us = segments(gate, cfg.gu_stride), segments(up, cfg.gu_stride)
        ds = segments(down, cfg.down_stride)
        T, K = ids.shape
        nbytes = mx.mxfp4_moe_workspace_bytes(n_slots, T, K, hidden, 64)
        ws = empty(nbytes // 4 + 4)
        act = empty(T * K * 64)
        y = empty(T * hidden)
        w_d = to_dev(wts)
        mx.mxfp4_moe_gate_up_seg(gs, us, seg_slots, hidden, 64, to_dev(x), T, K, to_dev(ids), act,
                                 ws, slot_of=to_dev(slot_of), n_experts=5, route_w=w_d, mode=V41,
                                 swiglu_limit=0.5)
        mx.mxfp4_moe_down_seg(ds, seg_slots, hidden, 64, act, T, K, y, ws, route_w=w_d, mode=V41)
        got = host(y).reshape(T, hidden)
        assert np.array_equal(got.view(np.uint32), y_ref.view(np.uint32)), (hidden, where)
