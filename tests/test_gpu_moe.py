"""GPU parity of the routed-expert passes against the CPU oracle: gate/up alone,
down alone on an injected activation (the stage injection of the q4tp MoE
kernel's run_stages), and the whole layer; experts with 0, 1 and more than 8
pairs; distinct scale planes per expert; out-of-range ids."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import REL_FP32, assert_bits_equal, assert_within, cuda, empty, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    return cuda()


def make_case(E, hidden, inter, T, K, seed, ids=None):
    cfg = synth.MoeConfig("case", E, hidden, inter, T, K, seed)
    gate, up, down = cfg.banks()
    x = cfg.activations()
    rid, wts = cfg.routes() if ids is None else (ids, synth.routes(seed, T, K, E)[1])
    return cfg, gate, up, down, x, np.ascontiguousarray(rid, dtype=np.int32), wts


def act_tolerance(ref):
    """Error allowed in act = silu(g)*u when g and u each carry 1e-5 * L1 error,
    plus a few float roundings of the product."""
    g, u = ref["g"], ref["u"]
    s = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    dsilu = np.abs(s * (1.0 + g * (1.0 - s)))
    prop = dsilu * ref["l1g"] * np.abs(u) + np.abs(g * s) * ref["l1u"]
    return REL_FP32 * prop + 4.0 * 2.0 ** -23 * np.abs(ref["act"]) + 1e-30


def run_gate_up(mx, cfg, gate, up, x, ids, ws=None, act=None):
    P = cfg.n_tokens * cfg.top_k
    nbytes = mx.mxfp4_moe_workspace_bytes(cfg.n_experts, cfg.n_tokens, cfg.top_k,
                                          cfg.hidden, cfg.inter)
    ws = empty(nbytes // 4 + 4) if ws is None else ws
    act = empty(P * cfg.inter) if act is None else act
    mx.mxfp4_moe_gate_up(to_dev(gate), to_dev(up), cfg.n_experts, cfg.hidden, cfg.inter,
                         to_dev(x), cfg.n_tokens, cfg.top_k, to_dev(ids), act, ws)
    return act, ws


def check_gate_up(act_got, ref, ids, E):
    valid = ((ids >= 0) & (ids < E)).reshape(-1)
    got = act_got.reshape(ref["act"].shape)[valid]
    want = ref["act"][valid]
    tol = act_tolerance(ref)[valid]
    err = np.abs(got.astype(np.float64) - want)
    assert not np.isnan(got).any()
    bad = np.flatnonzero(err > tol)
    assert bad.size == 0, f"{bad.size} act values over tolerance, worst {np.max(err / tol):.3g}"


@pytest.mark.parametrize("E,hidden,inter,T,K,seed", [
    (8, 64, 96, 12, 3, 1),       # some experts with no pair
    (5, 256, 128, 16, 2, 2),
    (64, 2880, 2880, 32, 4, 3),  # the MoE layer's workload
])
def test_gate_up_stage(mx, E, hidden, inter, T, K, seed):
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, seed)
    act, _ = run_gate_up(mx, cfg, gate, up, x, ids)
    ref = oracle.moe_gate_up(gate, up, cfg.gu_stride, E, hidden, inter, x, T, K, ids)
    check_gate_up(host(act), ref, ids, E)


def test_gate_up_expert_with_more_than_eight_pairs(mx):
    E, hidden, inter, T, K = 6, 128, 64, 20, 2
    ids = np.stack([[0, 1 + t % 5] for t in range(T)]).astype(np.int32)  # expert 0: 20 pairs
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 5, ids)
    act, _ = run_gate_up(mx, cfg, gate, up, x, ids)
    ref = oracle.moe_gate_up(gate, up, cfg.gu_stride, E, hidden, inter, x, T, K, ids)
    check_gate_up(host(act), ref, ids, E)


def test_gate_up_and_layer_when_rows_are_too_wide_for_the_tensor_path(mx):
    # 144 groups per row of gate/up (more than the tensor-core passes stage):
    # those run the FP32 expert passes; the down pass (64 groups) stays on the
    # tensor cores
    E, hidden, inter, T, K = 4, 4608, 64, 6, 2
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 17)
    act, _ = run_gate_up(mx, cfg, gate, up, x, ids)
    ref = oracle.moe_gate_up(gate, up, cfg.gu_stride, E, hidden, inter, x, T, K, ids)
    check_gate_up(host(act), ref, ids, E)
    y, _ = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                             x, T, K, ids, wts)
    assert_within(y, ref["out"], ref["bound_l1"] + ref["bound_prop"], REL_FP32, "wide MoE layer")


@pytest.mark.parametrize("E,hidden,inter,T,K,seed", [
    (8, 96, 64, 12, 3, 7), (64, 2880, 2880, 32, 4, 3)])
def test_down_stage_on_injected_act(mx, E, hidden, inter, T, K, seed):
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, seed)
    act = synth.normal_f32(seed + 1000, T * K * inter)
    # plan from a gate/up call (its act output is then overwritten by the injected act)
    act_d, ws = run_gate_up(mx, cfg, gate, up, x, ids)
    act_d.copy_(to_dev(act))
    y = empty(T * hidden)
    mx.mxfp4_moe_down(to_dev(down), E, hidden, inter, act_d, T, K, to_dev(ids), to_dev(wts),
                      y, ws)
    ref = oracle.moe_down(down, cfg.down_stride, E, hidden, inter, act, T, K, ids, wts)
    assert_within(host(y), ref["out"], ref["l1_out"], REL_FP32, "down stage")


def run_layer(mx, cfg, gate, up, down, x, ids, wts):
    act, ws = run_gate_up(mx, cfg, gate, up, x, ids)
    y = empty(cfg.n_tokens * cfg.hidden)
    mx.mxfp4_moe_down(to_dev(down), cfg.n_experts, cfg.hidden, cfg.inter, act, cfg.n_tokens,
                      cfg.top_k, to_dev(ids), to_dev(wts), y, ws)
    return host(y).reshape(cfg.n_tokens, cfg.hidden), ws


@pytest.mark.parametrize("E,hidden,inter,T,K,seed", [
    (8, 64, 96, 12, 3, 11), (64, 2880, 2880, 32, 4, 3)])
def test_whole_layer(mx, E, hidden, inter, T, K, seed):
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, seed)
    y, _ = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                             x, T, K, ids, wts)
    bound = ref["bound_l1"] + ref["bound_prop"]
    assert_within(y, ref["out"], bound, REL_FP32, "MoE layer")
    diff = y - ref["out"]
    nrmse = np.sqrt((diff ** 2).sum() / (ref["out"] ** 2).sum())
    cos = (y * ref["out"]).sum() / np.sqrt((y ** 2).sum() * (ref["out"] ** 2).sum())
    assert nrmse < 1e-4 and cos > 0.999999, (nrmse, cos)


def test_layer_is_deterministic(mx):
    cfg, gate, up, down, x, ids, wts = make_case(16, 256, 256, 24, 4, 13)
    a, _ = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    b, _ = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    assert_bits_equal(a, b, "rerun")


def test_out_of_range_ids_are_skipped_and_counted(mx):
    import torch
    cfg, gate, up, down, x, ids, wts = make_case(8, 64, 64, 10, 2, 17)
    ids = ids.copy()
    ids[3, 1] = 8
    ids[6, 0] = -1
    P = cfg.n_tokens * cfg.top_k
    act = torch.full((P * cfg.inter,), 123.0, device="cuda:0")
    act, ws = run_gate_up(mx, cfg, gate, up, x, ids, act=act)
    assert mx.mxfp4_moe_plan_errors(ws) == 2
    a = host(act).reshape(P, cfg.inter)
    assert (a[3 * 2 + 1] == 123.0).all() and (a[6 * 2 + 0] == 123.0).all()
    ref = oracle.moe_gate_up(gate, up, cfg.gu_stride, 8, 64, 64, x, 10, 2, ids)
    check_gate_up(a.reshape(-1), ref, ids, 8)
    # down on an injected act: the invalid pairs contribute nothing
    act_in = synth.normal_f32(99, P * cfg.inter)
    act.copy_(to_dev(act_in))
    y = empty(cfg.n_tokens * cfg.hidden)
    mx.mxfp4_moe_down(to_dev(down), 8, 64, 64, act, 10, 2, to_dev(ids), to_dev(wts), y, ws)
    refd = oracle.moe_down(down, cfg.down_stride, 8, 64, 64, act_in, 10, 2, ids, wts)
    assert_within(host(y), refd["out"], refd["l1_out"], REL_FP32, "down with invalid ids")


@pytest.mark.parametrize("E", [300, 2000, 5000])
def test_layer_with_many_experts(mx, E):
    # the routing plan's scans over several warps (300), several experts per
    # thread (2000) and the plan beyond 4096 experts (5000); past 1024 experts
    # the expert passes are the FP32 ones
    hidden, inter, T, K = 64, 32, 64, 4
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 23)
    y, ws = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    assert mx.mxfp4_moe_plan_errors(ws) == 0
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                             x, T, K, ids, wts)
    assert_within(y, ref["out"], ref["bound_l1"] + ref["bound_prop"], REL_FP32, f"{E} experts")


def test_passes_repeated_on_one_workspace(mx):
    # the passes' CTAs claim segments from a counter in the workspace, which the
    # plan zeroes and the last CTA of every pass zeroes again: the down pass run
    # three times on one plan, then a new plan on the same workspace, give the
    # same bits each time (about 1000 gate/up and 250 down segments, several
    # claims per CTA)
    cfg, gate, up, down, x, ids, wts = make_case(64, 1024, 2048, 64, 4, 17)
    act, ws = run_gate_up(mx, cfg, gate, up, x, ids)
    act0 = host(act).copy()
    outs = []
    for _ in range(3):
        y = empty(cfg.n_tokens * cfg.hidden)
        mx.mxfp4_moe_down(to_dev(down), cfg.n_experts, cfg.hidden, cfg.inter, act,
                          cfg.n_tokens, cfg.top_k, to_dev(ids), to_dev(wts), y, ws)
        outs.append(host(y))
    run_gate_up(mx, cfg, gate, up, x, ids, ws=ws, act=act)
    assert_bits_equal(host(act), act0, "gate/up again on the same workspace")
    y = empty(cfg.n_tokens * cfg.hidden)
    mx.mxfp4_moe_down(to_dev(down), cfg.n_experts, cfg.hidden, cfg.inter, act, cfg.n_tokens,
                      cfg.top_k, to_dev(ids), to_dev(wts), y, ws)
    outs.append(host(y))
    for o in outs[1:]:
        assert_bits_equal(o, outs[0], "down again on the same workspace")
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, cfg.n_experts,
                             cfg.hidden, cfg.inter, x, cfg.n_tokens, cfg.top_k, ids, wts)
    assert_within(outs[0].reshape(cfg.n_tokens, cfg.hidden), ref["out"],
                  ref["bound_l1"] + ref["bound_prop"], REL_FP32, "MoE layer")


def plant_scale(bank, stride, rows, cols, e, r, g, byte):
    """Set the E8M0 scale byte of (row r, group g) of expert e's matrix."""
    bank[e * stride + rows * cols // 2 + r * (cols // 32) + g] = byte


def test_layer_with_odd_scale_bytes_and_large_activations(mx):
    # scale bytes outside 1..200 in a few rows (0: the subnormal scale 2^-127 in
    # gate, up and down; 201 and 210: scales of 2^74 and 2^83 and 255: NaN, in
    # down only, so that no act row spans more than the split's range) and a
    # token whose largest |x| is over 2^15 (a negative power of two) send some
    # warps' units, not whole segments, through the table path and 2^-p per
    # group, next to warps of the same segment that stay in the 2^p domain.  NaN
    # where the oracle has NaN.
    E, hidden, inter, T, K = 12, 512, 640, 24, 4
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 29)
    gate, up, down, x = gate.copy(), up.copy(), down.copy(), x.copy()
    e0, e1 = int(ids[0, 0]), int(ids[1, 1])
    plant_scale(gate, cfg.gu_stride, inter, hidden, e0, 5, 3, 0)
    plant_scale(up, cfg.gu_stride, inter, hidden, e1, 100, 0, 0)
    plant_scale(down, cfg.down_stride, hidden, inter, e0, 300, 7, 201)
    plant_scale(down, cfg.down_stride, hidden, inter, e0, 301, 2, 210)
    plant_scale(down, cfg.down_stride, hidden, inter, e1, 33, 12, 255)
    plant_scale(down, cfg.down_stride, hidden, inter, e1, 400, 19, 0)
    t_big = next(t for t in range(T) if e0 not in ids[t] and e1 not in ids[t])
    x[t_big] *= np.float32(2.0 ** 14)
    y, _ = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                             x, T, K, ids, wts)
    assert np.isnan(ref["out"]).any() and (np.abs(ref["out"]) > 2.0 ** 60).any()
    assert_within(y, ref["out"], ref["bound_l1"] + ref["bound_prop"], REL_FP32,
                  "MoE layer with odd scale bytes")


def test_down_stage_error_floor_of_a_wide_range_act(mx):
    # The split of a vector into f16 hi and lo after scaling by 2^p (largest |x|
    # into [2^14, 2^15)) represents each element to within 2^-22 of itself or an
    # absolute 2^-25 * 2^-p (the f16 subnormal spacing), whichever is larger:
    # elements below about 2^-38 of the largest are lost.  Rows whose weight is
    # zero or small where the act row peaks can then be off by more than 1e-5 of
    # their L1 sum, by at most 2^-39 * max|act| * sum_c |w[r][c]|.  An act row
    # with one element of 2^60 among N(0, 1) elements checks that floor.
    E, hidden, inter, T, K = 6, 256, 512, 10, 2
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 31)
    P = T * K
    act = synth.normal_f32(1031, P * inter).reshape(P, inter)
    act[3, 17] = np.float32(2.0 ** 60)
    act[8, 500] = np.float32(-(2.0 ** 50))
    act_d, ws = run_gate_up(mx, cfg, gate, up, x, ids)
    act_d.copy_(to_dev(act.reshape(-1)))
    y = empty(T * hidden)
    mx.mxfp4_moe_down(to_dev(down), E, hidden, inter, act_d, T, K, to_dev(ids), to_dev(wts),
                      y, ws)
    ref = oracle.moe_down(down, cfg.down_stride, E, hidden, inter, act.reshape(-1), T, K, ids,
                          wts)
    # sum_j |w_tj| * 2^-39 * max|act[pair]| * sum_c |down_e[r][c]|
    floor = np.zeros((T, hidden))
    for t in range(T):
        for j in range(K):
            e, p = int(ids[t, j]), t * K + j
            w = oracle.dequant(down[e * cfg.down_stride:(e + 1) * cfg.down_stride], hidden, inter)
            floor[t] += abs(float(wts[t, j])) * 2.0 ** -39 * np.abs(act[p]).max() * \
                np.abs(w).sum(axis=1)
    got = host(y).reshape(T, hidden)
    err = np.abs(got.astype(np.float64) - ref["out"].reshape(T, hidden))
    tol = REL_FP32 * ref["l1_out"].reshape(T, hidden) + floor
    assert (err <= tol).all(), f"worst err/tol {np.max(err / tol):.3g}"
    # the floor is what lets it pass: somewhere the plain 1e-5 * L1 is exceeded
    assert (err > REL_FP32 * ref["l1_out"].reshape(T, hidden)).any()


def test_layer_with_more_vectors_than_split_blocks(mx):
    # 700 tokens (x split) and 1400 pairs (act split): more vectors than the
    # split kernel's 4 blocks per SM, so its blocks take several vectors each
    # (the block maximum's slot rotates per vector)
    E, hidden, inter, T, K = 16, 256, 128, 700, 2
    cfg, gate, up, down, x, ids, wts = make_case(E, hidden, inter, T, K, 37)
    y, ws = run_layer(mx, cfg, gate, up, down, x, ids, wts)
    assert mx.mxfp4_moe_plan_errors(ws) == 0
    ref = oracle.moe_forward(gate, up, down, cfg.gu_stride, cfg.down_stride, E, hidden, inter,
                             x, T, K, ids, wts)
    assert_within(y, ref["out"], ref["bound_l1"] + ref["bound_prop"], REL_FP32,
                  "MoE layer, 700 tokens")
