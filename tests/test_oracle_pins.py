"""Pins for the CPU oracle: each of its functions checked against something
other than itself -- the page's closed forms (fixtures under tests/golden/),
an independent encoder of the layout, numpy/scipy/torch library routines and
brute force on tiny shapes.  CPU only."""
import math

import numpy as np
import pytest

import synth
from golden_io import bits_to_f32, f32_to_bits, parse_value, rows
from mx_encode import dense, encode, random_case


def same_f32(a, b) -> bool:
    """Bit-identical float32, except that any NaN equals any NaN."""
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return f32_to_bits(a) == f32_to_bits(b)


def assert_same_f32_arrays(got, want):
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    assert got.shape == want.shape
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), "NaN positions differ"
    assert np.array_equal(got[~gn].view(np.uint32), want[~wn].view(np.uint32))


# --- scalar decode -----------------------------------------------------------

def test_e2m1_all_16_codes_match_page_construction(orc):
    seen = 0
    for code, bits, _ in rows("e2m1_codes.txt"):
        got = orc.e2m1(int(code))
        assert f32_to_bits(got) == int(bits, 16), (code, hex(f32_to_bits(got)))
        seen += 1
    assert seen == 16


def test_e2m1_code8_is_negative_zero(orc):
    v = orc.e2m1(8)
    assert v == 0.0 and math.copysign(1.0, v) == -1.0


def test_e8m0_edge_bytes_match_page(orc):
    for k, bits in rows("e8m0_bytes.txt"):
        got = orc.e8m0(int(k))
        if bits == "nan":
            assert math.isnan(got)
        else:
            assert f32_to_bits(got) == int(bits, 16), (k, hex(f32_to_bits(got)))


def test_e8m0_every_byte_is_a_power_of_two(orc):
    for k in range(255):
        want = np.ldexp(np.float32(1.0), k - 127)  # 2^-127 is a float32 subnormal
        assert same_f32(orc.e8m0(k), want), k
    assert math.isnan(orc.e8m0(255))


def test_decode_exhaustive_code_by_scale(orc):
    # 256 rows (one per scale byte) x 32 columns (each code twice).
    codes = np.tile(np.concatenate([np.arange(16), np.arange(16)]), (256, 1))
    scales = np.arange(256).reshape(256, 1)
    buf = encode(codes, scales)
    got = orc.dequant(buf, 256, 32)
    assert_same_f32_arrays(got, dense(codes, scales))
    # the subnormal scale keeps its products exact (no flush to zero)
    assert got[0, 1] == np.float32(2.0 ** -128) and got[0, 7] == np.float32(6 * 2.0 ** -127)


# --- layout ------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 32), (3, 64), (7, 96), (16, 256), (5, 512)])
def test_layout_against_independent_encoder(orc, shape):
    rng = np.random.default_rng(sum(shape))
    codes, scales = random_case(rng, *shape, lo=0, hi=255)
    buf = encode(codes, scales)
    assert_same_f32_arrays(orc.dequant(buf, *shape), dense(codes, scales))
    r, c = shape[0] - 1, shape[1] - 3
    assert orc.code_at(buf, *shape, r, c) == codes[r, c]
    assert orc.scale_at(buf, *shape, r, c // 32) == scales[r, c // 32]


def test_hand_worked_group(orc):
    lines = list(rows("hand_group.txt"))
    words = [int(w, 16) for w in lines[0][1:]]
    x = np.arange(1, 33, dtype=np.float32)
    for k, y_s, l1_s in lines[1:]:
        buf = np.zeros(32, dtype=np.uint8)
        buf[:16] = np.array(words, dtype="<u4").view(np.uint8)
        buf[16] = int(k)
        y, l1 = orc.matmat(buf, 1, 32, x, 1)
        want_y, want_l1 = parse_value(y_s), parse_value(l1_s)
        if math.isnan(want_y):
            assert math.isnan(y[0, 0]) and math.isnan(l1[0, 0])
        else:
            assert y[0, 0] == want_y and l1[0, 0] == want_l1, (k, y, l1)


def test_hand_worked_two_rows(orc):
    lines = list(rows("hand_two_rows.txt"))
    code_bytes = [int(b, 16) for b in lines[0][1:]]
    scale_bytes = [int(b) for b in lines[1][1:]]
    buf = np.zeros(80, dtype=np.uint8)
    for i, b in enumerate(code_bytes):
        buf[16 * i:16 * (i + 1)] = b
    buf[64:68] = scale_bytes
    x = np.concatenate([np.ones(32), 2 * np.ones(32)]).astype(np.float32)
    y, l1 = orc.matmat(buf, 2, 64, x, 1)
    for r, y_s, l1_s in lines[2:]:
        r = int(r)
        wy = parse_value(y_s)
        if math.isnan(wy):
            assert math.isnan(y[0, r])
        else:
            assert y[0, r] == wy and l1[0, r] == parse_value(l1_s)


def test_nbytes_matches_page_examples(orc):
    for r, c, n in rows("nbytes.txt"):
        assert orc.nbytes_exact(int(r), int(c)) == int(n)
    assert orc.nbytes_exact(4, 48) == 0 and orc.nbytes_exact(0, 32) == 0


# --- products ----------------------------------------------------------------

@pytest.mark.parametrize("shape,nb", [((1, 32), 1), ((9, 64), 2), ((33, 96), 3),
                                      ((64, 128), 5), ((17, 32), 8)])
def test_matmat_brute_force(orc, shape, nb):
    rng = np.random.default_rng(7 * shape[0] + nb)
    codes, scales = random_case(rng, *shape)
    W = dense(codes, scales).astype(np.float64)
    x = rng.standard_normal((nb, shape[1])).astype(np.float32)
    y, l1 = orc.matmat(encode(codes, scales), *shape, x, nb)
    want = x.astype(np.float64) @ W.T
    want_l1 = np.abs(x.astype(np.float64)) @ np.abs(W).T
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12 * want_l1.max())
    np.testing.assert_allclose(l1, want_l1, rtol=1e-13)


def test_matmat_exact_small_integers(orc):
    # integer activations and scales near 1: every product and partial sum is
    # exact in double, so any correct summation order gives the same bits.
    rng = np.random.default_rng(3)
    codes, scales = random_case(rng, 40, 256, lo=126, hi=128)
    x = rng.integers(-4, 5, size=(3, 256)).astype(np.float32)
    y, _ = orc.matmat(encode(codes, scales), 40, 256, x, 3)
    want = x.astype(np.float64) @ dense(codes, scales).astype(np.float64).T
    assert np.array_equal(y, want)


def test_matmat_row_window_and_samples_agree(orc):
    rng = np.random.default_rng(5)
    codes, scales = random_case(rng, 20, 64)
    buf = encode(codes, scales)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    y, l1 = orc.matmat(buf, 20, 64, x, 4)
    yw, _ = orc.matmat(buf, 20, 64, x, 4, 5, 11)
    assert np.array_equal(yw, y[:, 5:11])
    tok = np.array([0, 3, 2, 1]); row = np.array([19, 0, 7, 7])
    ys, l1s = orc.matmat_samples(buf, 20, 64, x, tok, row)
    assert np.array_equal(ys, y[tok, row]) and np.array_equal(l1s, l1[tok, row])


def test_matmat_nan_scale_poisons_only_its_row(orc):
    rng = np.random.default_rng(11)
    codes, scales = random_case(rng, 6, 64)
    scales[2, 1] = 255
    y, _ = orc.matmat(encode(codes, scales), 6, 64, np.ones((1, 64), np.float32), 1)
    assert np.isnan(y[0, 2]) and not np.isnan(np.delete(y[0], 2)).any()


def test_matmat_zero_activation_gives_zero(orc):
    rng = np.random.default_rng(12)
    codes, scales = random_case(rng, 8, 64)
    y, l1 = orc.matmat(encode(codes, scales), 8, 64, np.zeros((2, 64), np.float32), 2)
    assert not y.any() and not l1.any()


def test_bf16_rounding_fixture(orc):
    for a, b in rows("bf16_rne.txt"):
        got = orc.bf16_rne(bits_to_f32(int(a, 16)))
        assert f32_to_bits(got) == int(b, 16), (a, hex(f32_to_bits(got)))
    assert math.isnan(orc.bf16_rne(float("nan")))


def test_bf16_rounding_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    with np.errstate(over="ignore", invalid="ignore"):
        v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                            rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
                            .view(np.float32)]).astype(np.float32)
    v = v[np.isfinite(v)]
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert_same_f32_arrays(orc.round_bf16(v), want)


def test_silu_and_its_derivative(orc):
    scipy_special = pytest.importorskip("scipy.special")
    for g in [-50.0, -3.5, -1e-3, 0.0, 0.7, 4.0, 30.0]:
        assert orc.silu(g) == pytest.approx(g * scipy_special.expit(g), rel=1e-14, abs=1e-300)
        h = 1e-6
        num = (g + h) * scipy_special.expit(g + h) - (g - h) * scipy_special.expit(g - h)
        assert orc.silu_grad(g) == pytest.approx(num / (2 * h), rel=1e-6, abs=1e-9)
    assert orc.silu_grad(0.0) == 0.5


# --- routed experts ----------------------------------------------------------

def _tiny_moe(seed=0, E=5, hidden=64, inter=32, T=3, K=2):
    rng = np.random.default_rng(seed)
    banks, mats = {}, {}
    for role, (r, c) in {"gate": (inter, hidden), "up": (inter, hidden),
                         "down": (hidden, inter)}.items():
        bufs, ms = [], []
        for _ in range(E):
            codes, scales = random_case(rng, r, c)
            bufs.append(encode(codes, scales)); ms.append(dense(codes, scales).astype(np.float64))
        banks[role], mats[role] = np.concatenate(bufs), ms
    x = rng.standard_normal((T, hidden)).astype(np.float32)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, K)).astype(np.float32)
    stride_gu = synth.padded_nbytes(inter, hidden)
    stride_dn = synth.padded_nbytes(hidden, inter)
    return dict(E=E, hidden=hidden, inter=inter, T=T, K=K, banks=banks, mats=mats, x=x,
                ids=ids, wts=wts, stride_gu=stride_gu, stride_dn=stride_dn)


def test_moe_gate_up_against_dense_numpy(orc):
    m = _tiny_moe()
    res = orc.moe_gate_up(m["banks"]["gate"], m["banks"]["up"], m["stride_gu"], m["E"],
                          m["hidden"], m["inter"], m["x"], m["T"], m["K"], m["ids"])
    for t in range(m["T"]):
        for j in range(m["K"]):
            p, e = t * m["K"] + j, m["ids"][t, j]
            xt = m["x"][t].astype(np.float64)
            g = m["mats"]["gate"][e] @ xt
            u = m["mats"]["up"][e] @ xt
            np.testing.assert_allclose(res["g"][p], g, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(res["u"][p], u, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(res["l1g"][p], np.abs(m["mats"]["gate"][e]) @ np.abs(xt),
                                       rtol=1e-12)
            np.testing.assert_allclose(res["l1u"][p], np.abs(m["mats"]["up"][e]) @ np.abs(xt),
                                       rtol=1e-12)
            with np.errstate(over="ignore"):
                act = g / (1.0 + np.exp(-g)) * u
            np.testing.assert_allclose(res["act"][p], act, rtol=1e-11, atol=1e-12)


def test_moe_down_against_dense_numpy(orc):
    m = _tiny_moe(seed=1)
    rng = np.random.default_rng(9)
    act = rng.standard_normal((m["T"] * m["K"], m["inter"])).astype(np.float32)
    res = orc.moe_down(m["banks"]["down"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                       act, m["T"], m["K"], m["ids"], m["wts"], want_pairs=True)
    for t in range(m["T"]):
        want = np.zeros(m["hidden"])
        for j in range(m["K"]):
            p, e = t * m["K"] + j, m["ids"][t, j]
            o = m["mats"]["down"][e] @ act[p].astype(np.float64)
            np.testing.assert_allclose(res["o_pairs"][p], o, rtol=1e-12, atol=1e-12)
            want += np.float64(m["wts"][t, j]) * o
        np.testing.assert_allclose(res["out"][t], want, rtol=1e-12, atol=1e-12)


def test_moe_down_l1_terms_against_dense_numpy(orc):
    # l1_pairs[p] = |down_e| |act_p| and l1_out[t] = sum_j |w_tj| l1_pairs[t*K + j]: the
    # magnitudes the down stage's tolerance is relative to
    m = _tiny_moe(seed=4)
    rng = np.random.default_rng(10)
    act = rng.standard_normal((m["T"] * m["K"], m["inter"])).astype(np.float32)
    wts = m["wts"].copy()
    wts[0, 1] = -wts[0, 1]          # a negative route weight still adds |w|
    res = orc.moe_down(m["banks"]["down"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                       act, m["T"], m["K"], m["ids"], wts, want_pairs=True)
    for t in range(m["T"]):
        want = np.zeros(m["hidden"])
        for j in range(m["K"]):
            p, e = t * m["K"] + j, m["ids"][t, j]
            l1p = np.abs(m["mats"]["down"][e]) @ np.abs(act[p].astype(np.float64))
            np.testing.assert_allclose(res["l1_pairs"][p], l1p, rtol=1e-12)
            want += abs(np.float64(wts[t, j])) * l1p
        np.testing.assert_allclose(res["l1_out"][t], want, rtol=1e-12)


def test_moe_forward_is_gate_up_then_down_in_double(orc):
    m = _tiny_moe(seed=2)
    fw = orc.moe_forward(m["banks"]["gate"], m["banks"]["up"], m["banks"]["down"],
                         m["stride_gu"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                         m["x"], m["T"], m["K"], m["ids"], m["wts"])
    for t in range(m["T"]):
        want = np.zeros(m["hidden"])
        for j in range(m["K"]):
            e = m["ids"][t, j]
            xt = m["x"][t].astype(np.float64)
            g = m["mats"]["gate"][e] @ xt
            u = m["mats"]["up"][e] @ xt
            with np.errstate(over="ignore"):
                a = g / (1.0 + np.exp(-g)) * u
            want += np.float64(m["wts"][t, j]) * (m["mats"]["down"][e] @ a)
        np.testing.assert_allclose(fw["out"][t], want, rtol=1e-11, atol=1e-11)
    assert (fw["bound_l1"] >= np.abs(fw["out"]) * (1 - 1e-12)).all()
    assert (fw["bound_prop"] > 0).all()


def _dense_layer(m, x, wts, dg=None, du=None):
    """The layer in double from the dense matrices, with optional additive errors
    dg[p], du[p] on the gate and up dot products of pair p."""
    out = np.zeros((m["T"], m["hidden"]))
    acts = {}
    for t in range(m["T"]):
        xt = x[t].astype(np.float64)
        for j in range(m["K"]):
            p, e = t * m["K"] + j, m["ids"][t, j]
            g = m["mats"]["gate"][e] @ xt + (0.0 if dg is None else dg[p])
            u = m["mats"]["up"][e] @ xt + (0.0 if du is None else du[p])
            with np.errstate(over="ignore"):
                a = g / (1.0 + np.exp(-g)) * u
            acts[p] = (g, u, a)
            out[t] += np.float64(wts[t, j]) * (m["mats"]["down"][e] @ a)
    return out, acts


def test_moe_forward_bound_l1_against_dense_numpy(orc):
    m = _tiny_moe(seed=5)
    fw = orc.moe_forward(m["banks"]["gate"], m["banks"]["up"], m["banks"]["down"],
                         m["stride_gu"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                         m["x"], m["T"], m["K"], m["ids"], m["wts"])
    _, acts = _dense_layer(m, m["x"], m["wts"])
    for t in range(m["T"]):
        want = np.zeros(m["hidden"])
        for j in range(m["K"]):
            p, e = t * m["K"] + j, m["ids"][t, j]
            want += abs(np.float64(m["wts"][t, j])) * (np.abs(m["mats"]["down"][e]) @
                                                      np.abs(acts[p][2]))
        np.testing.assert_allclose(fw["bound_l1"][t], want, rtol=1e-12)


def test_moe_forward_bound_prop_is_the_worst_first_order_error(orc):
    # bound_prop's defining property: if every gate dot product g_c may be off by
    # eps * L1g_c and every up dot product u_c by eps * L1u_c, the largest first-order
    # change of out[t][r] is eps * bound_prop[t][r].  Attain it: for one output
    # (t, r), push g_c and u_c of each of t's pairs in the direction that moves
    # w_tj * down_e[r][c] * act_c upward (signs of w down silu'(g) u and w down
    # silu(g)), run the perturbed layer densely in numpy, and compare the change
    # over eps with the oracle's bound.  A bound that dropped |u|, the route
    # weight, |down| or either term would miss.
    m = _tiny_moe(seed=6, E=6, hidden=96, inter=64, T=3, K=3)
    wts = m["wts"].copy()
    wts[1, 2] = -0.6                  # signs of the route weights matter too
    fw = orc.moe_forward(m["banks"]["gate"], m["banks"]["up"], m["banks"]["down"],
                         m["stride_gu"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                         m["x"], m["T"], m["K"], m["ids"], wts)
    base, acts = _dense_layer(m, m["x"], wts)
    eps = 1e-7
    checked = 0
    for t in range(m["T"]):
        xt = np.abs(m["x"][t].astype(np.float64))
        for r in (0, 7, m["hidden"] - 1):
            dg, du = {}, {}
            for j in range(m["K"]):
                p, e = t * m["K"] + j, m["ids"][t, j]
                g, u, _ = acts[p]
                s = 1.0 / (1.0 + np.exp(-g))
                dsilu = s * (1.0 + g * (1.0 - s))
                coef = np.float64(wts[t, j]) * m["mats"]["down"][e][r]
                l1g = np.abs(m["mats"]["gate"][e]) @ xt
                l1u = np.abs(m["mats"]["up"][e]) @ xt
                dg[p] = eps * l1g * np.sign(coef * dsilu * u)
                du[p] = eps * l1u * np.sign(coef * g * s)
            for tt in range(m["T"]):
                for j in range(m["K"]):
                    dg.setdefault(tt * m["K"] + j, 0.0)
                    du.setdefault(tt * m["K"] + j, 0.0)
            moved, _ = _dense_layer(m, m["x"], wts, dg, du)
            rate = (moved[t, r] - base[t, r]) / eps
            assert rate == pytest.approx(fw["bound_prop"][t, r], rel=1e-4), (t, r)
            checked += 1
    assert checked == 3 * m["T"]


def test_moe_plan_is_a_stable_counting_sort(orc):
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 16, size=200).astype(np.int32)
    ids[[5, 77]] = [-1, 16]  # two invalid ids
    offsets, pair_of, bad = orc.moe_plan(ids, 16)
    assert bad == 2
    valid = np.flatnonzero((ids >= 0) & (ids < 16))
    order = valid[np.argsort(ids[valid], kind="stable")]
    assert np.array_equal(pair_of[:order.size], order)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(ids[valid],
                                                                            minlength=16))]))


# --- the seeded generator ----------------------------------------------------

def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 from state 0 (Vigna's reference splitmix64.c).
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert [int(v) for v in synth.splitmix64(0, 4)] == want
    assert [int(v) for v in synth.splitmix64(0, 2, start=2)] == want[2:]


def test_generator_is_deterministic_and_shaped():
    a = synth.TINY.weights()
    b = synth.TINY.weights()
    assert np.array_equal(a, b) and a.size == synth.padded_nbytes(256, 512) == 69632
    s = a[256 * 512 // 2: 256 * 512 // 2 + 256 * 16]
    assert s[3 * 16 + 5] == 0 and s[250 * 16 + 11] == 255
    body = np.delete(s, [3 * 16 + 5, 250 * 16 + 11])
    assert body.min() >= 118 and body.max() <= 136
    x = synth.TINY.activations()
    assert x.shape == (1, 512) and x.dtype == np.float32 and abs(x.mean()) < 0.2


def test_route_generator_distinct_ids_and_softmax():
    ids, w = synth.routes(3, 32, 4, 64)
    assert ids.shape == (32, 4) and (ids >= 0).all() and (ids < 64).all()
    assert all(len(set(r)) == 4 for r in ids.tolist())
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
    assert (w > 0).all()


def test_expert_banks_have_distinct_scale_planes():
    E, r, c = 5, 32, 64
    bank = synth.expert_bank(E, r, c, 3, 118, 130, "gate")
    stride = synth.padded_nbytes(r, c)
    planes = [bank[e * stride + r * c // 2: e * stride + r * c // 2 + r * c // 32].tobytes()
              for e in range(E)]
    assert len(set(planes)) == E


def test_adjacent_distinct_scale_pattern():
    buf = synth.mxfp4_matrix(8, 128, 4, 119, 123, scale_pattern="adjacent_distinct")
    s = buf[8 * 64: 8 * 64 + 32].astype(int)
    assert (np.diff(s) != 0).all() and s.min() >= 119 and s.max() <= 123


def test_moe_invalid_pair_contributes_nothing(orc):
    m = _tiny_moe(seed=3)
    ids = m["ids"].copy()
    ids[1, 0] = m["E"]          # out of range
    rng = np.random.default_rng(2)
    act = rng.standard_normal((m["T"] * m["K"], m["inter"])).astype(np.float32)
    res = orc.moe_down(m["banks"]["down"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                       act, m["T"], m["K"], ids, m["wts"], want_pairs=True)
    p_bad = 1 * m["K"] + 0
    assert np.isnan(res["o_pairs"][p_bad]).all()
    e1 = ids[1, 1]
    want = np.float64(m["wts"][1, 1]) * (m["mats"]["down"][e1] @ act[p_bad + 1].astype(np.float64))
    np.testing.assert_allclose(res["out"][1], want, rtol=1e-12, atol=1e-12)
    offsets, pair_of, bad = orc.moe_plan(ids.reshape(-1), m["E"])
    assert bad == 1 and p_bad not in pair_of[:offsets[-1]]


# --- the global-bank form: bf16 boundaries, SwiGLU limit, pre-weighting, slots ----

def _bf16(a):
    """Round-to-nearest-even bfloat16 of the float32 value (torch's conversion)."""
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)


def _dense_layer_ex(m, x, ids, wts, bf16_mode, limit, slot_of=None, dtype=np.float64):
    """The global-bank layer from the dense matrices, in numpy (float64 or
    float32 arithmetic), bf16 rounding by torch; slot_of maps ids to bank slots."""
    out = np.zeros((m["T"], m["hidden"]), dtype=np.float64)
    for t in range(m["T"]):
        xt = x[t].astype(dtype)
        acc = np.zeros(m["hidden"], dtype=dtype)
        for j in range(m["K"]):
            e = int(ids[t, j])
            if e < 0 or e >= m["E"]:
                continue
            s = e if slot_of is None else int(slot_of[e])
            if s < 0:
                continue
            G, U, D = (m["mats"][k][s].astype(dtype) for k in ("gate", "up", "down"))
            g, u = G @ xt, U @ xt
            if bf16_mode:
                g, u = _bf16(g).astype(dtype), _bf16(u).astype(dtype)
            if limit > 0:
                u = np.clip(u, -limit, limit)
                g = np.minimum(g, dtype(limit))
            with np.errstate(over="ignore"):
                a = g / (dtype(1.0) + np.exp(-g)) * u
            w = dtype(wts[t, j])
            if bf16_mode:
                a = _bf16(w * a).astype(dtype)
                acc = acc + D @ a
            else:
                acc = acc + w * (D @ a)
        out[t] = _bf16(acc) if bf16_mode else acc
    return out


def _fwd_ex(orc, m, ids, wts, **kw):
    return orc.moe_forward_ex(m["banks"]["gate"], m["banks"]["up"], m["banks"]["down"],
                              m["stride_gu"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                              m["x"], m["T"], m["K"], ids, wts, **kw)


def test_moe_forward_ex_generic_mode_is_the_f32_layer(orc):
    m = _tiny_moe(seed=7)
    ex = _fwd_ex(orc, m, m["ids"], m["wts"])
    fw = orc.moe_forward(m["banks"]["gate"], m["banks"]["up"], m["banks"]["down"],
                         m["stride_gu"], m["stride_dn"], m["E"], m["hidden"], m["inter"],
                         m["x"], m["T"], m["K"], m["ids"], m["wts"])
    assert np.array_equal(ex["out"], fw["out"]) and ex["cold"].size == 0


@pytest.mark.parametrize("limit", [0.0, 0.75])
def test_moe_forward_ex_bf16_mode_against_dense_numpy(orc, limit):
    m = _tiny_moe(seed=8, E=6, hidden=96, inter=64, T=4, K=3)
    ex = _fwd_ex(orc, m, m["ids"], m["wts"], bf16_mode=True, limit=limit)
    want = _dense_layer_ex(m, m["x"], m["ids"], m["wts"], True, limit)
    # the two sum in different orders before the bf16 roundings: equal but for
    # rare values on a rounding boundary, which land one bf16 step apart
    same = ex["out"] == want
    assert same.mean() > 0.97, same.mean()
    step = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(want), 1e-30))).astype(int) - 7)
    assert (np.abs(ex["out"] - want) <= 2 * step).all()
    # every output is a bfloat16 value
    assert np.array_equal(_bf16(ex["out"]), ex["out"])
    if limit > 0:   # the limit changes the result (it is active on this input)
        free = _dense_layer_ex(m, m["x"], m["ids"], m["wts"], True, 0.0)
        assert not np.array_equal(free, want)


def test_moe_forward_ex_slot_table_and_cold_experts(orc):
    m = _tiny_moe(seed=9, E=6, hidden=64, inter=64, T=5, K=2)
    # the same experts in a permuted bank, addressed through slot_of
    perm = np.array([3, 0, 5, 1, 4, 2], dtype=np.int32)        # expert e lives in slot perm[e]
    inv = np.argsort(perm)
    banks = {}
    for role, stride in (("gate", m["stride_gu"]), ("up", m["stride_gu"]),
                         ("down", m["stride_dn"])):
        b = m["banks"][role].reshape(m["E"], stride)
        banks[role] = np.ascontiguousarray(b[inv]).reshape(-1)
    ids = m["ids"].copy()
    ids[1, 0] = 4
    ids[3, 1] = 4
    base = _fwd_ex(orc, m, ids, m["wts"], bf16_mode=True, limit=0.5)
    mp = dict(m, banks=banks)
    moved = _fwd_ex(orc, mp, ids, m["wts"], slot_of=perm, bf16_mode=True, limit=0.5)
    assert np.array_equal(moved["out"], base["out"])
    # expert 4 cold: its pairs are listed (increasing pair order) and left out
    cold_tab = perm.copy()
    cold_tab[4] = -1
    cold = _fwd_ex(orc, mp, ids, m["wts"], slot_of=cold_tab, bf16_mode=True, limit=0.5)
    want_pairs = np.flatnonzero(ids.reshape(-1) == 4)
    assert np.array_equal(cold["cold"], want_pairs)
    ids_wo = ids.copy()
    ids_wo[ids_wo == 4] = -1
    assert np.array_equal(cold["out"], _fwd_ex(orc, m, ids_wo, m["wts"], bf16_mode=True,
                                               limit=0.5)["out"])
    # a slot outside the bank is invalid: not listed as cold, contributes nothing
    bad_tab = perm.copy()
    bad_tab[4] = m["E"]
    bad = _fwd_ex(orc, mp, ids, m["wts"], slot_of=bad_tab, bf16_mode=True, limit=0.5)
    assert bad["cold"].size == 0 and np.array_equal(bad["out"], cold["out"])


@pytest.mark.parametrize("bf16_mode,limit", [(False, 0.0), (True, 0.0), (True, 0.75),
                                             (False, 0.75)])
def test_moe_forward_ex_bound_holds_for_a_float32_layer(orc, bf16_mode, limit):
    # an implementation whose dot products are float32 (numpy, another order
    # than the oracle's) stays inside the bound, and the bound is tight enough
    # to mean something
    m = _tiny_moe(seed=10, E=6, hidden=96, inter=64, T=4, K=3)
    ex = _fwd_ex(orc, m, m["ids"], m["wts"], bf16_mode=bf16_mode, limit=limit)
    f32 = _dense_layer_ex(m, m["x"], m["ids"], m["wts"], bf16_mode, limit, dtype=np.float32)
    assert (np.abs(f32 - ex["out"]) <= ex["bound"]).all()
    # of the order of the errors it stands for: eps = 1e-5 of the L1 norms in the
    # generic mode (the cancellation of the sums makes L1 / |out| ~ 10-50 here);
    # in the bf16 mode a step of 2^-8..2^-7 at each of the act's elements
    rel = np.median(ex["bound"] / np.maximum(np.abs(ex["out"]), 1e-30))
    assert rel < (2.0 ** -3 if bf16_mode else 1e-3), rel
    # and tight enough to catch a mistake: the route weights dropped, or (with a
    # limit) the clamp of up left out
    wrong = _dense_layer_ex(m, m["x"], m["ids"], np.ones_like(m["wts"]), bf16_mode, limit)
    assert (np.abs(wrong - ex["out"]) > ex["bound"]).any()
    if limit > 0:
        m_wide = _dense_layer_ex(m, m["x"], m["ids"], m["wts"], bf16_mode, 1e30)
        assert (np.abs(m_wide - ex["out"]) > ex["bound"]).any()
