"""Pins for the float MoE oracle, independent of the oracle's own code.

The [MoE README] (com.microsoft.MoE kernel README: Description, Inputs,
Attributes) fixes: a softmax over every expert before top-k, optional
renormalisation of the selected weights, FC1/FC3/FC2 with optional biases
(the FC2 bias before the routing weight), and the activations relu, gelu,
silu, swiglu (three FC1/FC3 layouts) and identity.  The tests below pin the
oracle with layers worked out by hand, closed forms checked against scipy,
layout equivalences, brute force over every expert, agreement with the
separately pinned QMoE oracle on dequantised weights, and a numpy/scipy
composition of the whole layer.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "moe_hand_cases.json")) as f:
        return json.load(f)["cases"]


def _arr(case, key):
    return None if key not in case else np.array(case[key], np.float32)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_moe_hand_cases(case):
    y, sel, w = oracle.moe(_arr(case, "x"), _arr(case, "logits"), _arr(case, "w1"),
                           _arr(case, "w2"), k=case["k"], fc1_bias=_arr(case, "b1"),
                           fc2_bias=_arr(case, "b2"), fc3_w=_arr(case, "w3"),
                           fc3_bias=_arr(case, "b3"), activation_type=case["activation"],
                           swiglu_fusion=case["swiglu_fusion"], activation_alpha=case["alpha"],
                           activation_beta=case["beta"],
                           normalize_routing_weights=case["normalize"])
    assert sel.tolist() == case["expected_sel"]
    np.testing.assert_allclose(w, case["expected_w"], rtol=1e-14)
    np.testing.assert_allclose(y, case["expected_y"], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------

def test_route_k_equals_e_is_scipy_softmax():
    lg = np.random.default_rng(1).standard_normal((9, 7)).astype(np.float32)
    sel, w = oracle.moe_route(lg, 7, 0)
    ref = special.softmax(lg.astype(np.float64), axis=1)
    for t in range(9):
        assert sorted(sel[t].tolist()) == list(range(7))
        np.testing.assert_allclose(w[t], ref[t, sel[t]], rtol=1e-14)
        assert np.all(np.diff(w[t]) <= 0)


def test_route_unnormalized_weights_are_full_softmax_entries():
    lg = np.random.default_rng(2).standard_normal((11, 16)).astype(np.float32) * 2
    sel, w = oracle.moe_route(lg, 3, 0)
    ref = special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, sel.astype(np.int64), 1), rtol=1e-14)
    assert np.all(w.sum(1) < 1.0)
    order = np.argsort(-ref, axis=1, kind="stable")[:, :3]
    assert np.array_equal(sel, order)


def test_route_normalized_equals_selected_softmax():
    # Renormalising softmax(all) over the selection is the softmax of the
    # selected logits: the QMoE oracle's routing (pinned separately) computes that.
    lg = np.random.default_rng(3).standard_normal((13, 10)).astype(np.float32)
    sel, w = oracle.moe_route(lg, 4, 1)
    qsel, qp = oracle.route(lg, 4)
    assert np.array_equal(sel, qsel)
    np.testing.assert_allclose(w, qp, rtol=1e-14)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)


def test_route_k1_normalized_is_one_unnormalized_is_max_prob():
    lg = np.array([[0.0, 1.0, -1.0]], np.float32)
    _, w1 = oracle.moe_route(lg, 1, 1)
    assert w1[0, 0] == 1.0
    sel, w0 = oracle.moe_route(lg, 1, 0)
    assert sel[0, 0] == 1
    assert w0[0, 0] == pytest.approx(math.e / (1 + math.e + math.exp(-1)), rel=1e-15)


def test_route_ties_to_lower_index():
    sel, w = oracle.moe_route(np.array([[0.5, 2.0, 2.0, 0.5]], np.float32), 3, 0)
    assert sel.tolist() == [[1, 2, 0]]
    assert w[0, 0] == w[0, 1]


# ----------------------------------------------------------------------------
# Activations
# ----------------------------------------------------------------------------

H_VALUES = np.array([-6.0, -2.5, -1.0, -0.1, 0.0, 0.3, 1.0, 2.0, 7.5])


def test_gelu_is_x_times_normal_cdf():
    a = oracle.moe_activation(H_VALUES, H_VALUES.size, "gelu")
    np.testing.assert_allclose(a, H_VALUES * stats.norm.cdf(H_VALUES), rtol=1e-14, atol=1e-300)


def test_silu_is_x_times_expit_and_fc3_multiplies():
    a = oracle.moe_activation(H_VALUES, H_VALUES.size, "silu")
    np.testing.assert_allclose(a, H_VALUES * special.expit(H_VALUES), rtol=1e-14)
    h3 = np.linspace(-2, 2, H_VALUES.size)
    a3 = oracle.moe_activation(H_VALUES, H_VALUES.size, "silu", h3=h3)
    np.testing.assert_allclose(a3, H_VALUES * special.expit(H_VALUES) * h3, rtol=1e-14)


def test_relu_and_identity():
    r = oracle.moe_activation(H_VALUES, H_VALUES.size, "relu")
    assert np.array_equal(r, np.maximum(H_VALUES, 0.0))
    i = oracle.moe_activation(H_VALUES, H_VALUES.size, "identity")
    assert np.array_equal(i, H_VALUES)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.702, 1.0)])
def test_swiglu_layouts_agree(alpha, beta):
    g = np.array([-2.0, -0.5, 0.0, 0.7, 3.0])
    u = np.array([1.5, -1.0, 2.0, 0.25, -3.0])
    ref = g * special.expit(alpha * g) * (u + beta)
    inter = np.empty(10)
    inter[0::2], inter[1::2] = g, u
    kw = dict(alpha=alpha, beta=beta)
    a0 = oracle.moe_activation(g, 5, "swiglu", h3=u, swiglu_fusion=0, **kw)
    a1 = oracle.moe_activation(inter, 5, "swiglu", swiglu_fusion=1, **kw)
    a2 = oracle.moe_activation(np.concatenate([g, u]), 5, "swiglu", swiglu_fusion=2, **kw)
    for a in (a0, a1, a2):
        np.testing.assert_allclose(a, ref, rtol=1e-14, atol=1e-300)


# ----------------------------------------------------------------------------
# Whole layers
# ----------------------------------------------------------------------------

def _rand(seed, T=6, H=24, I=12, E=5, act="relu", fusion=0, fc3=False, biases=True):
    rng = np.random.default_rng(seed)
    rows = 2 * I if (act == "swiglu" and fusion != 0) else I
    d = dict(
        x=rng.standard_normal((T, H)).astype(np.float32),
        logits=rng.standard_normal((T, E)).astype(np.float32),
        fc1_w=(rng.standard_normal((E, rows, H)) / math.sqrt(H)).astype(np.float32),
        fc2_w=(rng.standard_normal((E, H, I)) / math.sqrt(I)).astype(np.float32))
    if fc3:
        d["fc3_w"] = (rng.standard_normal((E, I, H)) / math.sqrt(H)).astype(np.float32)
    if biases:
        d["fc1_bias"] = rng.standard_normal((E, rows)).astype(np.float32) * 0.1
        d["fc2_bias"] = rng.standard_normal((E, H)).astype(np.float32) * 0.1
        if fc3:
            d["fc3_bias"] = rng.standard_normal((E, I)).astype(np.float32) * 0.1
    return d


def _run(d, **kw):
    d = dict(d)
    return oracle.moe(d.pop("x"), d.pop("logits"), d.pop("fc1_w"), d.pop("fc2_w"), **d, **kw)


def _numpy_layer(d, k, act, fusion=0, alpha=1.0, beta=0.0, normalize=0):
    """The layer composed from numpy/scipy primitives (softmax, argsort, matmul,
    erf, expit), one selection at a time."""
    x = d["x"].astype(np.float64)
    p = special.softmax(d["logits"].astype(np.float64), axis=1)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    w = np.take_along_axis(p, order, 1)
    if normalize:
        w = w / w.sum(1, keepdims=True)
    y = np.zeros_like(x)
    f64 = lambda key: None if key not in d else d[key].astype(np.float64)
    W1, W2, W3 = f64("fc1_w"), f64("fc2_w"), f64("fc3_w")
    B1, B2, B3 = f64("fc1_bias"), f64("fc2_bias"), f64("fc3_bias")
    I = W2.shape[2]
    for t in range(x.shape[0]):
        for i in range(k):
            e = order[t, i]
            h1 = W1[e] @ x[t] + (0 if B1 is None else B1[e])
            h3 = None if W3 is None else W3[e] @ x[t] + (0 if B3 is None else B3[e])
            if act == "relu":
                a = np.maximum(h1, 0)
            elif act == "gelu":
                a = 0.5 * h1 * (1 + special.erf(h1 / math.sqrt(2)))
            elif act == "identity":
                a = h1
            elif act == "silu":
                a = h1 * special.expit(h1) * (1 if h3 is None else h3)
            else:
                g, u = ((h1, h3) if fusion == 0 else
                        (h1[0::2], h1[1::2]) if fusion == 1 else (h1[:I], h1[I:]))
                a = g * special.expit(alpha * g) * (u + beta)
            y[t] += w[t, i] * (W2[e] @ a + (0 if B2 is None else B2[e]))
    return y, order, w


@pytest.mark.parametrize("act,fusion,fc3,normalize", [
    ("relu", 0, False, 0), ("gelu", 0, False, 1), ("identity", 0, False, 0),
    ("silu", 0, False, 0), ("silu", 0, True, 1), ("swiglu", 0, True, 0),
    ("swiglu", 1, False, 1), ("swiglu", 2, False, 0)])
def test_layer_equals_numpy_composition(act, fusion, fc3, normalize):
    d = _rand(20, act=act, fusion=fusion, fc3=fc3)
    kw = dict(k=3, activation_type=act, swiglu_fusion=fusion, activation_alpha=1.3,
              activation_beta=0.4, normalize_routing_weights=normalize)
    y, sel, w = _run(d, **kw)
    y_ref, order, w_ref = _numpy_layer(d, 3, act, fusion, 1.3, 0.4, normalize)
    assert np.array_equal(sel, order)
    np.testing.assert_allclose(w, w_ref, rtol=1e-13)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-13)


def test_swiglu_fusion_layouts_give_the_same_layer():
    d0 = _rand(21, act="swiglu", fusion=0, fc3=True)
    g_w, u_w = d0["fc1_w"], d0["fc3_w"]
    g_b, u_b = d0["fc1_bias"], d0["fc3_bias"]
    E, I, H = g_w.shape
    inter_w = np.empty((E, 2 * I, H), np.float32)
    inter_w[:, 0::2], inter_w[:, 1::2] = g_w, u_w
    inter_b = np.empty((E, 2 * I), np.float32)
    inter_b[:, 0::2], inter_b[:, 1::2] = g_b, u_b
    kw = dict(k=2, activation_type="swiglu", activation_alpha=1.702, activation_beta=1.0)
    y0, _, _ = _run(d0, swiglu_fusion=0, **kw)
    base = {k: v for k, v in d0.items() if not k.startswith("fc3") and not k.startswith("fc1")}
    y1, _, _ = _run(dict(base, fc1_w=inter_w, fc1_bias=inter_b), swiglu_fusion=1, **kw)
    y2, _, _ = _run(dict(base, fc1_w=np.concatenate([g_w, u_w], 1),
                         fc1_bias=np.concatenate([g_b, u_b], 1)), swiglu_fusion=2, **kw)
    assert np.array_equal(y0, y1) and np.array_equal(y0, y2)


def test_silu_with_fc3_is_swiglu_with_default_alpha_beta():
    d = _rand(22, act="swiglu", fusion=0, fc3=True)
    ys, _, _ = _run(d, k=2, activation_type="silu")
    yw, _, _ = _run(d, k=2, activation_type="swiglu", swiglu_fusion=0)
    assert np.array_equal(ys, yw)


def test_fc3_ignored_by_other_activations():
    d = _rand(23, fc3=True)
    for act in ("relu", "gelu", "identity"):
        y, _, _ = _run(d, k=2, activation_type=act)
        base = {k: v for k, v in d.items() if not k.startswith("fc3")}
        y2, _, _ = _run(base, k=2, activation_type=act)
        assert np.array_equal(y, y2)


@pytest.mark.parametrize("act,fusion,fc3", [("relu", 0, False), ("swiglu", 2, False),
                                            ("silu", 0, True)])
def test_dense_brute_force_matches(act, fusion, fc3):
    d = _rand(24, act=act, fusion=fusion, fc3=fc3, E=4)
    kw = dict(k=2, activation_type=act, swiglu_fusion=fusion)
    y, _, _ = _run(d, **kw)
    yd, _, _ = _run(d, dense=True, **kw)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_zero_weights_leave_the_bias_path():
    # FC1 weights 0: h = b1; with relu, o = W2 relu(b1) + b2 for every token.
    d = _rand(25, T=4, H=8, I=4, E=3)
    d["fc1_w"] = np.zeros_like(d["fc1_w"])
    y, sel, w = _run(d, k=2, activation_type="relu")
    o = (np.einsum("ehi,ei->eh", d["fc2_w"].astype(np.float64),
                   np.maximum(d["fc1_bias"].astype(np.float64), 0))
         + d["fc2_bias"].astype(np.float64))
    ref = np.einsum("tk,tkh->th", w, o[sel])
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_matches_qmoe_oracle_on_dequantised_weights():
    """The float layer with renormalised routing, no biases and the QMoE
    weights dequantised equals the QMoE layer (whose softmax over the selected
    logits is the renormalised full softmax)."""
    rng = np.random.default_rng(26)
    T, H, I, E, k = 5, 16, 8, 4, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    w1 = rng.integers(0, 256, (E, 2 * I, H), dtype=np.uint8)
    w2 = rng.integers(0, 256, (E, H, I), dtype=np.uint8)
    s1 = np.full((E, 2 * I), 0.25, np.float32)        # powers of two: exact in fp32
    s2 = np.full((E, H), 0.125, np.float32)
    yq, selq, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, k=k, expert_weight_bits=8,
                              activation_type="swiglu", activation_alpha=1.5,
                              activation_beta=0.5)
    f1 = ((w1.astype(np.float32) - 128) * 0.25).astype(np.float32)
    f2 = ((w2.astype(np.float32) - 128) * 0.125).astype(np.float32)
    yf, self_, _ = oracle.moe(x, lg, f1, f2, k=k, activation_type="swiglu", swiglu_fusion=1,
                              activation_alpha=1.5, activation_beta=0.5,
                              normalize_routing_weights=1)
    assert np.array_equal(selq, self_)
    np.testing.assert_allclose(yf, yq, rtol=1e-13, atol=1e-13)


def test_rank3_subset_and_threads_match_full():
    d = _rand(27, T=12)
    y, _, _ = _run(d, k=2)
    d3 = dict(d, x=d["x"].reshape(3, 4, -1))
    y3, _, _ = _run(d3, k=2)
    assert np.array_equal(y, y3)
    sub = np.array([0, 7, 11])
    ys, _, _ = _run(d, k=2, tokens=sub, nthreads=3)
    assert np.array_equal(ys, y[sub])


def test_swiglu_fusion0_without_fc3_is_rejected():
    d = _rand(28, act="swiglu", fusion=0, fc3=False)
    with pytest.raises(ValueError):
        _run(d, k=1, activation_type="swiglu", swiglu_fusion=0)
