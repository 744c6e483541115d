"""Pins for the CPU oracle, independent of the oracle's own code.

Each test fixes a value or a property that the operator pages or plain
mathematics determine: the GroupedMatMul worked examples (inputs printed on
the ONNX page, outputs worked out by hand), hand-packed nibble/byte codes,
small QMoE layers computed on paper, closed forms (k = 1, zero scales,
k = E), invariants (expert permutation, 4-bit/8-bit repack, column-wise vs
block-wise) and brute force (dense evaluation over every expert, the
Gather/Expand/MatMul decomposition, numpy einsum).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# GroupedMatMul
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("ex", _load("grouped_matmul_examples.json")["examples"],
                         ids=lambda e: e["name"])
def test_gmm_worked_examples(ex):
    if "expected" not in ex:
        x = np.zeros(ex["input_shape"])
        w = np.arange(np.prod(ex["weights_shape"]), dtype=np.float64).reshape(ex["weights_shape"])
        idx = np.zeros(ex["group_indices_shape"], dtype=np.int64)
        out, st = oracle.grouped_matmul(x, w, idx)
        assert st == oracle.OK
        assert list(out.shape) == ex["expected_shape"]
        return
    bias = None if ex["bias"] is None else np.array(ex["bias"])
    for decomposed in (False, True):
        out, st = oracle.grouped_matmul(np.array(ex["input"]), np.array(ex["weights"]),
                                        np.array(ex["group_indices"]), bias,
                                        decomposed=decomposed)
        assert st == oracle.OK
        np.testing.assert_allclose(out, np.array(ex["expected"], dtype=np.float64),
                                   rtol=0, atol=1e-12)


def test_gmm_decomposition_matches_direct_exactly():
    rng = np.random.default_rng(11)
    M, K, G, N, S = 7, 5, 4, 6, 3
    x = rng.integers(-4, 5, (M, K)).astype(np.float64)
    w = rng.integers(-4, 5, (G, K, N)).astype(np.float64)
    b = rng.integers(-4, 5, (G, N)).astype(np.float64)
    idx = rng.integers(0, G, (M, S))
    a, st1 = oracle.grouped_matmul(x, w, idx, b)
    d, st2 = oracle.grouped_matmul(x, w, idx, b, decomposed=True)
    assert st1 == st2 == oracle.OK
    assert np.array_equal(a, d)


def test_gmm_matches_einsum():
    rng = np.random.default_rng(12)
    M, K, G, N, S = 9, 33, 5, 17, 2
    x = rng.standard_normal((M, K))
    w = rng.standard_normal((G, K, N))
    b = rng.standard_normal((G, N))
    idx = rng.integers(0, G, (M, S))
    out, st = oracle.grouped_matmul(x, w, idx, b)
    assert st == oracle.OK
    ref = np.einsum("mk,mskn->msn", x, w[idx]) + b[idx]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bad", [-1, 3, 100])
def test_gmm_out_of_range_index_reported(bad):
    x = np.ones((2, 2))
    w = np.ones((3, 2, 2))
    idx = np.array([[0], [bad]])
    _, st = oracle.grouped_matmul(x, w, idx)
    assert st == oracle.BAD_INDEX


# ----------------------------------------------------------------------------
# Dequantization codes
# ----------------------------------------------------------------------------

def test_nibble_codes_low_first():
    # byte 0x8F: element 0 = low nibble 15 -> +7, element 1 = high nibble 8 -> 0
    out = oracle.dequant_rows(np.array([[0x8F]], np.uint8), np.array([[1.0]], np.float32),
                              2, 4, 0)
    assert out.tolist() == [[7.0, 0.0]]
    out = oracle.dequant_rows(np.array([[0x07]], np.uint8), np.array([[0.5]], np.float32),
                              2, 4, 0)
    assert out.tolist() == [[-0.5, -4.0]]


def test_byte_codes_8bit():
    out = oracle.dequant_rows(np.array([[0x00, 0x80, 0xFF]], np.uint8),
                              np.array([[2.0]], np.float32), 3, 8, 0)
    assert out.tolist() == [[-256.0, 0.0, 254.0]]


def test_block_scale_indexing():
    codes = np.full((1, 32), 128, np.uint8)
    codes[0, 3] = 130
    codes[0, 20] = 125
    out = oracle.dequant_rows(codes, np.array([[0.5, 2.0]], np.float32), 32, 8, 16)
    assert out[0, 3] == 1.0 and out[0, 20] == -6.0
    assert np.count_nonzero(out) == 2


# ----------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------

def test_route_hand_case():
    sel, p = oracle.route(np.array([[1.0, 3.0, 2.0, 0.0]], np.float32), 2)
    assert sel.tolist() == [[1, 2]]
    e1 = math.exp(-1.0)
    np.testing.assert_allclose(p[0], [1 / (1 + e1), e1 / (1 + e1)], rtol=1e-15)


def test_route_tie_goes_to_lower_index():
    sel, _ = oracle.route(np.array([[1.0, 1.0, 0.0]], np.float32), 1)
    assert sel.tolist() == [[0]]
    sel, p = oracle.route(np.array([[0.0, 2.0, 2.0]], np.float32), 2)
    assert sel.tolist() == [[1, 2]]
    assert p.tolist() == [[0.5, 0.5]]


def test_route_k1_weight_exactly_one():
    lg = np.random.default_rng(3).standard_normal((50, 16)).astype(np.float32)
    _, p = oracle.route(lg, 1)
    assert np.all(p == 1.0)


def test_route_k_equals_e_is_full_softmax():
    from scipy.special import softmax
    lg = np.random.default_rng(4).standard_normal((20, 8)).astype(np.float32)
    sel, p = oracle.route(lg, 8)
    full = softmax(lg.astype(np.float64), axis=1)
    for t in range(20):
        np.testing.assert_allclose(p[t], full[t, sel[t]], rtol=1e-14)
        assert sorted(sel[t].tolist()) == list(range(8))
        assert np.all(np.diff(lg[t, sel[t]]) <= 0)


# ----------------------------------------------------------------------------
# Hand-computed layers
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("case", _load("qmoe_hand_cases.json")["cases"], ids=lambda c: c["name"])
def test_qmoe_hand_cases(case):
    y, sel, p = oracle.qmoe(np.array(case["x"], np.float32), np.array(case["logits"], np.float32),
                            np.array(case["w1"], np.uint8), np.array(case["s1"], np.float32),
                            np.array(case["w2"], np.uint8), np.array(case["s2"], np.float32),
                            k=case["k"], expert_weight_bits=case["bits"],
                            block_size=case["block_size"], activation_type=case["activation"],
                            activation_alpha=case["alpha"], activation_beta=case["beta"])
    assert sel.tolist() == case["expected_sel"]
    np.testing.assert_allclose(p, case["expected_p"], rtol=1e-15)
    np.testing.assert_allclose(y, case["expected_y"], rtol=1e-14, atol=1e-15)


def test_swiglu_limit_reading():
    # Reading of the swiglu_limit attribute (no page value pins it): the gate is
    # clamped from above, the linear branch on both sides.
    # g = 10 -> 5, u = -20 -> -5: a = 5 * sigmoid(5) * (-5).
    a = oracle.activation(np.array([10.0, -20.0]), 1, "swiglu", swiglu_limit=5.0)
    assert a[0] == pytest.approx(-25.0 / (1.0 + math.exp(-5.0)), rel=1e-15)
    a = oracle.activation(np.array([-10.0, 20.0]), 1, "swiglu", swiglu_limit=5.0)
    assert a[0] == pytest.approx(-10.0 / (1.0 + math.exp(10.0)) * 5.0, rel=1e-15)


# ----------------------------------------------------------------------------
# Invariants and brute force on small random layers
# ----------------------------------------------------------------------------

def _rand_layer(seed, T=6, H=32, I=16, E=5, k=2, bits=4, bs=0, act="swiglu"):
    rng = np.random.default_rng(seed)
    f = 2 if act == "swiglu" else 1
    pk = 2 if bits == 4 else 1
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    w1 = rng.integers(0, 256, (E, f * I, H // pk), dtype=np.uint8)
    w2 = rng.integers(0, 256, (E, H, I // pk), dtype=np.uint8)
    if bs:
        s1 = rng.uniform(0.01, 0.05, (E, f * I, H // bs)).astype(np.float32)
        s2 = rng.uniform(0.01, 0.05, (E, H, I // bs)).astype(np.float32)
    else:
        s1 = rng.uniform(0.01, 0.05, (E, f * I)).astype(np.float32)
        s2 = rng.uniform(0.01, 0.05, (E, H)).astype(np.float32)
    attrs = dict(k=k, expert_weight_bits=bits, block_size=bs, activation_type=act)
    return x, lg, w1, s1, w2, s2, attrs


def test_zero_scales_give_exact_zero():
    for act in ("relu", "swiglu"):
        x, lg, w1, s1, w2, s2, attrs = _rand_layer(5, act=act)
        y, _, _ = oracle.qmoe(x, lg, w1, s1 * 0, w2, s2, activation_beta=0.7, **attrs)
        assert np.all(y == 0.0)


def test_relu_all_negative_preactivation_gives_zero():
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(6, act="relu", bits=8)
    x = np.abs(x) + 0.1
    w1 = np.full_like(w1, 100)           # code 100 - 128 < 0 with positive scales
    y, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("bits,bs,act", [(4, 0, "swiglu"), (8, 16, "relu"), (4, 16, "swiglu")])
def test_dense_brute_force_matches(bits, bs, act):
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(7, bits=bits, bs=bs, act=act, E=4, k=2)
    y, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    yd, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, dense=True, **attrs)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_expert_permutation_invariance():
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(8, E=6, k=3)
    y, sel, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    perm = np.random.default_rng(9).permutation(6)
    y2, sel2, _ = oracle.qmoe(x, lg[:, perm], w1[perm], s1[perm], w2[perm], s2[perm], **attrs)
    np.testing.assert_allclose(y2, y, rtol=1e-13, atol=1e-13)
    assert np.array_equal(perm[sel2], sel)


def test_4bit_equals_8bit_repack():
    rng = np.random.default_rng(10)
    T, H, I, E = 5, 16, 8, 3
    c1 = rng.integers(-8, 8, (E, 2 * I, H))
    c2 = rng.integers(-8, 8, (E, H, I))

    def pack4(c):
        u = (c + 8).astype(np.uint8)
        return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)

    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    s1 = rng.uniform(0.01, 0.05, (E, 2 * I)).astype(np.float32)
    s2 = rng.uniform(0.01, 0.05, (E, H)).astype(np.float32)
    kw = dict(k=2, activation_type="swiglu")
    y4, _, _ = oracle.qmoe(x, lg, pack4(c1), s1, pack4(c2), s2, expert_weight_bits=4, **kw)
    y8, _, _ = oracle.qmoe(x, lg, (c1 + 128).astype(np.uint8), s1, (c2 + 128).astype(np.uint8),
                           s2, expert_weight_bits=8, **kw)
    assert np.array_equal(y4, y8)


def test_columnwise_equals_blockwise_with_equal_scales():
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(13, H=64, I=32, bs=0)
    bs = 16
    s1b = np.repeat(s1[:, :, None], 64 // bs, axis=2)
    s2b = np.repeat(s2[:, :, None], 32 // bs, axis=2)
    y, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    attrs["block_size"] = bs
    yb, _, _ = oracle.qmoe(x, lg, w1, s1b, w2, s2b, **attrs)
    assert np.array_equal(y, yb)


def test_rank3_equals_rank2():
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(14, T=6)
    y2, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    y3, _, _ = oracle.qmoe(x.reshape(2, 3, -1), lg, w1, s1, w2, s2, **attrs)
    assert np.array_equal(y2, y3)


def test_token_subset_and_threads_match_full():
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(15, T=12)
    y, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    sub = np.array([1, 5, 11])
    ys, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2, tokens=sub, nthreads=3, **attrs)
    assert np.array_equal(ys, y[sub])


def test_qmoe_equals_grouped_matmul_composition():
    """QMoE as DequantizeLinear + GroupedMatMul (GroupedMatMul-29 Summary,
    third paragraph), with the dequantization and softmax done in numpy here."""
    x, lg, w1, s1, w2, s2, attrs = _rand_layer(16, T=7, H=32, I=16, E=5, k=3, bits=4, bs=16)
    T, H = x.shape
    E, I, k = 5, 16, 3

    def np_dequant4(packed, scales, K, bs):
        lo = (packed & 0x0F).astype(np.int64)
        hi = (packed >> 4).astype(np.int64)
        codes = np.empty(packed.shape[:-1] + (K,), np.int64)
        codes[..., 0::2] = lo
        codes[..., 1::2] = hi
        sc = np.repeat(scales.astype(np.float64), bs, axis=-1)
        return (codes - 8) * sc

    W1 = np_dequant4(w1, s1, H, 16)                # [E, 2I, H]
    W2 = np_dequant4(w2, s2, I, 16)                # [E, H, I]
    order = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :k]
    sel_lg = np.take_along_axis(lg.astype(np.float64), order, 1)
    p = np.exp(sel_lg - sel_lg[:, :1])
    p /= p.sum(1, keepdims=True)
    h, st = oracle.grouped_matmul(x, np.transpose(W1, (0, 2, 1)), order)   # [T,k,2I]
    assert st == oracle.OK
    g, u = h[..., 0::2], h[..., 1::2]
    a = g / (1.0 + np.exp(-g)) * u                                          # [T,k,I]
    o, st = oracle.grouped_matmul(a.reshape(T * k, I), np.transpose(W2, (0, 2, 1)),
                                  order.reshape(T * k, 1))
    assert st == oracle.OK
    y_ref = (o.reshape(T, k, H) * p[:, :, None]).sum(1)
    y, sel, pp = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)
    assert np.array_equal(sel, order)
    np.testing.assert_allclose(pp, p, rtol=1e-14)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)


def test_inter_zero_gives_zero():
    x = np.ones((3, 4), np.float32)
    lg = np.array([[0.1, 0.2]] * 3, np.float32)
    y, _, _ = oracle.qmoe(x, lg, np.zeros((2, 0, 2), np.uint8), np.zeros((2, 0), np.float32),
                          np.zeros((2, 4, 0), np.uint8), np.zeros((2, 4), np.float32), k=1)
    assert np.all(y == 0.0) and y.shape == (3, 4)
