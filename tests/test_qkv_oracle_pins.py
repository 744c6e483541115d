"""Pins for the RMSNorm + 4-bit Q/K/V projection oracle, independent of its code.

The [MatMulNBitsQkv manifest] (com.microsoft.MatMulNBitsQkv WebGPU kernel
manifest: passes RmsNorm then Projection, derive.defaultZero = 8,
codesPerByte, codeMask, kBlocks, blobSize, outputs residualT) fixes the
operator.  The tests pin the oracle with layers worked out by hand, a numpy
composition, the separately pinned QMoE oracle's 4-bit dequantisation, and
invariants (zero codes, scale linearity, power-of-two input scaling, padding
codes, skip = folded input).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "qkv_hand_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_qkv_hand_cases(case):
    arr = lambda k, dt=np.float64: None if case.get(k) is None else np.array(case[k], dt)
    out = oracle.qkv(arr("A"), arr("norm_scale"), arr("q_B", np.uint8), arr("q_scales"),
                     arr("k_B", np.uint8), arr("k_scales"), arr("v_B", np.uint8),
                     arr("v_scales"), skip=arr("skip"), block_size=case["block_size"],
                     epsilon=case["epsilon"], residual="expected_residual" in case)
    np.testing.assert_allclose(out[0], case["expected_Q"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out[1], case["expected_K"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out[2], case["expected_V"], rtol=1e-14, atol=1e-15)
    if "expected_residual" in case:
        assert np.array_equal(out[3], np.array(case["expected_residual"]))


def _rand(seed, rows=5, K=96, Nq=40, Nkv=24, block=32):
    rng = np.random.default_rng(seed)
    kb = (K + block - 1) // block
    blob = block // 2
    d = dict(
        A=rng.standard_normal((rows, K)),
        norm_scale=rng.uniform(0.5, 1.5, K),
        q_B=rng.integers(0, 256, (Nq, kb, blob), dtype=np.uint8),
        q_scales=rng.uniform(0.01, 0.05, (Nq, kb)),
        k_B=rng.integers(0, 256, (Nkv, kb, blob), dtype=np.uint8),
        k_scales=rng.uniform(0.01, 0.05, (Nkv, kb)),
        v_B=rng.integers(0, 256, (Nkv, kb, blob), dtype=np.uint8),
        v_scales=rng.uniform(0.01, 0.05, (Nkv, kb)))
    return d


def _run(d, **kw):
    return oracle.qkv(d["A"], d["norm_scale"], d["q_B"], d["q_scales"], d["k_B"], d["k_scales"],
                      d["v_B"], d["v_scales"], **kw)


def _np_dequant(B, scales, K, block=32):
    """[N, kBlocks, blob] codes (low nibble first) -> [N, K] float64 weights."""
    N = B.shape[0]
    lo = (B & 15).astype(np.int64)
    hi = (B >> 4).astype(np.int64)
    codes = np.empty(B.shape[:-1] + (block,), np.int64)
    codes[..., 0::2] = lo
    codes[..., 1::2] = hi
    w = (codes - 8) * scales[..., None]
    return w.reshape(N, -1)[:, :K]


@pytest.mark.parametrize("K", [96, 100])
def test_matches_numpy_composition(K):
    d = _rand(1, K=K)
    Q, Ko, V, nrm = _run(d, normed=True)
    x = d["A"]
    ref_n = x / np.sqrt((x * x).mean(1, keepdims=True) + oracle.QKV_EPSILON) * d["norm_scale"]
    np.testing.assert_allclose(nrm, ref_n, rtol=1e-14)
    for out, b, s in ((Q, "q_B", "q_scales"), (Ko, "k_B", "k_scales"), (V, "v_B", "v_scales")):
        np.testing.assert_allclose(out, ref_n @ _np_dequant(d[b], d[s], K).T, rtol=1e-12,
                                   atol=1e-12)


def test_packing_matches_qmoe_oracle_dequant():
    """The [N, kBlocks, 16] layout read as [N, K/2] rows is the QMoE manifest's
    4-bit block-32 packing; the (separately pinned) QMoE oracle dequantises it."""
    d = _rand(2, K=128, Nq=16)
    K = 128
    W = oracle.dequant_rows(d["q_B"].reshape(16, K // 2), d["q_scales"].astype(np.float32), K, 4,
                            32)
    d["q_scales"] = d["q_scales"].astype(np.float32).astype(np.float64)
    Q, _, _, nrm = _run(d, normed=True)
    np.testing.assert_allclose(Q, nrm @ W.T, rtol=1e-12, atol=1e-12)


def test_code_layout_low_nibble_first():
    B = np.zeros((2, 2, 16), np.uint8)
    B[1, 1, 3] = 0x5A      # elements 6 and 7 of block 1 of row 1: codes 10 and 5
    assert oracle.qkv_code(B, 1, 32 + 6, 64) == 0xA
    assert oracle.qkv_code(B, 1, 32 + 7, 64) == 0x5
    assert oracle.qkv_code(B, 0, 32 + 6, 64) == 0


def test_all_zero_point_codes_give_exact_zero():
    d = _rand(3)
    for b in ("q_B", "k_B", "v_B"):
        d[b] = np.full_like(d[b], 0x88)
    for out in _run(d):
        assert np.all(out == 0.0)


def test_zero_norm_scale_gives_exact_zero():
    d = _rand(4)
    d["norm_scale"] = np.zeros_like(d["norm_scale"])
    for out in _run(d):
        assert np.all(out == 0.0)


def test_scale_linearity():
    d = _rand(5)
    a = _run(d)
    for s in ("q_scales", "k_scales", "v_scales"):
        d[s] = d[s] * 2.0
    b = _run(d)
    for x, y in zip(a, b):
        assert np.array_equal(2.0 * x, y)


def test_power_of_two_input_scaling_is_exact_without_epsilon():
    d = _rand(6)
    a = _run(d, epsilon=0.0)
    d["A"] = d["A"] * 64.0
    b = _run(d, epsilon=0.0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_padding_codes_take_no_part():
    d = _rand(7, K=72)                         # 3 blocks, the last with 8 valid codes
    a = _run(d)
    rng = np.random.default_rng(8)
    for b in ("q_B", "k_B", "v_B"):
        d[b][:, 2, 4:] = rng.integers(0, 256, d[b][:, 2, 4:].shape, dtype=np.uint8)
    b = _run(d)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_skip_is_the_folded_input_and_residual():
    d = _rand(9)
    rng = np.random.default_rng(10)
    skip = np.round(rng.standard_normal(d["A"].shape) * 64) / 64      # exact sums
    d["A"] = np.round(d["A"] * 64) / 64
    Q, Ko, V, res = _run(d, skip=skip, residual=True)
    assert np.array_equal(res, d["A"] + skip)
    d2 = dict(d, A=d["A"] + skip)
    Q2, K2, V2 = _run(d2)
    assert np.array_equal(Q, Q2) and np.array_equal(Ko, K2) and np.array_equal(V, V2)


def test_rank3_rows_are_independent():
    d = _rand(11, rows=6)
    Q, Ko, V = _run(d)
    d3 = dict(d, A=d["A"].reshape(2, 3, -1))
    Q3, K3, V3 = _run(d3)
    assert np.array_equal(Q, Q3) and np.array_equal(Ko, K3)
    one = dict(d, A=d["A"][4:5])
    Q1, _, _ = _run(one)
    assert np.array_equal(Q1[0], Q[4])


def test_residual_without_skip_is_rejected():
    with pytest.raises(ValueError):
        _run(_rand(12), residual=True)
