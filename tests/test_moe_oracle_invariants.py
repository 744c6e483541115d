"""Invariants of the float MoE definition (com.microsoft.MoE README: Description,
Attributes), checked on the CPU oracle over a seeded sweep of configurations.

Each property follows from the README's definition, not from the oracle's code:
the softmax over all logits is unchanged by a per-token shift; normalising the
selected weights divides each token's output by the sum of its unnormalised
selected weights; FC2 is affine, so scaling its weights and bias by c scales the
output by c; without biases, identity and ReLU layers are positively homogeneous
in x; SwiGLU, in each of its three row layouts, is affine in beta; relabelling
experts changes nothing.
"""
import itertools
import zlib

import numpy as np
import pytest

import oracle

ACTS = [("relu", 0, False), ("gelu", 0, False), ("silu", 0, True), ("identity", 0, False),
        ("swiglu", 0, True), ("swiglu", 1, False), ("swiglu", 2, False)]
SWEEP = [dict(act=a, fusion=f, fc3=f3, k=k, E=E, biases=b, normalize=nz)
         for ((a, f, f3), (k, E), b, nz) in itertools.product(
             ACTS, ((1, 3), (2, 5), (4, 4)), (False, True), (0, 1))]


def _ids(c):
    return "{act}{fusion}-fc3{fc3:d}-k{k}of{E}-b{biases:d}-n{normalize}".format(**c)


def _layer(seed, act, fusion, fc3, k, E, biases, normalize, T=4, H=24, I=16):
    rng = np.random.default_rng(seed)
    rows = 2 * I if act == "swiglu" and fusion != 0 else I
    d = dict(x=rng.standard_normal((T, H)).astype(np.float32),
             logits=rng.standard_normal((T, E)).astype(np.float32),
             fc1_w=(rng.standard_normal((E, rows, H)) / np.sqrt(H)).astype(np.float32),
             fc2_w=(rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32))
    kw = dict(k=k, activation_type=act, swiglu_fusion=fusion, normalize_routing_weights=normalize)
    if fc3:
        kw["fc3_w"] = (rng.standard_normal((E, I, H)) / np.sqrt(H)).astype(np.float32)
    if biases:
        kw["fc1_bias"] = (0.1 * rng.standard_normal((E, rows))).astype(np.float32)
        kw["fc2_bias"] = (0.1 * rng.standard_normal((E, H))).astype(np.float32)
        if fc3:
            kw["fc3_bias"] = (0.1 * rng.standard_normal((E, I))).astype(np.float32)
    return d, kw


def _run(d, kw, **over):
    args = dict(kw, **over)
    return oracle.moe(d["x"], d["logits"], d["fc1_w"], d["fc2_w"], **args)


def _close(a, b, rtol=1e-12):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=rtol * max(1.0, float(np.abs(b).max())))


@pytest.mark.parametrize("cfg", SWEEP, ids=[_ids(c) for c in SWEEP])
def test_invariants(cfg):
    seed = zlib.crc32(_ids(cfg).encode())
    d, kw = _layer(seed, **cfg)
    y, sel, w = _run(d, kw)

    # per-token logit shift
    shifted = dict(d, logits=d["logits"] + np.float32(4.0) *
                   np.arange(1, d["x"].shape[0] + 1, dtype=np.float32)[:, None])
    y_s, sel_s, w_s = _run(shifted, kw)
    assert np.array_equal(sel_s, sel)
    _close(w_s, w, 1e-6)
    _close(y_s, y, 1e-5)

    # normalising divides by the sum of the unnormalised selected weights
    y0, _, w0 = _run(d, kw, normalize_routing_weights=0)
    y1, _, w1 = _run(d, kw, normalize_routing_weights=1)
    _close(w1, w0 / w0.sum(1, keepdims=True))
    _close(y1, y0 / w0.sum(1, keepdims=True))

    # FC2 weights and bias scaled by 4 (exact): output scaled by 4
    over = dict(kw)
    if "fc2_bias" in kw:
        over["fc2_bias"] = kw["fc2_bias"] * np.float32(4.0)
    y_c, _, _ = _run(dict(d, fc2_w=d["fc2_w"] * np.float32(4.0)), over)
    _close(y_c, 4.0 * y)

    if cfg["act"] in ("relu", "identity") and not cfg["biases"]:
        y_x, _, _ = _run(dict(d, x=d["x"] * np.float32(2.0)), kw)
        _close(y_x, 2.0 * y)
    if cfg["act"] == "swiglu":
        ys = [_run(d, kw, activation_beta=b)[0] for b in (0.0, 1.0, 2.0)]
        _close(ys[2] - ys[1], ys[1] - ys[0], 1e-10)

    # relabelling experts
    perm = np.random.default_rng(seed + 1).permutation(cfg["E"])
    dp = dict(d, logits=d["logits"][:, perm], fc1_w=d["fc1_w"][perm], fc2_w=d["fc2_w"][perm])
    kp = {key: (val[perm] if isinstance(val, np.ndarray) else val) for key, val in kw.items()}
    y_p, sel_p, _ = _run(dp, kp)
    _close(y_p, y, 1e-13)
    assert np.array_equal(perm[sel_p], sel)
