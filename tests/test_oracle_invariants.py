"""Invariants of the QMoE definition, checked on the CPU oracle over a seeded sweep
of layer configurations (bit width, scale layout, activation, k, sizes).

Each property follows from the QMoE manifest's definition alone, not from the
oracle's code: the softmax over the selected logits is unchanged by adding a
constant to a token's logits; FC2 is linear, so scaling every FC2 scale by c
scales the output by c; ReLU layers are positively homogeneous in x; the SwiGLU
output a = g * sigmoid(alpha g) * (u + beta) is affine in beta, so the layer is
too; relabelling experts (logit columns and weight tensors together) changes
nothing; a 4-bit code stored as the equivalent 8-bit code (q + 120) gives the
same layer.
"""
import itertools
import zlib

import numpy as np
import pytest

import oracle

SWEEP = [dict(bits=b, bs=bs, act=a, k=k, E=E, T=T, H=H, I=I)
         for (b, bs, a, (k, E), (T, H, I)) in itertools.product(
             (4, 8), (0, 16, 32), ("relu", "swiglu"), ((1, 3), (2, 5), (4, 4)),
             ((3, 32, 32), (5, 64, 16)))
         if not (bs and (H % bs or I % bs))]


def _layer(seed, bits, bs, act, k, E, T, H, I):
    rng = np.random.default_rng(seed)
    f = 2 if act == "swiglu" else 1
    pk = 2 if bits == 4 else 1
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    w1 = rng.integers(0, 256, (E, f * I, H // pk), dtype=np.uint8)
    w2 = rng.integers(0, 256, (E, H, I // pk), dtype=np.uint8)
    s1_shape = (E, f * I, H // bs) if bs else (E, f * I)
    s2_shape = (E, H, I // bs) if bs else (E, H)
    s1 = rng.uniform(0.01, 0.05, s1_shape).astype(np.float32)
    s2 = rng.uniform(0.01, 0.05, s2_shape).astype(np.float32)
    attrs = dict(k=k, expert_weight_bits=bits, block_size=bs, activation_type=act)
    return x, lg, w1, s1, w2, s2, attrs


def _close(a, b, rtol=1e-12):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=rtol * max(1.0, float(np.abs(b).max())))


def _ids(c):
    return "{bits}b-bs{bs}-{act}-k{k}of{E}-T{T}H{H}I{I}".format(**c)


@pytest.mark.parametrize("cfg", SWEEP, ids=[_ids(c) for c in SWEEP])
def test_invariants(cfg):
    seed = zlib.crc32(_ids(cfg).encode())
    x, lg, w1, s1, w2, s2, attrs = _layer(seed, **cfg)
    y, sel, p = oracle.qmoe(x, lg, w1, s1, w2, s2, **attrs)

    # softmax over the selected logits: a per-token shift changes neither choice nor weights
    shift = np.float32(4.0) * np.arange(1, x.shape[0] + 1, dtype=np.float32)[:, None]
    y_s, sel_s, p_s = oracle.qmoe(x, lg + shift, w1, s1, w2, s2, **attrs)
    assert np.array_equal(sel_s, sel)
    _close(p_s, p, 1e-6)        # the shifted fp32 logits differ from the originals by rounding
    _close(y_s, y, 1e-5)

    # FC2 is linear: scaling every FC2 scale by 4 (exact in fp32) scales y by 4
    y_c, _, _ = oracle.qmoe(x, lg, w1, s1, w2, s2 * np.float32(4.0), **attrs)
    _close(y_c, 4.0 * y)

    if cfg["act"] == "relu":
        # ReLU(c v) = c ReLU(v) for c > 0 and routing ignores x
        y_x, _, _ = oracle.qmoe(x * np.float32(2.0), lg, w1, s1, w2, s2, **attrs)
        _close(y_x, 2.0 * y)
    else:
        # affine in beta: y(2) - y(1) == y(1) - y(0)
        ys = [oracle.qmoe(x, lg, w1, s1, w2, s2, activation_beta=b, **attrs)[0] for b in (0., 1., 2.)]
        _close(ys[2] - ys[1], ys[1] - ys[0], 1e-10)

    # relabelling experts
    perm = np.random.default_rng(seed + 1).permutation(cfg["E"])
    y_p, sel_p, _ = oracle.qmoe(x, lg[:, perm], w1[perm], s1[perm], w2[perm], s2[perm], **attrs)
    _close(y_p, y, 1e-13)
    assert np.array_equal(perm[sel_p], sel)

    if cfg["bits"] == 4:
        # the same codes as 8-bit bytes: q8 = (q4 - 8) + 128
        def unpack(w):
            c = np.empty(w.shape[:-1] + (2 * w.shape[-1],), np.int64)
            c[..., 0::2] = w & 0x0F
            c[..., 1::2] = w >> 4
            return (c + 120).astype(np.uint8)
        a8 = dict(attrs, expert_weight_bits=8)
        y8, _, _ = oracle.qmoe(x, lg, unpack(w1), s1, unpack(w2), s2, **a8)
        assert np.array_equal(y8, y)
