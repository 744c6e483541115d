"""Invariants of the RMSNorm + 4-bit Q/K/V projection (com.microsoft.MatMulNBitsQkv
manifest: passes RmsNorm then Projection), checked on the CPU oracle over a seeded
sweep of K (ragged and whole blocks), widths, row counts and skip inputs.

Each property follows from the definition, not from the oracle's code: with the
normalised rows fixed, every output is linear in each weight block, so doubling
the scale of block b changes the output by exactly that block's own contribution
(the output computed with every other block's codes set to the zero point 8);
the contributions of all blocks sum to the output; with epsilon 0 the RMSNorm
makes the outputs invariant to scaling a row by a power of two.
"""
import itertools
import zlib

import numpy as np
import pytest

import oracle

SWEEP = [dict(K=K, Nq=nq, Nkv=nkv, rows=r, skip=sk)
         for (K, (nq, nkv), r, sk) in itertools.product(
             (32, 96, 100, 256), ((8, 4), (24, 8)), (1, 3), (False, True))]


def _ids(c):
    return "K{K}-Nq{Nq}-Nkv{Nkv}-r{rows}-skip{skip:d}".format(**c)


def _inputs(seed, K, Nq, Nkv, rows, skip):
    rng = np.random.default_rng(seed)
    kb = (K + 31) // 32
    d = dict(A=rng.standard_normal((rows, K)), norm_scale=rng.uniform(0.5, 1.5, K),
             skip=0.5 * rng.standard_normal((rows, K)) if skip else None)
    for name, n in (("q", Nq), ("k", Nkv), ("v", Nkv)):
        d[name + "_B"] = rng.integers(0, 256, (n, kb, 16), dtype=np.uint8)
        d[name + "_scales"] = rng.uniform(0.002, 0.01, (n, kb))
    return d


def _run(d, epsilon=oracle.QKV_EPSILON):
    return oracle.qkv(d["A"], d["norm_scale"], d["q_B"], d["q_scales"], d["k_B"], d["k_scales"],
                      d["v_B"], d["v_scales"], skip=d["skip"], epsilon=epsilon)


def _only_block(d, b):
    """The same layer with every block but b holding the zero-point code 8 (0x88)."""
    out = dict(d)
    for name in "qkv":
        B = np.full_like(d[name + "_B"], 0x88)
        B[:, b] = d[name + "_B"][:, b]
        out[name + "_B"] = B
    return out


@pytest.mark.parametrize("cfg", SWEEP, ids=[_ids(c) for c in SWEEP])
def test_invariants(cfg):
    seed = zlib.crc32(_ids(cfg).encode())
    d = _inputs(seed, **cfg)
    base = _run(d)
    kb = (cfg["K"] + 31) // 32
    scale = max(float(np.abs(o).max()) for o in base)

    # block contributions add up to the output
    parts = [_run(_only_block(d, b)) for b in range(kb)]
    for j in range(3):
        np.testing.assert_allclose(sum(p[j] for p in parts), base[j], rtol=0, atol=1e-12 * scale)

    # doubling one block's scales adds exactly that block's contribution
    b = int(np.random.default_rng(seed).integers(kb))
    d2 = dict(d)
    for name in "qkv":
        s = d[name + "_scales"].copy()
        s[:, b] *= 2.0
        d2[name + "_scales"] = s
    doubled = _run(d2)
    for j in range(3):
        np.testing.assert_allclose(doubled[j] - base[j], parts[b][j], rtol=0, atol=1e-12 * scale)

    # RMSNorm with epsilon 0: a row (and its skip) scaled by 4 gives the same outputs
    d4 = dict(d, A=d["A"] * 4.0, skip=None if d["skip"] is None else d["skip"] * 4.0)
    for got, ref in zip(_run(d4, epsilon=0.0), _run(d, epsilon=0.0)):
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13 * scale)
