"""The seeded input generators hold to their stated recipe (CPU only).

The five QMoE configurations keep the shapes, expert counts, k, bit widths, scale
layouts and activations of the benchmark table; router logits have no tie among
each row's k+1 largest values (so the selected set is unique); the many-small
configuration's Zipf bias skews expert load; every generator is deterministic
in (workload, tensor, salt).  Only the small tensors are drawn here: the large
configurations are checked through their logits and their declared shapes.
"""
import numpy as np
import pytest

from quantized_mixture_experts_gb300 import workloads as W

# input shape, T, H, I, E, k, bits, block size (0 = column-wise), activation
TABLE = {
    "tiny": ((16, 64), 16, 64, 128, 4, 2, 4, 0, "relu"),
    "decode": ((8, 4096), 8, 4096, 14336, 8, 2, 4, 32, "swiglu"),
    "prefill": ((2, 2048, 4096), 4096, 4096, 14336, 8, 2, 4, 128, "swiglu"),
    "many_small": ((2048, 2048), 2048, 2048, 1024, 64, 8, 8, 0, "swiglu"),
    "large_e": ((4, 4096, 2048), 16384, 2048, 768, 128, 8, 4, 64, "swiglu"),
}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_config_table(name):
    wl = W.WORKLOADS[name]
    got = (wl.input_shape, wl.tokens, wl.hidden, wl.inter, wl.experts, wl.k, wl.bits,
           wl.block_size, wl.activation)
    assert got == TABLE[name]
    # block sizes divide hidden and inter (quantBlockSizeOk)
    if wl.block_size:
        assert wl.hidden % wl.block_size == 0 and wl.inter % wl.block_size == 0


def test_tiny_tensor_shapes_and_ranges():
    wl = W.WORKLOADS["tiny"]
    d = W.make_inputs(wl)
    assert d["input"].shape == (16, 64) and d["input"].dtype == np.float32
    assert d["router_probs"].shape == (16, 4)
    assert d["fc1_experts_weights"].shape == (4, 128, 32)
    assert d["fc2_experts_weights"].shape == (4, 64, 64)
    assert d["fc1_scales"].shape == (4, 128) and d["fc2_scales"].shape == (4, 64)
    for s in (d["fc1_scales"], d["fc2_scales"]):
        assert s.min() >= 0.005 and s.max() <= 0.02
    w = d["fc1_experts_weights"]
    lo, hi = w & 0xF, w >> 4
    assert set(np.unique(lo)) == set(range(16)) and set(np.unique(hi)) == set(range(16))


@pytest.mark.parametrize("name", sorted(TABLE))
def test_logits_have_unique_top_k_plus_one(name):
    wl = W.WORKLOADS[name]
    lg = W._logits(wl, wl.tokens, 0)
    assert lg.shape == (wl.tokens, wl.experts) and lg.dtype == np.float32
    m = min(wl.k + 1, wl.experts)
    top = -np.sort(-lg, axis=1)[:, :m]
    assert np.all(top[:, :-1] > top[:, 1:])
    if wl.zipf_s == 0 and lg.size >= 10000:   # enough draws for the spread to show
        assert abs(float(lg.std()) - wl.logit_sigma) < 0.05 * wl.logit_sigma


def test_many_small_load_is_skewed():
    wl = W.WORKLOADS["many_small"]
    lg = W._logits(wl, wl.tokens, 0)
    sel = np.argsort(-lg, axis=1, kind="stable")[:, :wl.k]
    load = np.bincount(sel.ravel(), minlength=wl.experts)
    perm = W._rng(wl, 7, 0).permutation(wl.experts)
    # the expert with bias 0 (perm 0) is the most popular; the least popular
    # experts (largest perm) receive far fewer tokens than the mean
    assert load[int(np.argmin(perm))] == load.max()
    assert load.max() > 3 * load.mean()
    tail = load[np.argsort(perm)[-16:]]
    assert tail.mean() < 0.5 * load.mean()


def test_generators_are_deterministic_and_salted():
    wl = W.WORKLOADS["tiny"]
    a, b, c = W.make_inputs(wl), W.make_inputs(wl), W.make_inputs(wl, salt=1)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k])


def test_float_tiny_recipe():
    wl = W.FLOAT_WORKLOADS["float_tiny"]
    d = W.make_float_inputs(wl)
    assert d["fc1_experts_weights"].shape == (4, 128, 64)
    assert d["fc2_experts_weights"].shape == (4, 64, 128)
    assert abs(float(d["fc1_experts_weights"].std()) * np.sqrt(64) - 1) < 0.05
    assert abs(float(d["fc2_experts_weights"].std()) * np.sqrt(128) - 1) < 0.05
    assert abs(float(d["fc1_experts_bias"].std()) - 0.1) < 0.02


def test_qkv_tiny_recipe():
    wl = W.QKV_WORKLOADS["qkv_tiny"]
    d = W.make_qkv_inputs(wl)
    assert d["q_B"].shape == (128, 8, 16) and d["k_B"].shape == (64, 8, 16)
    assert d["q_scales"].shape == (128, 8)
    assert d["norm_scale"].min() >= 0.5 and d["norm_scale"].max() <= 1.5
    assert "skip" in d and d["skip"].shape == wl.input_shape


def test_gmm_recipe():
    wl = W.GMM_WORKLOADS["gmm_tiny"]
    d = W.make_gmm_inputs(wl)
    x, w, idx = d["input"], d["weights"], d["group_indices"]
    assert x.shape == (300, 128) and w.shape == (5, 128, 200) and idx.shape == (300, 2)
    assert idx.dtype == np.int64 and idx.min() >= 0 and idx.max() < wl.G
    assert np.all(idx[:, 0] != idx[:, 1])          # S distinct groups per row
    assert np.abs(x).max() <= np.sqrt(3.0) and abs(float(x.var()) - 1) < 0.05
    assert np.abs(w).max() <= np.sqrt(3.0 / wl.K) and abs(float(w.var()) * wl.K - 1) < 0.05
    # every group is used, roughly evenly
    load = np.bincount(idx.ravel(), minlength=wl.G)
    assert load.min() > 0.7 * load.mean()
    big = W.GMM_WORKLOADS["gmm_prefill"]
    assert (big.M, big.K, big.G, big.N, big.S) == (4096, 4096, 8, 2 * 14336, 2)
    assert big.flops == 2 * 4096 * 2 * 4096 * 28672
