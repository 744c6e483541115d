"""GPU parity of the float MoE layer (com.microsoft.MoE README) against the
fp64 oracle, through the C ABI.

Small layers cover every activation and SwiGLU layout, biases, both routing
modes, ragged tails and several token tiles per expert on both kernel paths
(TF32 tensor cores and scalar fp32), compared on every token.  The decode and
prefill workloads at full size are compared on a seeded token sample that
touches every selected expert.
"""
import os

import numpy as np
import pytest

import oracle
from helpers import check_outputs, check_routing
from quantized_mixture_experts_gb300.workloads import (FLOAT_WORKLOADS, FloatWorkload,
                                                       make_float_inputs, sample_tokens,
                                                       tied_logits)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OPTIONAL = ("fc1_experts_bias", "fc2_experts_bias", "fc3_experts_weights", "fc3_experts_bias")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _to_dev(inp, dev):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in inp.items()}


def _run(wl: FloatWorkload, t: dict, path: int, dev):
    import quantized_mixture_experts_gb300 as q
    attrs = q.make_moe_attrs(path=path, **wl.attrs())
    T = t["router_probs"].shape[0]
    sel = torch.full((T, wl.k), -7, dtype=torch.int32, device=dev)
    pw = torch.full((T, wl.k), -7.0, dtype=torch.float32, device=dev)
    y = q.moe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                      t["fc2_experts_weights"], attrs=attrs, topk_idx=sel, topk_w=pw,
                      **{k: t.get(k) for k in OPTIONAL})
    torch.cuda.synchronize()
    H = t["input"].shape[-1]
    return (y.reshape(-1, H).cpu().numpy().astype(np.float64), sel.cpu().numpy(),
            pw.cpu().numpy().astype(np.float64))


def _reference(wl: FloatWorkload, inp: dict, tokens=None):
    return oracle.moe(inp["input"], inp["router_probs"], inp["fc1_experts_weights"],
                      inp["fc2_experts_weights"], fc1_bias=inp.get("fc1_experts_bias"),
                      fc2_bias=inp.get("fc2_experts_bias"),
                      fc3_w=inp.get("fc3_experts_weights"),
                      fc3_bias=inp.get("fc3_experts_bias"), tokens=tokens,
                      nthreads=os.cpu_count() or 1, **wl.attrs())


SMALL = [
    FLOAT_WORKLOADS["float_tiny"],
    FloatWorkload("gelu_ragged_norm", 50, (37, 96), 96, 64, 6, 2, "gelu", biases=True,
                  normalize=1),
    FloatWorkload("identity_k1", 51, (40, 64), 64, 96, 5, 1, "identity"),
    FloatWorkload("silu_no_fc3", 52, (33, 128), 128, 64, 4, 2, "silu", biases=True),
    FloatWorkload("silu_fc3", 53, (50, 64), 64, 128, 8, 3, "silu", fc3=True, biases=True),
    FloatWorkload("swiglu_fc3", 54, (64, 128), 128, 96, 8, 2, "swiglu", swiglu_fusion=0,
                  fc3=True, biases=True, alpha=1.702, beta=1.0),
    FloatWorkload("swiglu_interleaved", 55, (45, 64), 64, 160, 4, 2, "swiglu", swiglu_fusion=1,
                  biases=True, normalize=1),
    FloatWorkload("swiglu_concat_limit", 56, (30, 96), 96, 64, 4, 2, "swiglu", swiglu_fusion=2,
                  alpha=1.5, beta=0.5, swiglu_limit=0.7),
    # several token tiles per expert, ragged last tile, 128-row tail of FC2 output rows
    FloatWorkload("two_tiles_relu", 57, (600, 160), 160, 96, 2, 1, "relu", biases=True),
    FloatWorkload("k_eq_E_swiglu", 58, (24, 64), 64, 64, 4, 4, "swiglu", swiglu_fusion=2),
    FloatWorkload("rank3_many_experts", 59, (2, 96, 128), 128, 64, 64, 8, "swiglu",
                  swiglu_fusion=0, fc3=True, normalize=1),
    FloatWorkload("decode_like", 60, (8, 512), 512, 1024, 8, 2, "swiglu", swiglu_fusion=0,
                  fc3=True, logit_sigma=2.0),
    FloatWorkload("odd_hidden_generic", 61, (20, 40), 40, 24, 3, 2, "gelu", biases=True),
    # batches of 128+ routed rows run on CTA pairs (cta_group::2): every SwiGLU layout, an
    # unpaired activation, ragged tiles and several tiles per expert
    FloatWorkload("pair_interleaved", 64, (300, 64), 64, 160, 4, 2, "swiglu", swiglu_fusion=1,
                  biases=True),
    FloatWorkload("pair_concat_limit", 65, (200, 96), 96, 96, 4, 2, "swiglu", swiglu_fusion=2,
                  alpha=1.3, beta=0.2, swiglu_limit=0.8, normalize=1),
    FloatWorkload("pair_gelu_k1", 66, (260, 96), 96, 288, 8, 1, "gelu", biases=True),
    FloatWorkload("pair_fc3_tiles", 67, (700, 128), 128, 96, 2, 1, "swiglu", swiglu_fusion=0,
                  fc3=True, biases=True),
    # past 4096 slots (multi-CTA routing): all-expert softmax over 200 experts (eight
    # register slots per lane) with the serial in-chunk ranking (k = 20), renormalised
    FloatWorkload("route_e200_k20", 68, (300, 64), 64, 64, 200, 20, "relu", normalize=1),
]


def _paths(wl: FloatWorkload):
    import quantized_mixture_experts_gb300 as q
    out = []
    for path in (q.MOE_PATH_AUTO, q.MOE_PATH_GROUPED, q.MOE_PATH_GENERIC):
        a = q.make_moe_attrs(path=path, **wl.attrs())
        try:
            q.moe_choose_path(wl.input_shape, (wl.experts, wl.fc1_rows, wl.hidden), a)
        except q.QmoeError as e:
            assert e.status == q.binding.ERR_NOT_SUPPORTED
            continue
        out.append(path)
    return out


def _cases():
    return [pytest.param(wl, p, id=f"{wl.name}-p{p}") for wl in SMALL for p in _paths(wl)]


@pytest.mark.parametrize("wl,path", _cases())
def test_small_parity_all_tokens(dev, wl, path):
    inp = make_float_inputs(wl)
    y_ref, sel_ref, w_ref = _reference(wl, inp)
    y, sel, w = _run(wl, _to_dev(inp, dev), path, dev)
    check_routing(sel, w, sel_ref, w_ref, wl.name)
    check_outputs(y, y_ref, f"{wl.name} path {path}")


# All-expert softmax routing with exact ties in the logits (so in the
# probabilities): the oracle takes the k most probable experts ordered by
# (probability descending, index ascending).  Register selection at 1, 2 and 8
# slots per lane, the general selection (E > 256), the one-launch and the
# multi-CTA routing kernels, with and without renormalisation.
TIES = [
    FloatWorkload("tie_e8_k2", 70, (16, 64), 64, 64, 8, 2, "relu"),
    FloatWorkload("tie_e64_k8_norm", 71, (64, 64), 64, 64, 64, 8, "silu", normalize=1),
    FloatWorkload("tie_e200_k8_multi", 72, (600, 64), 64, 64, 200, 8, "relu", normalize=1),
    FloatWorkload("tie_e300_k4_general", 73, (40, 64), 64, 64, 300, 4, "gelu"),
]


@pytest.mark.parametrize("wl,path", [pytest.param(w, p, id=f"{w.name}-p{p}")
                                     for w in TIES for p in _paths(w)])
def test_tied_logits_select_like_the_oracle(dev, wl, path):
    inp = make_float_inputs(wl)
    inp["router_probs"] = tied_logits(wl.tokens, wl.experts, seed=wl.index)
    srt = -np.sort(-inp["router_probs"], axis=1)
    assert np.mean(srt[:, wl.k - 1] == srt[:, wl.k]) > 0.3
    y_ref, sel_ref, w_ref = _reference(wl, inp)
    y, sel, w = _run(wl, _to_dev(inp, dev), path, dev)
    check_routing(sel, w, sel_ref, w_ref, f"{wl.name} path {path} (tied logits)")
    check_outputs(y, y_ref, f"{wl.name} path {path} (tied logits)")


def test_tensor_core_path_is_taken(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[5]
    assert q.moe_choose_path(wl.input_shape, (wl.experts, wl.fc1_rows, wl.hidden),
                             q.make_moe_attrs(**wl.attrs())) == q.MOE_PATH_GROUPED
    t = _to_dev(make_float_inputs(wl), dev)
    n0 = q.launch_count()
    _run(wl, t, q.MOE_PATH_AUTO, dev)
    # routing + grouping, gather, FC1, FC2, combine
    assert q.launch_count() - n0 >= 5


def test_repeat_is_bit_identical(dev):
    wl = SMALL[4]
    t = _to_dev(make_float_inputs(wl), dev)
    a = _run(wl, t, 0, dev)
    b = _run(wl, t, 0, dev)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_empty_batch_and_zero_inter(dev):
    import quantized_mixture_experts_gb300 as q
    wl = FloatWorkload("empty", 62, (0, 64), 64, 32, 4, 2, "relu")
    x = torch.zeros((0, 64), device=dev)
    lg = torch.zeros((0, 4), device=dev)
    w1 = torch.zeros((4, 32, 64), device=dev)
    w2 = torch.zeros((4, 64, 32), device=dev)
    y = q.moe_forward(x, lg, w1, w2, **wl.attrs())
    assert y.shape == (0, 64)
    # inter_size 0: FC2 reduces to its bias, weighted by the routing weights
    inp = make_float_inputs(FloatWorkload("zi", 63, (10, 64), 64, 8, 4, 2, "relu", biases=True))
    inp["fc1_experts_weights"] = inp["fc1_experts_weights"][:, :0]
    inp["fc1_experts_bias"] = inp["fc1_experts_bias"][:, :0]
    inp["fc2_experts_weights"] = inp["fc2_experts_weights"][:, :, :0]
    wz = FloatWorkload("zi", 63, (10, 64), 64, 0, 4, 2, "relu", biases=True)
    y_ref, sel_ref, w_ref = _reference(wz, inp)
    y, sel, w = _run(wz, _to_dev(inp, dev), q.MOE_PATH_AUTO, dev)
    check_routing(sel, w, sel_ref, w_ref, "zero inter")
    check_outputs(y, y_ref, "zero inter")


def test_hostio_matches_device_call(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[5]
    inp = make_float_inputs(wl)
    t = _to_dev(inp, dev)
    y_dev, _, _ = _run(wl, t, 0, dev)
    attrs = q.make_moe_attrs(**wl.attrs())
    ws = q.alloc_workspace(q.moe_workspace_size(wl.input_shape, (wl.experts, wl.fc1_rows,
                                                                 wl.hidden), attrs, hostio=True),
                           dev)
    hx = torch.from_numpy(inp["input"]).pin_memory()
    hl = torch.from_numpy(inp["router_probs"]).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    q.moe_forward_hostio(hx, hl, t["fc1_experts_weights"], t["fc2_experts_weights"], hy,
                         attrs=attrs, workspace=ws, **{k: t.get(k) for k in OPTIONAL})
    torch.cuda.synchronize()
    assert np.array_equal(hy.numpy().reshape(y_dev.shape).astype(np.float64), y_dev)


def test_misaligned_weights_fall_back_to_generic(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[2]
    inp = make_float_inputs(wl)
    t = _to_dev(inp, dev)
    # the same FC1 weights at an address 4 bytes past a 16-byte boundary
    buf = torch.empty(t["fc1_experts_weights"].numel() + 1, device=dev)
    w1 = buf[1:].view_as(t["fc1_experts_weights"])
    w1.copy_(t["fc1_experts_weights"])
    t["fc1_experts_weights"] = w1
    y_ref, _, _ = _reference(wl, inp)
    y, _, _ = _run(wl, t, q.MOE_PATH_AUTO, dev)
    check_outputs(y, y_ref, "misaligned FC1 weights")
    with pytest.raises(q.QmoeError):
        _run(wl, t, q.MOE_PATH_GROUPED, dev)


@pytest.mark.parametrize("name,n", [("float_decode", 8), ("float_prefill", 48)])
def test_full_size_sampled(dev, name, n):
    wl = FLOAT_WORKLOADS[name]
    inp = make_float_inputs(wl)
    t = _to_dev(inp, dev)
    y, sel, w = _run(wl, t, 0, dev)
    # routing on every token
    sel_all, w_all = oracle.moe_route(inp["router_probs"], wl.k, wl.normalize)
    check_routing(sel, w, sel_all, w_all, name)
    tokens = sample_tokens(sel_all, wl.tokens, n, seed=wl.index)
    y_ref, _, _ = _reference(wl, inp, tokens)
    check_outputs(y[tokens], y_ref, f"{name} sampled")
