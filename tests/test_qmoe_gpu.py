"""GPU parity of the QMoE layer against the fp64 oracle, through the C ABI.

Small layers (several tiles, ragged tails) are compared on every token; the
five benchmark workloads at full size are compared on every token (tiny,
decode) or on a seeded token sample that touches every selected expert
(prefill, many-small, large-E), in the launch configuration the bench uses.
"""
import os

import numpy as np
import pytest

import oracle
from helpers import check_outputs, check_routing, run_cuda, to_dev
from quantized_mixture_experts_gb300.workloads import (WORKLOADS, Workload, make_inputs,
                                                       sample_tokens, tied_logits)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _paths(wl: Workload):
    """Every kernel path that accepts this shape (AUTO included)."""
    import quantized_mixture_experts_gb300 as q
    out = []
    for path in (q.PATH_AUTO, q.PATH_DECODE, q.PATH_GROUPED, q.PATH_GENERIC):
        a = q.make_attrs(path=path, **wl.attrs())
        try:
            q.choose_path(wl.input_shape, (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack),
                          a)
        except q.QmoeError as e:
            assert e.status == q.binding.ERR_NOT_SUPPORTED
            continue
        out.append(path)
    return out


SMALL = [
    WORKLOADS["tiny"],
    Workload("ragged_swiglu_bs32", 20, (300, 256), 256, 192, 8, 2, 4, 32, "swiglu"),
    Workload("relu_8bit_col", 21, (100, 128), 128, 128, 16, 4, 8, 0, "relu"),
    Workload("k1_bs64", 22, (40, 128), 128, 64, 6, 1, 4, 64, "swiglu"),
    Workload("k_eq_E_8bit_bs16", 23, (24, 64), 64, 64, 4, 4, 8, 16, "swiglu"),
    Workload("limit_alpha_beta", 24, (50, 128), 128, 64, 8, 2, 4, 0, "swiglu",
             alpha=1.7, beta=0.3, swiglu_limit=0.4),
    Workload("decode_like", 25, (8, 512), 512, 1024, 8, 2, 4, 32, "swiglu", logit_sigma=2.0),
    Workload("prefill_like_rank3", 26, (2, 96, 256), 256, 256, 8, 2, 4, 128, "swiglu",
             logit_sigma=2.0),
    Workload("many_small_like", 27, (256, 256), 256, 128, 64, 8, 8, 0, "swiglu", zipf_s=1.1),
    Workload("large_e_like", 28, (2, 256, 256), 256, 128, 128, 8, 4, 64, "swiglu"),
    Workload("odd_hidden_generic", 29, (33, 48), 48, 32, 5, 2, 4, 16, "swiglu"),
    # decode-sized layers: 8-bit, column-wise, ReLU, two token tiles per expert,
    # partial K chunk, block sizes 16/64/128, clamp
    Workload("decode_8bit_col_relu", 30, (12, 256), 256, 384, 6, 2, 8, 0, "relu"),
    Workload("decode_bs16_two_tiles", 31, (16, 640), 640, 256, 2, 2, 4, 16, "swiglu"),
    Workload("decode_bs128_k1", 32, (5, 1024), 1024, 512, 16, 1, 4, 128, "swiglu"),
    Workload("decode_8bit_bs64", 33, (9, 512), 512, 256, 4, 3, 8, 64, "swiglu"),
    Workload("decode_limit", 34, (4, 256), 256, 256, 4, 2, 4, 0, "swiglu", alpha=1.3,
             beta=-0.2, swiglu_limit=0.3),
    # block size 256: FC1 scales staged by TMA (4 blocks per row), FC2 scales read
    # directly (2 blocks per row, not a multiple of four)
    Workload("bs256", 35, (40, 1024), 1024, 512, 4, 2, 4, 256, "swiglu"),
    # 4-bit column-wise codes with two token tiles per expert on the grouped path
    Workload("col4_two_tiles_relu", 36, (600, 256), 256, 128, 4, 2, 4, 0, "relu"),
    # k = E on the decode path: every token reaches every expert
    Workload("decode_k_eq_E", 37, (8, 256), 256, 256, 4, 4, 4, 32, "swiglu"),
    # routing forms past 4096 slots (the multi-CTA routing kernel): eight register slots
    # per lane (128 < E <= 256) with the serial in-chunk ranking (k > 16); the general
    # selection and more than 32 sorted copies per token (k > 32); eight slots with the
    # parallel ranking
    Workload("route_e200_k20", 38, (300, 64), 64, 64, 200, 20, 4, 32, "swiglu"),
    Workload("route_e96_k40", 39, (120, 64), 64, 64, 96, 40, 8, 0, "relu"),
    Workload("route_e150_k8", 40, (600, 128), 128, 128, 150, 8, 4, 64, "swiglu"),
]


def _small_cases():
    cases = []
    for wl in SMALL:
        for path in _paths(wl):
            cases.append(pytest.param(wl, path, id=f"{wl.name}-p{path}"))
    return cases


_ref_cache = {}


def _reference(wl: Workload, inp: dict, tokens=None):
    key = (wl.name, None if tokens is None else tuple(tokens.tolist()))
    if key not in _ref_cache:
        _ref_cache[key] = oracle.qmoe(inp["input"], inp["router_probs"],
                                      inp["fc1_experts_weights"], inp["fc1_scales"],
                                      inp["fc2_experts_weights"], inp["fc2_scales"],
                                      tokens=tokens, nthreads=os.cpu_count() or 1, **wl.attrs())
    return _ref_cache[key]


@pytest.mark.parametrize("wl,path", _small_cases())
def test_small_parity_all_tokens(dev, wl, path):
    inp = make_inputs(wl)
    y_ref, sel_ref, p_ref = _reference(wl, inp)
    y, sel, p = run_cuda(inp, wl.attrs(), path, dev)
    check_routing(sel, p, sel_ref, p_ref, wl.name)
    check_outputs(y, y_ref, f"{wl.name} path {path}")
    if wl.k == 1:
        assert np.all(p == 1.0)


# Router logits with exact ties (including -0 against +0) on every routing form:
# the one-launch small-batch kernel (<= 4096 slots) and the multi-CTA routing
# kernel, each with the register selection at 1, 2, 4 and 8 slots per lane
# (E <= 32, 64, 128, 256) and the general selection (E > 256 or k > 32).  The
# oracle orders the selection by (logit descending, expert index ascending); the
# selected lists must be identical.
TIES = [
    Workload("tie_decode_e8", 60, (8, 256), 256, 256, 8, 2, 4, 32, "swiglu"),
    Workload("tie_e64_k8", 61, (64, 128), 128, 64, 64, 8, 8, 0, "swiglu"),
    Workload("tie_e128_k8_multi", 62, (600, 64), 64, 64, 128, 8, 4, 64, "swiglu"),
    Workload("tie_e150_k8_multi", 63, (600, 64), 64, 64, 150, 8, 4, 32, "swiglu"),
    Workload("tie_e300_k4_general", 64, (40, 64), 64, 64, 300, 4, 8, 0, "relu"),
    Workload("tie_e96_k40_general_multi", 65, (120, 64), 64, 64, 96, 40, 4, 0, "relu"),
]


def _tie_cases():
    return [pytest.param(wl, path, id=f"{wl.name}-p{path}") for wl in TIES
            for path in _paths(wl)]


@pytest.mark.parametrize("wl,path", _tie_cases())
def test_tied_logits_select_like_the_oracle(dev, wl, path):
    inp = make_inputs(wl)
    inp["router_probs"] = tied_logits(wl.tokens, wl.experts, seed=wl.index)
    y_ref, sel_ref, p_ref = oracle.qmoe(inp["input"], inp["router_probs"],
                                        inp["fc1_experts_weights"], inp["fc1_scales"],
                                        inp["fc2_experts_weights"], inp["fc2_scales"],
                                        nthreads=os.cpu_count() or 1, **wl.attrs())
    srt = -np.sort(-inp["router_probs"], axis=1)
    assert np.mean(srt[:, wl.k - 1] == srt[:, wl.k]) > 0.3   # ties at the top-k boundary
    y, sel, p = run_cuda(inp, wl.attrs(), path, dev)
    check_routing(sel, p, sel_ref, p_ref, f"{wl.name} path {path} (tied logits)")
    check_outputs(y, y_ref, f"{wl.name} path {path} (tied logits)")


# Scales small enough that fp16 copies of scale-multiplied weights (or of the
# scales) fall below the fp16 normal range (6.1e-5): 8-bit block-wise scales in
# U[1e-5, 1e-4], 4-bit in U[1e-4, 1e-3], on every path that takes each shape.
SMALL_SCALES = [
    Workload("small_s_8bit_bs32", 66, (300, 256), 256, 256, 8, 2, 8, 32, "swiglu",
             scale_lo=1e-5, scale_hi=1e-4),
    Workload("small_s_8bit_bs128_decode", 67, (8, 512), 512, 512, 8, 2, 8, 128, "swiglu",
             scale_lo=1e-5, scale_hi=1e-4),
    Workload("small_s_4bit_bs64", 68, (300, 256), 256, 256, 8, 2, 4, 64, "swiglu",
             scale_lo=1e-4, scale_hi=1e-3),
    Workload("small_s_4bit_bs16_decode", 69, (8, 512), 512, 512, 8, 2, 4, 16, "swiglu",
             scale_lo=1e-4, scale_hi=1e-3),
    Workload("small_s_4bit_bs32_decode", 70, (12, 1024), 1024, 512, 4, 2, 4, 32, "relu",
             scale_lo=1e-4, scale_hi=1e-3),
    Workload("small_s_4bit_col", 71, (300, 256), 256, 256, 8, 2, 4, 0, "swiglu",
             scale_lo=1e-4, scale_hi=1e-3),
]


def _small_scale_cases():
    return [pytest.param(wl, path, id=f"{wl.name}-p{path}") for wl in SMALL_SCALES
            for path in _paths(wl)]


@pytest.mark.parametrize("wl,path", _small_scale_cases())
def test_small_scales_parity(dev, wl, path):
    inp = make_inputs(wl)
    y_ref, sel_ref, p_ref = _reference(wl, inp)
    y, sel, p = run_cuda(inp, wl.attrs(), path, dev)
    check_routing(sel, p, sel_ref, p_ref, wl.name)
    check_outputs(y, y_ref, f"{wl.name} path {path}")


def test_repeat_is_bit_identical(dev):
    wl = SMALL[1]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    a = run_cuda(inp, wl.attrs(), 0, dev, t=t)
    b = run_cuda(inp, wl.attrs(), 0, dev, t=t)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_zero_scales_exact_zero(dev):
    wl = SMALL[1]
    inp = make_inputs(wl)
    inp["fc1_scales"] = np.zeros_like(inp["fc1_scales"])
    for path in _paths(wl):
        y, _, _ = run_cuda(inp, dict(wl.attrs(), activation_beta=0.5), path, dev)
        assert np.all(y == 0.0), path


def test_zero_tokens_is_noop(dev):
    import quantized_mixture_experts_gb300 as q
    wl = WORKLOADS["tiny"].with_tokens(0)
    inp = make_inputs(WORKLOADS["tiny"])
    inp["input"] = np.zeros((0, 64), np.float32)
    inp["router_probs"] = np.zeros((0, 4), np.float32)
    t = to_dev(inp, dev)
    y = q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                       t["fc2_experts_weights"], t["fc2_scales"], **wl.attrs())
    torch.cuda.synchronize()
    assert y.shape == (0, 64)


def test_inter_zero_writes_zeros(dev):
    import quantized_mixture_experts_gb300 as q
    T, H, E = 12, 64, 4
    x = torch.randn(T, H, device=dev)
    lg = torch.randn(T, E, device=dev)
    w1 = torch.zeros((E, 0, H // 2), dtype=torch.uint8, device=dev)
    s1 = torch.zeros((E, 0), device=dev)
    w2 = torch.zeros((E, H, 0), dtype=torch.uint8, device=dev)
    s2 = torch.zeros((E, H), device=dev)
    y = torch.full((T, H), 3.0, device=dev)
    sel = torch.full((T, 2), -1, dtype=torch.int32, device=dev)
    q.qmoe_forward(x, lg, w1, s1, w2, s2, output=y, topk_idx=sel, k=2)
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    ref_sel, _ = oracle.route(lg.cpu().numpy(), 2)
    assert np.array_equal(sel.cpu().numpy(), ref_sel)


def test_hostio_matches_device_path(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[6]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(**wl.attrs())
    y_dev = q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                           t["fc1_scales"], t["fc2_experts_weights"], t["fc2_scales"],
                           attrs=attrs)
    hx = torch.from_numpy(inp["input"]).pin_memory()
    hl = torch.from_numpy(inp["router_probs"]).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape,
                                            attrs, hostio=True))
    q.qmoe_forward_hostio(hx, hl, t["fc1_experts_weights"], t["fc1_scales"],
                          t["fc2_experts_weights"], t["fc2_scales"], hy, attrs=attrs,
                          workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(hy.numpy(), y_dev.cpu().numpy())


@pytest.mark.parametrize("wl", [SMALL[6], SMALL[1],
                                Workload("hostio_over_limit", 29, (600, 512), 512, 256, 8, 2, 4,
                                         32, "swiglu")],
                         ids=lambda w: w.name)
def test_hostio_in_place_and_copied_agree(dev, wl):
    """Host-IO with mapped page-locked buffers (read and written in place by the kernels
    when the activations fit QMOE_HOSTIO_DIRECT_BYTES, copied otherwise) and with pageable
    buffers (always copied) give the device path's output bit for bit."""
    import quantized_mixture_experts_gb300 as q
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(**wl.attrs())
    y_dev = q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                           t["fc1_scales"], t["fc2_experts_weights"], t["fc2_scales"],
                           attrs=attrs).cpu().numpy()
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape,
                                            attrs, hostio=True))
    for pinned in (True, False):
        hx = torch.from_numpy(inp["input"].copy())
        hl = torch.from_numpy(inp["router_probs"].copy())
        hy = torch.full_like(hx, float("nan"))
        if pinned:
            hx, hl, hy = hx.pin_memory(), hl.pin_memory(), hy.pin_memory()
        for _ in range(2):
            q.qmoe_forward_hostio(hx, hl, t["fc1_experts_weights"], t["fc1_scales"],
                                  t["fc2_experts_weights"], t["fc2_scales"], hy, attrs=attrs,
                                  workspace=ws)
            torch.cuda.synchronize()
            assert np.array_equal(hy.numpy(), y_dev), (wl.name, pinned)
    assert (wl.name == "hostio_over_limit") == (inp["input"].nbytes > q.binding.HOSTIO_DIRECT_BYTES)


def test_device_error_clean_after_forward(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[1]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(**wl.attrs())
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape, attrs))
    ws.fill_(0xAB)   # stale garbage: the call must clear its error word
    q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                   t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs, workspace=ws)
    assert q.get_device_error(ws) == q.DEVERR_NONE


@pytest.mark.parametrize("path,which", [(2, "fc1"), (2, "fc2"), (1, "fc1")])
def test_fp16_overflow_sets_nonfinite(dev, path, which):
    """Scales so large that the FC1 activations (or the weighted FC2 rows of the
    grouped path) leave the fp16 range: the call records QMOE_DEVERR_NONFINITE;
    the same layer with its normal scales records nothing."""
    import quantized_mixture_experts_gb300 as q
    tokens = 8 if path == 1 else 40   # the decode path takes at most 16 tokens
    wl = Workload("overflow", 41, (tokens, 256), 256, 128, 4, 2, 4, 32, "swiglu")
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(path=path, **wl.attrs())
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape, attrs))
    q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                   t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs, workspace=ws)
    assert q.get_device_error(ws) == q.DEVERR_NONE
    s1 = t["fc1_scales"] * (1e4 if which == "fc1" else 1.0)
    s2 = t["fc2_scales"] * (1e7 if which == "fc2" else 1.0)
    q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], s1,
                   t["fc2_experts_weights"], s2, attrs=attrs, workspace=ws)
    assert q.get_device_error(ws) == q.DEVERR_NONFINITE


# ----------------------------------------------------------------------------
# Full-size workloads
# ----------------------------------------------------------------------------

FULL = ["tiny", "decode", "prefill", "many_small", "large_e"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(dev, name):
    import quantized_mixture_experts_gb300 as q
    wl = WORKLOADS[name]
    path = q.choose_path(wl.input_shape, (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack),
                         q.make_attrs(**wl.attrs()))
    if wl.tokens > 64 and path == q.PATH_GENERIC:
        pytest.skip("full-size run needs a tensor-core path for this shape")
    inp = make_inputs(wl)
    y, sel, p = run_cuda(inp, wl.attrs(), q.PATH_AUTO, dev)
    sel_all, p_all = oracle.route(inp["router_probs"], wl.k)
    check_routing(sel, p, sel_all, p_all, name + " (all tokens)")
    tokens = None if wl.tokens <= 64 else sample_tokens(sel_all, wl.tokens, 256,
                                                        seed=1234 + wl.index)
    y_ref, sel_ref, p_ref = _reference(wl, inp, tokens)
    if tokens is not None:
        y, sel, p = y[tokens], sel[tokens], p[tokens]
    check_routing(sel, p, sel_ref, p_ref, name)
    check_outputs(y, y_ref, name)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "many_small", "large_e"])
def test_full_size_parity_every_token(dev, name):
    """The three large workloads at full size, in the bench's launch
    configuration, compared with the oracle on every token (the oracle's batched
    evaluation: per-expert fp64 matrix products, pinned to the token-by-token
    restatement on the CPU)."""
    import quantized_mixture_experts_gb300 as q
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    y, sel, p = run_cuda(inp, wl.attrs(), q.PATH_AUTO, dev)
    y_ref, sel_ref, p_ref = oracle.qmoe_batched(
        inp["input"], inp["router_probs"], inp["fc1_experts_weights"], inp["fc1_scales"],
        inp["fc2_experts_weights"], inp["fc2_scales"], **wl.attrs())
    check_routing(sel, p, sel_ref, p_ref, name + " (every token)")
    check_outputs(y, y_ref, name + " (every token)")
    # and token by token: no token's error hides in the whole-batch norms
    err = np.linalg.norm(y - y_ref, axis=1) / np.maximum(np.linalg.norm(y_ref, axis=1), 1e-300)
    assert err.max() <= 4 * 5e-3, f"{name}: worst token rel-L2 {err.max():.3e}"


@pytest.mark.parametrize("name,path", [("decode", 1), ("prefill_like_rank3", 2)])
def test_wait_timeout_reports_error_and_recovers(dev, name, path):
    """One pipeline stage is never filled (test hook), so a consumer waits on a
    barrier nothing completes: with a 50 ms wait limit the kernels must record
    QMOE_DEVERR_TIMEOUT, drain, free their resources and return, and the next
    call with the normal limit must be correct."""
    import quantized_mixture_experts_gb300 as q
    from quantized_mixture_experts_gb300 import binding as b
    wl = WORKLOADS[name] if name in WORKLOADS else [w for w in SMALL if w.name == name][0]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(path=path, **wl.attrs())
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape, attrs))
    q.set_wait_limit_ns(50_000_000)
    b.debug_drop_stage(1)
    try:
        q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                       t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs, workspace=ws)
        code = q.get_device_error(ws)
    finally:
        b.debug_drop_stage(-1)
        q.set_wait_limit_ns(2_000_000_000)
    assert code == q.DEVERR_TIMEOUT
    y, sel, p = run_cuda(inp, wl.attrs(), path, dev, t=t, workspace=ws)
    tokens = np.arange(min(wl.tokens, 64), dtype=np.int64)
    y_ref, sel_ref, p_ref = _reference(wl, inp, tokens)
    check_routing(sel[tokens], p[tokens], sel_ref, p_ref, name)
    check_outputs(y[tokens], y_ref, name + " after timeout")
    assert q.get_device_error(ws) == q.DEVERR_NONE


def test_hooks_apply_to_the_setting_thread_only(dev):
    """A short wait limit and the dropped-stage hook set by one host thread do not
    reach a layer that another thread runs: that layer completes without a device
    error and within the parity bar."""
    import threading

    import quantized_mixture_experts_gb300 as q
    from quantized_mixture_experts_gb300 import binding as b
    wl = [w for w in SMALL if w.name == "prefill_like_rank3"][0]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(path=q.PATH_GROUPED, **wl.attrs())
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, t["fc1_experts_weights"].shape, attrs))
    out = {}

    def other_thread():
        try:
            out["run"] = run_cuda(inp, wl.attrs(), q.PATH_GROUPED, dev, t=t, workspace=ws)
            out["err"] = q.get_device_error(ws)
        except Exception as e:   # reported in the main thread
            out["exc"] = e

    q.set_wait_limit_ns(50_000_000)
    b.debug_drop_stage(1)
    try:
        th = threading.Thread(target=other_thread)
        th.start()
        th.join()
    finally:
        b.debug_drop_stage(-1)
        q.set_wait_limit_ns(2_000_000_000)
    assert "exc" not in out, out.get("exc")
    assert out["err"] == q.DEVERR_NONE
    y, sel, p = out["run"]
    tokens = np.arange(64, dtype=np.int64)
    y_ref, sel_ref, p_ref = _reference(wl, inp, tokens)
    check_routing(sel[tokens], p[tokens], sel_ref, p_ref, wl.name)
    check_outputs(y[tokens], y_ref, wl.name + " in another thread")


@pytest.mark.parametrize("name,calls", [("many_small", 600), ("large_e", 60)])
def test_repeated_calls_bit_identical(dev, name, calls):
    """Hundreds of calls on the same inputs give the same output bit for bit: a race
    between the CTA pair's operand writes and the other CTA's tensor core showed up as
    an occasional call (about one in a few hundred) with whole token tiles wrong."""
    import quantized_mixture_experts_gb300 as q
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(**wl.attrs())
    args = (t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
            t["fc2_experts_weights"], t["fc2_scales"])
    ref = q.qmoe_forward(*args, attrs=attrs).clone()
    out = torch.empty_like(ref)
    bad = 0
    for _ in range(calls):
        q.qmoe_forward(*args, attrs=attrs, output=out)
        bad += int(not torch.equal(out, ref))
    torch.cuda.synchronize()
    assert bad == 0, f"{bad} of {calls} calls differ"
