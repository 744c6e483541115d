"""qmoe_forward_noalloc, the entry point for callers that cannot allocate
device memory (for example a plugin whose host runtime owns the device memory
pool and offers no allocator, or a latency-critical loop that cannot take the
implicit device synchronization of cudaMalloc).  It runs the layer in the
library's fixed scratch array instead of a caller workspace.

Through the C ABI, on every kernel path that takes each shape, two calls in a
row (the second finds the first one's leftovers in the shared array):
  * the output and the routing are bit-identical to qmoe_forward with a caller
    workspace on the same path (the same kernels run on the same inputs);
  * the output meets the parity bar against the fp64 oracle, and the routing
    equals the oracle's.
Also: the device error word of these calls, read through
qmoe_noalloc_get_device_error, reports an fp16 overflow and is clean after a
normal call; shapes that need more scratch than the array holds are refused
before anything runs.  This file is collected last so that a run stopping at
the first failure has already run every other test.
"""
import os

import numpy as np
import pytest

from helpers import check_outputs, check_routing, to_dev
from quantized_mixture_experts_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


CASES = [WORKLOADS["decode"], WORKLOADS["tiny"],
         Workload("noalloc_8bit", 40, (12, 512), 512, 256, 6, 2, 8, 0, "relu")]


def _params():
    """(workload, path) for every path that takes the shape within the array."""
    import quantized_mixture_experts_gb300 as q
    out = []
    for wl in CASES:
        fc1 = (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack)
        for path in (q.PATH_AUTO, q.PATH_DECODE, q.PATH_GROUPED, q.PATH_GENERIC):
            attrs = q.make_attrs(path=path, **wl.attrs())
            try:
                need = q.workspace_size(wl.input_shape, fc1, attrs)
            except q.QmoeError:
                continue
            if need <= q.load().qmoe_noalloc_scratch_bytes():
                out.append(pytest.param(wl, path, id=f"{wl.name}-p{path}"))
    return out


def _run_both(wl, path, dev, salt):
    import quantized_mixture_experts_gb300 as q
    inp = make_inputs(wl, salt=salt)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(path=path, **wl.attrs())
    T, k, H = wl.tokens, wl.k, wl.hidden
    sel_ws = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    pw_ws = torch.zeros((T, k), dtype=torch.float32, device=dev)
    y_ws = q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                          t["fc1_scales"], t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs,
                          topk_idx=sel_ws, topk_w=pw_ws)
    y_na = torch.full_like(t["input"], float("nan"))
    sel = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    pw = torch.zeros((T, k), dtype=torch.float32, device=dev)
    q.binding.qmoe_forward_noalloc(t["input"], t["router_probs"], t["fc1_experts_weights"],
                                   t["fc1_scales"], t["fc2_experts_weights"], t["fc2_scales"],
                                   attrs=attrs, output=y_na, topk_idx=sel, topk_w=pw)
    torch.cuda.synchronize()
    return (inp, y_na.reshape(-1, H).cpu().numpy(), y_ws.reshape(-1, H).cpu().numpy(),
            sel.cpu().numpy(), pw.cpu().numpy(), sel_ws.cpu().numpy(), pw_ws.cpu().numpy())


@pytest.mark.parametrize("wl,path", _params())
def test_noalloc_matches_workspace_entry_twice(dev, wl, path):
    import oracle
    import quantized_mixture_experts_gb300 as q
    for call in range(2):   # the second call reuses scratch left by the first
        inp, y_na, y_ws, sel, pw, sel_ws, pw_ws = _run_both(wl, path, dev, salt=call)
        what = f"{wl.name} path {path} call {call}"
        assert np.array_equal(y_na, y_ws), f"{what}: output differs from the workspace entry"
        assert np.array_equal(sel, sel_ws) and np.array_equal(pw, pw_ws), \
            f"{what}: routing differs from the workspace entry"
        y_ref, sel_ref, p_ref = oracle.qmoe(
            inp["input"], inp["router_probs"], inp["fc1_experts_weights"], inp["fc1_scales"],
            inp["fc2_experts_weights"], inp["fc2_scales"], nthreads=os.cpu_count() or 1,
            **wl.attrs())
        check_routing(sel, pw.astype(np.float64), sel_ref, p_ref, what)
        check_outputs(y_na.astype(np.float64), y_ref.reshape(-1, wl.hidden), what)
        assert q.binding.noalloc_get_device_error() == q.DEVERR_NONE, what


def test_noalloc_device_error_reports_overflow(dev):
    """FC1 scales so large that the fp16 activations overflow: the call's error
    word, read through qmoe_noalloc_get_device_error, says QMOE_DEVERR_NONFINITE;
    reading clears it, and the next normal call leaves it clean."""
    import quantized_mixture_experts_gb300 as q
    wl = Workload("noalloc_overflow", 41, (40, 256), 256, 128, 4, 2, 4, 32, "swiglu")
    inp = make_inputs(wl)
    t = to_dev(inp, dev)
    attrs = q.make_attrs(path=q.PATH_GROUPED, **wl.attrs())
    y = torch.empty_like(t["input"])
    args = (t["input"], t["router_probs"], t["fc1_experts_weights"])
    q.binding.qmoe_forward_noalloc(*args, t["fc1_scales"] * 1e4, t["fc2_experts_weights"],
                                   t["fc2_scales"], attrs=attrs, output=y)
    assert q.binding.noalloc_get_device_error() == q.DEVERR_NONFINITE
    assert q.binding.noalloc_get_device_error() == q.DEVERR_NONE
    q.binding.qmoe_forward_noalloc(*args, t["fc1_scales"], t["fc2_experts_weights"],
                                   t["fc2_scales"], attrs=attrs, output=y)
    assert q.binding.noalloc_get_device_error() == q.DEVERR_NONE


def test_noalloc_rejects_too_large(dev):
    import ctypes

    import quantized_mixture_experts_gb300 as q
    from quantized_mixture_experts_gb300 import binding as b
    wl = WORKLOADS["prefill"]
    attrs = q.make_attrs(**wl.attrs())
    fc1 = (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack)
    assert q.workspace_size(wl.input_shape, fc1, attrs) > q.load().qmoe_noalloc_scratch_bytes()
    # NULL data pointers: the size check refuses the call on the host, and a check
    # that ever moved behind a launch would fail on the NULL pointers, not on the GPU
    r = (wl.tokens, wl.experts)
    s1 = (wl.experts, fc1[1], wl.hidden // wl.block_size)
    fc2 = (wl.experts, wl.hidden, wl.inter // wl.pack)
    s2 = (wl.experts, wl.hidden, wl.inter // wl.block_size)
    st = q.load().qmoe_forward_noalloc(
        None, b._shape(wl.input_shape), len(wl.input_shape), None, b._shape(r), None,
        b._shape(fc1), None, b._shape(s1), 3, None, b._shape(fc2), None, b._shape(s2), 3, None,
        ctypes.byref(attrs), None, None, None)
    assert st == b.ERR_WORKSPACE_TOO_SMALL
