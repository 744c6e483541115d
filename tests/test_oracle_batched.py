"""The oracle's batched evaluation (qmoe_batched: per-expert fp64 matrix
products, used to check every token of the large workloads) against the
token-by-token C restatement (qmoe), on layers that cover both bit widths,
column- and block-wise scales, ReLU, SwiGLU with alpha/beta/limit, k = 1 and
k = E, rank-3 input and an expert that no token selects.  The two differ only
in fp64 rounding order, so they must agree to 1e-12 of the output scale.
"""
import numpy as np
import pytest

import oracle
from quantized_mixture_experts_gb300.workloads import WORKLOADS, Workload, make_inputs

CASES = [
    WORKLOADS["tiny"],
    Workload("b_swiglu_bs32", 80, (50, 128), 128, 96, 8, 2, 4, 32, "swiglu"),
    Workload("b_8bit_col_relu", 81, (40, 64), 64, 64, 16, 4, 8, 0, "relu"),
    Workload("b_k1_rank3", 82, (2, 20, 64), 64, 64, 6, 1, 4, 16, "swiglu"),
    Workload("b_k_eq_E", 83, (12, 64), 64, 32, 4, 4, 8, 32, "swiglu"),
    Workload("b_limit", 84, (30, 64), 64, 64, 8, 2, 4, 0, "swiglu", alpha=1.7, beta=0.3,
             swiglu_limit=0.4),
    Workload("b_unused_expert", 85, (3, 64), 64, 64, 32, 2, 4, 0, "relu"),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_batched_equals_token_by_token(wl):
    inp = make_inputs(wl)
    args = (inp["input"], inp["router_probs"], inp["fc1_experts_weights"], inp["fc1_scales"],
            inp["fc2_experts_weights"], inp["fc2_scales"])
    y, sel, p = oracle.qmoe(*args, nthreads=4, **wl.attrs())
    yb, selb, pb = oracle.qmoe_batched(*args, **wl.attrs())
    assert np.array_equal(sel, selb) and np.array_equal(p, pb)
    scale = np.abs(y).max()
    assert scale > 0
    assert np.abs(yb - y).max() <= 1e-12 * scale
    if wl.name == "b_unused_expert":
        assert len(np.unique(sel)) < wl.experts


def test_batched_zero_inter_is_zero():
    wl = Workload("b_zero", 86, (5, 64), 64, 0, 4, 2, 4, 0, "relu")
    inp = make_inputs(wl)
    y, _, _ = oracle.qmoe_batched(inp["input"], inp["router_probs"], inp["fc1_experts_weights"],
                                  inp["fc1_scales"], inp["fc2_experts_weights"],
                                  inp["fc2_scales"], **wl.attrs())
    assert np.all(y == 0.0)
