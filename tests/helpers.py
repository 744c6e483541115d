"""Shared helpers of the GPU parity tests: run the CUDA layer through the C
ABI and compare with the oracle under the acceptance bar.

Bar (per output tensor, against the fp64 oracle):
  selected experts     identical lists (logits are drawn without ties)
  routing weights      |p - p_ref| <= 1e-6 * p_ref
  outputs              ||y - y_ref||_2 <= 5e-3 * ||y_ref||_2 and
                       max |y - y_ref| <= 2e-2 * rms(y_ref)
"""
from __future__ import annotations

import numpy as np

REL_L2 = 5e-3
MAX_RMS = 2e-2
ROUTE_REL = 1e-6


def to_dev(inp: dict, dev):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in inp.items()}


def run_cuda(inp: dict, wl_attrs: dict, path: int, dev, t=None, workspace=None, stream=None):
    """Run qmoe_forward; returns (y [T,H] np.float64, sel [T,k] np.int32, p [T,k] np.float64)."""
    import torch
    import quantized_mixture_experts_gb300 as q
    t = t if t is not None else to_dev(inp, dev)
    attrs = q.make_attrs(path=path, **wl_attrs)
    T = t["router_probs"].shape[0]
    k = wl_attrs["k"]
    sel = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    pw = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
    y = q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                       t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs, topk_idx=sel,
                       topk_w=pw, workspace=workspace, stream=stream)
    torch.cuda.synchronize()
    H = t["input"].shape[-1]
    return (y.reshape(-1, H).cpu().numpy().astype(np.float64), sel.cpu().numpy(),
            pw.cpu().numpy().astype(np.float64))


def check_outputs(y: np.ndarray, y_ref: np.ndarray, what: str = ""):
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    diff = y - y_ref
    nref = np.linalg.norm(y_ref)
    rel = np.linalg.norm(diff) / max(nref, 1e-300)
    rms = np.sqrt(np.mean(y_ref ** 2))
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_RMS * rms, f"{what}: max err {mx:.3e} > {MAX_RMS} * rms {rms:.3e}"
    return rel, mx / max(rms, 1e-300)


def check_routing(sel, p, sel_ref, p_ref, what: str = ""):
    assert np.array_equal(sel, sel_ref), f"{what}: selected experts differ"
    assert np.all(np.abs(p - p_ref) <= ROUTE_REL * np.abs(p_ref)), \
        f"{what}: routing weights off by {np.max(np.abs(p - p_ref) / p_ref):.3e}"
