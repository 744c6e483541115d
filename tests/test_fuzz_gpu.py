"""Seeded randomized-shape parity sweep of the three operators against the
fp64 oracle, through the C ABI, on every path AUTO picks and on the forced
alternatives.  Shapes, attributes and routing are drawn from a fixed seed so a
failure names a reproducible case.
"""
import os

import numpy as np
import pytest

import oracle
from helpers import check_outputs, check_routing, run_cuda
from quantized_mixture_experts_gb300.workloads import (FloatWorkload, QkvWorkload, Workload,
                                                       make_float_inputs, make_inputs,
                                                       make_qkv_inputs)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _qmoe_cases(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([2, 4, 8, 16, 64]))
        k = int(rng.integers(1, min(E, 8) + 1))
        H = int(rng.choice([64, 128, 192, 256, 512, 1024]))
        I = int(rng.choice([64, 128, 256, 384]))
        T = int(rng.choice([1, 3, 8, 16, 17, 40, 130, 300]))
        bits = int(rng.choice([4, 8]))
        bs = int(rng.choice([0, 16, 32, 64]))
        if bs and (H % bs or I % bs):
            bs = 0
        act = str(rng.choice(["relu", "swiglu"]))
        out.append(Workload(f"fq{i}", 200 + i, (T, H), H, I, E, k, bits, bs, act,
                            alpha=float(rng.choice([1.0, 1.7])),
                            beta=float(rng.choice([0.0, 0.5])),
                            swiglu_limit=None if rng.random() < 0.7 else 1.5,
                            logit_sigma=float(rng.choice([1.0, 2.0]))))
    return out


@pytest.mark.parametrize("wl", _qmoe_cases(), ids=lambda w: w.name)
def test_qmoe_fuzz(dev, wl):
    import quantized_mixture_experts_gb300 as q
    inp = make_inputs(wl)
    y_ref, sel_ref, p_ref = oracle.qmoe(inp["input"], inp["router_probs"],
                                        inp["fc1_experts_weights"], inp["fc1_scales"],
                                        inp["fc2_experts_weights"], inp["fc2_scales"],
                                        nthreads=os.cpu_count() or 1, **wl.attrs())
    for path in (q.PATH_AUTO, q.PATH_DECODE, q.PATH_GROUPED, q.PATH_GENERIC):
        a = q.make_attrs(path=path, **wl.attrs())
        try:
            q.choose_path(wl.input_shape, (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack), a)
        except q.QmoeError:
            continue
        y, sel, p = run_cuda(inp, wl.attrs(), path, dev)
        check_routing(sel, p, sel_ref, p_ref, f"{wl.name} path {path}")
        check_outputs(y, y_ref, f"{wl.name} path {path} {wl}")


def _float_cases(n=12, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([2, 4, 8, 32]))
        k = int(rng.integers(1, min(E, 4) + 1))
        H = int(rng.choice([32, 64, 96, 160, 256, 40]))
        I = int(rng.choice([32, 64, 96, 128, 24]))
        T = int(rng.choice([1, 5, 16, 33, 150, 400]))
        act = str(rng.choice(["relu", "gelu", "silu", "swiglu", "identity"]))
        fusion = int(rng.choice([0, 1, 2])) if act == "swiglu" else 0
        fc3 = (act == "swiglu" and fusion == 0) or (act == "silu" and rng.random() < 0.5)
        out.append(FloatWorkload(f"ff{i}", 300 + i, (T, H), H, I, E, k, act, swiglu_fusion=fusion,
                                 fc3=fc3, biases=bool(rng.random() < 0.6),
                                 normalize=int(rng.integers(0, 2)),
                                 alpha=float(rng.choice([1.0, 1.702])),
                                 beta=float(rng.choice([0.0, 1.0]))))
    return out


@pytest.mark.parametrize("wl", _float_cases(), ids=lambda w: w.name)
def test_float_moe_fuzz(dev, wl):
    import quantized_mixture_experts_gb300 as q
    inp = make_float_inputs(wl)
    opt = ("fc1_experts_bias", "fc2_experts_bias", "fc3_experts_weights", "fc3_experts_bias")
    y_ref, sel_ref, w_ref = oracle.moe(inp["input"], inp["router_probs"],
                                       inp["fc1_experts_weights"], inp["fc2_experts_weights"],
                                       fc1_bias=inp.get("fc1_experts_bias"),
                                       fc2_bias=inp.get("fc2_experts_bias"),
                                       fc3_w=inp.get("fc3_experts_weights"),
                                       fc3_bias=inp.get("fc3_experts_bias"),
                                       nthreads=os.cpu_count() or 1, **wl.attrs())
    t = {kk: torch.from_numpy(v).to(dev) for kk, v in inp.items()}
    for path in (q.MOE_PATH_AUTO, q.MOE_PATH_GROUPED, q.MOE_PATH_GENERIC):
        a = q.make_moe_attrs(path=path, **wl.attrs())
        try:
            q.moe_choose_path(wl.input_shape, (wl.experts, wl.fc1_rows, wl.hidden), a)
        except q.QmoeError:
            continue
        sel = torch.empty((wl.tokens, wl.k), dtype=torch.int32, device=dev)
        pw = torch.empty((wl.tokens, wl.k), dtype=torch.float32, device=dev)
        y = q.moe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                          t["fc2_experts_weights"], attrs=a, topk_idx=sel, topk_w=pw,
                          **{kk: t.get(kk) for kk in opt})
        torch.cuda.synchronize()
        check_routing(sel.cpu().numpy(), pw.cpu().numpy().astype(np.float64), sel_ref, w_ref,
                      f"{wl.name} path {path}")
        check_outputs(y.cpu().numpy().astype(np.float64), y_ref, f"{wl.name} path {path} {wl}")


def _qkv_cases(n=12, seed=5):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([128, 256, 384, 512, 1024, 2048, 96, 160]))
        Nq = int(rng.choice([64, 128, 200, 512]))
        Nkv = int(rng.choice([32, 64, 128, 72]))
        rows = int(rng.choice([1, 2, 7, 8, 9, 16, 20]))
        skip = bool(rng.random() < 0.5)
        out.append(QkvWorkload(f"fk{i}", 400 + i, (rows, K), K, Nq, Nkv,
                               str(rng.choice(["float32", "float16"])), skip,
                               skip and bool(rng.random() < 0.5)))
    return out


@pytest.mark.parametrize("wl", _qkv_cases(), ids=lambda w: w.name)
def test_qkv_fuzz(dev, wl):
    import quantized_mixture_experts_gb300 as q
    inp = make_qkv_inputs(wl)
    f = lambda kk: None if kk not in inp else inp[kk].astype(np.float64)
    ref = oracle.qkv(f("A"), f("norm_scale"), inp["q_B"], f("q_scales"), inp["k_B"], f("k_scales"),
                     inp["v_B"], f("v_scales"), skip=f("skip"), residual=wl.residual)
    t = {kk: torch.from_numpy(v).to(dev) for kk, v in inp.items()}
    dt = t["A"].dtype
    for path in (q.QKV_PATH_AUTO, q.QKV_PATH_DECODE, q.QKV_PATH_GENERIC):
        a = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv, path=path)
        try:
            q.qkv_choose_path(wl.input_shape, a, dt)
        except q.QmoeError:
            continue
        got = q.matmul_nbits_qkv(t["A"], t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                                 t["k_scales"], t["v_B"], t["v_scales"], skip=t.get("skip"),
                                 residual=wl.residual, attrs=a)
        torch.cuda.synchronize()
        got = [g.float().cpu().numpy().astype(np.float64) for g in got]
        for name, g_, r_ in zip("QKV", got[:3], ref[:3]):
            check_outputs(g_, r_, f"{wl.name} path {path} {name} {wl}")
        if wl.residual:
            tol = 1e-3 if wl.dtype == "float16" else 1e-6
            np.testing.assert_allclose(got[3], ref[3], rtol=tol, atol=tol)
