"""GPU parity of the RMSNorm + 4-bit Q/K/V projection (com.microsoft.
MatMulNBitsQkv manifest) against the fp64 oracle, through the C ABI.

Small cases cover both T1 types, skip and residual, 1 to 16 rows on the GEMV
path, ragged output rows, K values the GEMV path does not take (scalar path),
many rows and rank-3 inputs; the decode workloads are compared in full.
"""
import numpy as np
import pytest

import oracle
from helpers import check_outputs
from quantized_mixture_experts_gb300.workloads import (QKV_WORKLOADS, QkvWorkload,
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


def _reference(inp, wl: QkvWorkload):
    f = lambda k: None if k not in inp else inp[k].astype(np.float64)
    return oracle.qkv(f("A"), f("norm_scale"), inp["q_B"], f("q_scales"), inp["k_B"],
                      f("k_scales"), inp["v_B"], f("v_scales"), skip=f("skip"),
                      residual=wl.residual)


def _run(inp, wl: QkvWorkload, path, dev):
    import quantized_mixture_experts_gb300 as q
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in inp.items()}
    attrs = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv, path=path)
    out = q.matmul_nbits_qkv(t["A"], t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                             t["k_scales"], t["v_B"], t["v_scales"], skip=t.get("skip"),
                             residual=wl.residual, attrs=attrs)
    torch.cuda.synchronize()
    return [o.reshape(-1, o.shape[-1]).float().cpu().numpy().astype(np.float64) for o in out]


SMALL = [
    QKV_WORKLOADS["qkv_tiny"],
    QkvWorkload("f16_skip", 80, (5, 512), 512, 256, 128, "float16", True, False),
    QkvWorkload("one_row", 81, (1, 1024), 1024, 384, 128, "float32"),
    QkvWorkload("sixteen_rows_f16", 82, (16, 768), 768, 256, 256, "float16", True, True),
    QkvWorkload("nine_rows_ragged_n", 83, (9, 384), 384, 200, 72, "float32"),
    QkvWorkload("rank3", 84, (2, 3, 512), 512, 128, 64, "float32", True, True),
    QkvWorkload("k_not_mult_128", 85, (6, 200), 200, 96, 40, "float32", True, True),
    QkvWorkload("k_not_mult_32", 86, (3, 100), 100, 64, 32, "float16"),
    QkvWorkload("many_rows", 87, (40, 256), 256, 128, 64, "float32", True, True),
    QkvWorkload("f16_k384_scalar", 88, (4, 384), 384, 128, 128, "float16"),
    # few output rows and a long K: eight CTAs share each row block; the one holding
    # its first chunks adds the others' partial sums
    QkvWorkload("split_k_f16", 90, (4, 4096), 4096, 128, 64, "float16", True, True),
    QkvWorkload("split_k_f32", 91, (11, 2048), 2048, 200, 72, "float32"),
]


def _paths(wl):
    import quantized_mixture_experts_gb300 as q
    out = []
    for path in (q.QKV_PATH_AUTO, q.QKV_PATH_DECODE, q.QKV_PATH_GENERIC):
        a = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv, path=path)
        try:
            q.qkv_choose_path(wl.input_shape, a, torch.float16 if wl.dtype == "float16"
                              else torch.float32)
        except q.QmoeError as e:
            assert e.status == q.binding.ERR_NOT_SUPPORTED
            continue
        out.append(path)
    return out


def _cases():
    return [pytest.param(wl, p, id=f"{wl.name}-p{p}") for wl in SMALL for p in _paths(wl)]


def _check(got, ref, wl, what):
    for name, g, r in zip(("Q", "K", "V"), got[:3], ref[:3]):
        check_outputs(g, r, f"{what} {name}")
    if wl.residual:
        tol = 1e-3 if wl.dtype == "float16" else 1e-6
        np.testing.assert_allclose(got[3], ref[3].reshape(got[3].shape), rtol=tol, atol=tol)


@pytest.mark.parametrize("wl,path", _cases())
def test_small_parity(dev, wl, path):
    inp = make_qkv_inputs(wl)
    ref = _reference(inp, wl)
    got = _run(inp, wl, path, dev)
    _check(got, ref, wl, f"{wl.name} path {path}")


def test_decode_path_taken_for_few_rows(dev):
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[3]
    a = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv)
    assert q.qkv_choose_path(wl.input_shape, a, torch.float16) == q.QKV_PATH_DECODE
    inp = make_qkv_inputs(wl)
    n0 = q.launch_count()
    _run(inp, wl, q.QKV_PATH_AUTO, dev)
    assert q.launch_count() - n0 == 2          # normalisation; projection with partial sums


def _call(q, t, wl, outputs, ws):
    attrs = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv)
    res = torch.empty_like(t["A"]) if wl.residual else None
    q.matmul_nbits_qkv(t["A"], t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                       t["k_scales"], t["v_B"], t["v_scales"], skip=t.get("skip"),
                       residual=res, attrs=attrs, outputs=outputs, workspace=ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["split_k_f16", "split_k_f32", "qkv_decode"])
def test_repeat_into_poisoned_outputs(dev, name):
    # The same outputs and workspace (with the shared row blocks' completion flags left
    # by the call before) are reused after every output element is set to NaN: each
    # call must write every element again, with the same bits.
    import quantized_mixture_experts_gb300 as q
    wl = {w.name: w for w in SMALL}.get(name) or QKV_WORKLOADS[name]
    inp = make_qkv_inputs(wl)
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in inp.items()}
    dt = t["A"].dtype
    attrs = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv)
    assert q.qkv_choose_path(wl.input_shape, attrs, dt) == q.QKV_PATH_DECODE
    ws = q.alloc_workspace(q.qkv_workspace_size(wl.input_shape, attrs, dt), dev)
    lead = tuple(wl.input_shape[:-1])
    outs = tuple(torch.empty(lead + (n,), dtype=dt, device=dev) for n in (wl.Nq, wl.Nkv, wl.Nkv))
    _call(q, t, wl, outs, ws)
    first = [o.clone() for o in outs]
    assert all(bool(torch.isfinite(o).all()) for o in first)
    for _ in range(5):
        for o in outs:
            o.fill_(float("nan"))
        _call(q, t, wl, outs, ws)
        assert all(torch.equal(o, f) for o, f in zip(outs, first))


def test_in_place_residual(dev):
    # residual written over A: each row is read whole before its residual is written
    import quantized_mixture_experts_gb300 as q
    wl = SMALL[3]                                   # sixteen rows, fp16, skip
    inp = make_qkv_inputs(wl)
    ref = _reference(inp, wl)
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in inp.items()}
    A = t["A"].clone()
    out = q.matmul_nbits_qkv(A, t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                             t["k_scales"], t["v_B"], t["v_scales"], skip=t["skip"], residual=A)
    torch.cuda.synchronize()
    got = [o.reshape(-1, o.shape[-1]).float().cpu().numpy().astype(np.float64) for o in out]
    _check(got, ref, wl, "in-place residual")


def test_repeat_is_bit_identical(dev):
    wl = SMALL[1]
    inp = make_qkv_inputs(wl)
    a = _run(inp, wl, 0, dev)
    b = _run(inp, wl, 0, dev)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_zero_rows(dev):
    import quantized_mixture_experts_gb300 as q
    wl = QkvWorkload("zero_rows", 89, (0, 256), 256, 64, 32, "float32")
    inp = make_qkv_inputs(QkvWorkload("zr", 89, (1, 256), 256, 64, 32, "float32"))
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    A = torch.zeros((0, 256), device=dev)
    out = q.matmul_nbits_qkv(A, t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                             t["k_scales"], t["v_B"], t["v_scales"])
    assert out[0].shape == (0, 64) and out[1].shape == (0, 32)


@pytest.mark.parametrize("name", ["qkv_decode", "qkv_decode_f32"])
def test_full_size(dev, name):
    wl = QKV_WORKLOADS[name]
    inp = make_qkv_inputs(wl)
    ref = _reference(inp, wl)
    got = _run(inp, wl, 0, dev)
    _check(got, ref, wl, name)
