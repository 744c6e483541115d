"""GPU parity of grouped_matmul (ONNX GroupedMatMul-29) through the C ABI.

The page's worked examples run for every element type and index type; random
cases are compared with the oracle under the bound of the accumulation type:
|out - ref| <= c * eps_acc * K * sum_k |x_k||w_k| (+ output rounding for 16-bit
outputs), with eps_acc = 2^-24 (fp32 accumulate) or 2^-53 (fp64).
"""
import json
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "grouped_matmul_examples.json")
DTYPES = {"f32": "float32", "f16": "float16", "bf16": "bfloat16", "f64": "float64"}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("idt", ["int32", "int64"])
@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_page_examples(dev, ex, dt, idt):
    import quantized_mixture_experts_gb300 as q
    tdt = getattr(torch, DTYPES[dt])
    if "expected" not in ex:
        x = torch.zeros(ex["input_shape"], dtype=tdt, device=dev)
        w = torch.zeros(ex["weights_shape"], dtype=tdt, device=dev)
        idx = torch.zeros(ex["group_indices_shape"], dtype=getattr(torch, idt), device=dev)
        out = q.grouped_matmul(x, w, idx)
        torch.cuda.synchronize()
        assert list(out.shape) == ex["expected_shape"]
        return
    x = torch.tensor(ex["input"], dtype=tdt, device=dev)
    w = torch.tensor(ex["weights"], dtype=tdt, device=dev)
    idx = torch.tensor(ex["group_indices"], dtype=getattr(torch, idt), device=dev)
    bias = None if ex["bias"] is None else torch.tensor(ex["bias"], dtype=tdt, device=dev)
    ws = q.alloc_workspace(256)
    out = q.grouped_matmul(x, w, idx, bias, workspace=ws)
    torch.cuda.synchronize()
    exp = torch.tensor(ex["expected"], dtype=tdt).double().numpy()   # expected, rounded to T
    np.testing.assert_array_equal(out.double().cpu().numpy(), exp)
    assert q.get_device_error(ws) == q.DEVERR_NONE


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("shape", [(37, 70, 5, 33, 3), (128, 256, 8, 96, 2), (1, 1, 1, 1, 1),
                                   (65, 0, 3, 9, 2)])
def test_random_vs_oracle(dev, dt, shape):
    import quantized_mixture_experts_gb300 as q
    M, K, G, N, S = shape
    rng = np.random.default_rng(sum(shape))
    tdt = getattr(torch, DTYPES[dt])
    x = torch.from_numpy(rng.standard_normal((M, K))).to(tdt)
    w = torch.from_numpy(rng.standard_normal((G, K, N))).to(tdt)
    b = torch.from_numpy(rng.standard_normal((G, N))).to(tdt)
    idx = torch.from_numpy(rng.integers(0, G, (M, S)))
    out = q.grouped_matmul(x.to(dev), w.to(dev), idx.to(dev), b.to(dev))
    torch.cuda.synchronize()
    xr, wr, br = x.double().numpy(), w.double().numpy(), b.double().numpy()
    ref, st = oracle.grouped_matmul(xr, wr, idx.numpy(), br)
    assert st == oracle.OK
    mag = np.einsum("mk,mskn->msn", np.abs(xr), np.abs(wr)[idx.numpy()]) + np.abs(br)[idx.numpy()]
    eps_acc = 2.0 ** -53 if dt == "f64" else 2.0 ** -24
    eps_out = {"f32": 2.0 ** -24, "f64": 2.0 ** -53, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}[dt]
    bound = 2 * (K + 2) * eps_acc * mag + eps_out * np.abs(ref) + 1e-300
    err = np.abs(out.double().cpu().numpy() - ref)
    assert np.all(err <= bound), float(np.max(err / bound))


def test_out_of_range_index_sets_error_and_zero_row(dev):
    import quantized_mixture_experts_gb300 as q
    x = torch.ones((3, 4), device=dev)
    w = torch.ones((2, 4, 5), device=dev)
    idx = torch.tensor([[0], [2], [-1]], dtype=torch.int64, device=dev)
    ws = q.alloc_workspace(256)
    out = q.grouped_matmul(x, w, idx, workspace=ws)
    assert q.get_device_error(ws) == q.DEVERR_INDEX
    o = out.cpu().numpy()
    assert np.all(o[0] == 4.0) and np.all(o[1] == 0.0) and np.all(o[2] == 0.0)
    assert q.get_device_error(ws) == q.DEVERR_NONE   # read clears the word


def _oracle_check(out, x, w, idx, b, dt, K):
    xr, wr = x.double().cpu().numpy(), w.double().cpu().numpy()
    br = None if b is None else b.double().cpu().numpy()
    ix = idx.cpu().numpy()
    ref, st = oracle.grouped_matmul(xr, wr, ix, br)
    assert st == oracle.OK
    mag = np.einsum("mk,mskn->msn", np.abs(xr), np.abs(wr)[ix])
    if br is not None:
        mag = mag + np.abs(br)[ix]
    eps_out = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}[dt]
    bound = 2 * (K + 2) * 2.0 ** -24 * mag + eps_out * np.abs(ref) + 1e-300
    err = np.abs(out.double().cpu().numpy() - ref)
    assert np.all(err <= bound), float(np.max(err / bound))


def _launches():
    import quantized_mixture_experts_gb300 as q
    return q.load().qmoe_launch_count()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape,idt", [((600, 512, 7, 384, 2), "int32"),
                                       ((300, 128, 40, 200, 3), "int64"),
                                       ((17, 64, 3, 8, 1), "int32")],
                         ids=["tiles_bias", "ragged_n_i64", "tiny"])
def test_tensor_core_path_vs_oracle(dev, dt, shape, idt):
    """f16/bf16 with K % 64 == 0 and N % 8 == 0 take the tensor-core path (more
    than one launch: grouping, gather, GEMM) when the workspace allows it."""
    import quantized_mixture_experts_gb300 as q
    M, K, G, N, S = shape
    rng = np.random.default_rng(sum(shape) + len(dt))
    tdt = getattr(torch, DTYPES[dt])
    x = torch.from_numpy(rng.standard_normal((M, K))).to(tdt).to(dev)
    w = torch.from_numpy(rng.standard_normal((G, K, N)) / np.sqrt(K)).to(tdt).to(dev)
    b = torch.from_numpy(rng.standard_normal((G, N))).to(tdt).to(dev)
    idx = torch.from_numpy(rng.integers(0, G, (M, S))).to(getattr(torch, idt)).to(dev)
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(M, K, G, N, S, tdt))
    n0 = _launches()
    out = q.grouped_matmul(x, w, idx, b, workspace=ws)
    torch.cuda.synchronize()
    n_tc = _launches() - n0
    assert q.get_device_error(ws) == q.DEVERR_NONE
    _oracle_check(out, x, w, idx, b, dt, K)
    # the same call with the minimal workspace runs the general kernel (one launch
    # after clearing the error word): same bound
    ws_small = q.alloc_workspace(256)
    n0 = _launches()
    out2 = q.grouped_matmul(x, w, idx, b, workspace=ws_small)
    torch.cuda.synchronize()
    n_general = _launches() - n0
    assert n_general == 2 and n_tc > n_general, (n_tc, n_general)
    _oracle_check(out2, x, w, idx, b, dt, K)


def _oracle_check_f32(out, x, w, idx, b, K):
    xr, wr = x.double().cpu().numpy(), w.double().cpu().numpy()
    br = None if b is None else b.double().cpu().numpy()
    ix = idx.cpu().numpy()
    ref, st = oracle.grouped_matmul(xr, wr, ix, br)
    assert st == oracle.OK
    mag = np.einsum("mk,mskn->msn", np.abs(xr), np.abs(wr)[ix])
    if br is not None:
        mag = mag + np.abs(br)[ix]
    bound = 2 * (K + 2) * 2.0 ** -24 * mag + 2.0 ** -24 * np.abs(ref) + 1e-300
    err = np.abs(out.double().cpu().numpy() - ref)
    assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.parametrize("shape,idt", [((600, 512, 7, 384, 2), "int32"),
                                       ((300, 128, 40, 200, 3), "int64"),
                                       ((17, 64, 3, 8, 1), "int32"),
                                       ((257, 96, 2, 100, 2), "int64")],
                         ids=["tiles_bias", "ragged_n_i64", "tiny", "partial_tile"])
def test_f32_tensor_core_path_vs_oracle(dev, shape, idt):
    """f32 with K % 32 == 0 and N % 4 == 0 takes the tensor-core path (three TF32
    products per step) and is held to the same fp32 bound as the general kernel."""
    import quantized_mixture_experts_gb300 as q
    M, K, G, N, S = shape
    rng = np.random.default_rng(sum(shape) + 32)
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(dev)
    w = torch.from_numpy(rng.standard_normal((G, K, N)).astype(np.float32)).to(dev)
    b = torch.from_numpy(rng.standard_normal((G, N)).astype(np.float32)).to(dev)
    idx = torch.from_numpy(rng.integers(0, G, (M, S))).to(getattr(torch, idt)).to(dev)
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(M, K, G, N, S, torch.float32))
    n0 = _launches()
    out = q.grouped_matmul(x, w, idx, b, workspace=ws)
    torch.cuda.synchronize()
    assert _launches() - n0 > 2   # grouping, gather, GEMM
    assert q.get_device_error(ws) == q.DEVERR_NONE
    _oracle_check_f32(out, x, w, idx, b, K)
    # without bias, and against the general kernel's result under the same bound
    out_nb = q.grouped_matmul(x, w, idx, workspace=ws)
    torch.cuda.synchronize()
    _oracle_check_f32(out_nb, x, w, idx, None, K)


def test_f32_tensor_core_path_invalid_index(dev):
    import quantized_mixture_experts_gb300 as q
    M, K, G, N, S = 40, 64, 3, 64, 2
    x = torch.ones((M, K), dtype=torch.float32, device=dev)
    w = torch.ones((G, K, N), dtype=torch.float32, device=dev) / 64
    idx = torch.zeros((M, S), dtype=torch.int64, device=dev)
    idx[3, 1] = G
    idx[7, 0] = -5
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(M, K, G, N, S, torch.float32))
    out = torch.full((M, S, N), float("nan"), dtype=torch.float32, device=dev)
    n0 = _launches()
    q.grouped_matmul(x, w, idx, output=out, workspace=ws)
    torch.cuda.synchronize()
    assert _launches() - n0 > 2
    assert q.get_device_error(ws) == q.DEVERR_INDEX
    o = out.cpu().numpy()
    assert np.all(o[3, 1] == 0.0) and np.all(o[7, 0] == 0.0)
    mask = np.ones((M, S), dtype=bool)
    mask[3, 1] = mask[7, 0] = False
    assert np.all(o[mask] == 1.0)


def test_tensor_core_path_invalid_index(dev):
    import quantized_mixture_experts_gb300 as q
    M, K, G, N, S = 40, 64, 3, 64, 2
    x = torch.ones((M, K), dtype=torch.float16, device=dev)
    w = torch.ones((G, K, N), dtype=torch.float16, device=dev) / 64
    idx = torch.zeros((M, S), dtype=torch.int64, device=dev)
    idx[3, 1] = G
    idx[7, 0] = -5
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(M, K, G, N, S, torch.float16))
    out = torch.full((M, S, N), float("nan"), dtype=torch.float16, device=dev)
    n0 = _launches()
    q.grouped_matmul(x, w, idx, output=out, workspace=ws)
    torch.cuda.synchronize()
    assert _launches() - n0 > 2   # the tensor-core path
    assert q.get_device_error(ws) == q.DEVERR_INDEX
    o = out.float().cpu().numpy()
    assert np.all(o[3, 1] == 0.0) and np.all(o[7, 0] == 0.0)
    mask = np.ones((M, S), dtype=bool)
    mask[3, 1] = mask[7, 0] = False
    assert np.all(o[mask] == 1.0)


@pytest.mark.parametrize("name", ["gmm_prefill", "gmm_prefill_bf16", "gmm_prefill_f32",
                                  "gmm_prefill_f64"])
def test_bench_workload_sampled_vs_oracle(dev, name):
    """The benchmark's GroupedMatMul workloads (the prefill layer's FC1 shape as a dense
    grouped product in f16, bf16, f32 and f64: M 4096, K 4096, G 8, N 28672, S 2) at full size through
    the call the benchmark times.  Sampled rows and columns (the last of each
    included) are compared with the oracle on the sampled problem: input[rows] and
    weights[:, :, cols] give exactly those outputs under the Summary definition."""
    import quantized_mixture_experts_gb300 as q
    from quantized_mixture_experts_gb300.workloads import GMM_WORKLOADS, make_gmm_inputs
    wl = GMM_WORKLOADS[name]
    dt = {"float16": "f16", "bfloat16": "bf16", "float32": "f32", "float64": "f64"}[wl.dtype]
    tdt = getattr(torch, DTYPES[dt])
    inp = make_gmm_inputs(wl)
    x = torch.from_numpy(inp["input"]).to(dev).to(tdt)
    w = torch.from_numpy(inp["weights"]).to(dev).to(tdt)
    del inp["weights"]
    idx = torch.from_numpy(inp["group_indices"]).to(dev)
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(wl.M, wl.K, wl.G, wl.N,
                                                                   wl.S, tdt), dev)
    n0 = _launches()
    out = q.grouped_matmul(x, w, idx, workspace=ws)
    torch.cuda.synchronize()
    # error-word clear, grouping (3), gather, tensor-core GEMM; f64: clear, general kernel
    assert _launches() - n0 == (2 if dt == "f64" else 6)
    assert q.get_device_error(ws) == q.DEVERR_NONE
    rng = np.random.default_rng(11)
    r = np.unique(np.append(rng.choice(wl.M, 48, replace=False), wl.M - 1))
    c = np.unique(np.append(rng.choice(wl.N, 384, replace=False), wl.N - 1))
    rt, ct = torch.from_numpy(r).to(dev), torch.from_numpy(c).to(dev)
    xr = x[rt].double().cpu().numpy()
    wr = w[:, :, ct].double().cpu().numpy()
    ix = inp["group_indices"][r]
    got = out[rt][:, :, ct].double().cpu().numpy()
    ref, st = oracle.grouped_matmul(xr, wr, ix)
    assert st == oracle.OK
    mag = np.stack([np.stack([np.abs(xr[m]) @ np.abs(wr[g]) for g in ix[m]]) for m in range(len(r))])
    eps_out = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 2.0 ** -24, "f64": 2.0 ** -53}[dt]
    eps_acc = 2.0 ** -53 if dt == "f64" else 2.0 ** -24
    bound = 2 * (wl.K + 2) * eps_acc * mag + eps_out * np.abs(ref) + 1e-300
    err = np.abs(got - ref)
    assert np.all(err <= bound), float(np.max(err / bound))
