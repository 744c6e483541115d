"""Host-side checks of the float MoE C ABI (include/moe.h) that need no GPU.

Attribute defaults must equal the com.microsoft.MoE README's Attributes
table, and validation (README Inputs and Attributes) must reject bad calls
before anything is launched, so these calls never touch a device.
"""
import ctypes

import pytest

import __graft_entry__
import quantized_mixture_experts_gb300 as q
from quantized_mixture_experts_gb300 import binding as b


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return q.load()


def test_moe_exports(lib):
    for n in ("moe_attrs_default", "moe_workspace_size", "moe_choose_path", "moe_forward",
              "moe_hostio_workspace_size", "moe_forward_hostio", "moe_get_device_error"):
        assert n in q.declared_functions()
        assert hasattr(lib, n)


def test_moe_attr_defaults_match_readme(lib):
    a = b.MoeAttrs()
    lib.moe_attrs_default(ctypes.byref(a))
    assert a.k == 1 and a.activation_type == b.MOE_ACTIVATIONS["relu"]
    assert a.swiglu_fusion == 0 and a.activation_alpha == 1.0 and a.activation_beta == 0.0
    assert a.has_swiglu_limit == 0 and a.normalize_routing_weights == 0
    assert a.use_sparse_mixer == 0 and a.path == b.MOE_PATH_AUTO
    assert ctypes.sizeof(b.MoeAttrs) == 48


def _call(attrs, T=8, H=64, I=32, E=4, rows1=None, router=None, fc2=None, fc3=None,
          input_shape=None, ws_bytes=1 << 30, with_fc3=False):
    fused = attrs.activation_type == b.MOE_ACTIVATIONS["swiglu"] and attrs.swiglu_fusion != 0
    rows1 = rows1 if rows1 is not None else (2 * I if fused else I)
    input_shape = input_shape or (T, H)
    router = router or (T, E)
    fc1 = (E, rows1, H)
    fc2 = fc2 or (E, H, I)
    fake = 0x1000  # never dereferenced: validation fails before any launch
    f3 = fake if (with_fc3 or fc3) else None
    s3 = b._shape(fc3 or (E, I, H)) if (with_fc3 or fc3) else None
    return q.load().moe_forward(
        fake, b._shape(input_shape), len(input_shape), fake, b._shape(router),
        fake, b._shape(fc1), None, fake, b._shape(fc2), None, f3, s3, None,
        fake, ctypes.byref(attrs), 0x10000, ws_bytes, None, None, None)


def A(**kw):
    return q.make_moe_attrs(**kw)


@pytest.mark.parametrize("kw,call,status", [
    (dict(k=5), {}, b.ERR_INVALID_ARGUMENT),                                # k > E
    (dict(k=0), {}, b.ERR_INVALID_ARGUMENT),                                # k < 1
    (dict(k=2, activation_type="tanh"), {}, b.ERR_INVALID_ARGUMENT),        # unknown activation
    (dict(k=2, activation_type="relu", swiglu_fusion=1), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, activation_type="swiglu", swiglu_fusion=3), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, activation_type="swiglu", swiglu_fusion=0), {}, b.ERR_INVALID_ARGUMENT),  # no FC3
    (dict(k=2, activation_type="swiglu", swiglu_fusion=2), dict(rows1=33),
     b.ERR_INVALID_ARGUMENT),                                               # odd fused rows
    (dict(k=2, use_sparse_mixer=1), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, use_sparse_mixer=2), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, normalize_routing_weights=2), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2), dict(router=(7, 4)), b.ERR_INVALID_ARGUMENT),               # router rows
    (dict(k=2), dict(fc2=(4, 64, 16)), b.ERR_INVALID_ARGUMENT),             # fc2 inner dim
    (dict(k=2, activation_type="silu"), dict(fc3=(4, 32, 48)), b.ERR_INVALID_ARGUMENT),
    (dict(k=2), dict(input_shape=(2, 4, 64, 1)), b.ERR_INVALID_ARGUMENT),   # rank 4
    (dict(k=2), dict(ws_bytes=16), b.ERR_WORKSPACE_TOO_SMALL),
    (dict(k=2, path=b.MOE_PATH_GROUPED), dict(H=48), b.ERR_NOT_SUPPORTED),  # H % 32
    (dict(k=2, path=1), {}, b.ERR_INVALID_ARGUMENT),                        # no decode path
])
def test_moe_contract_rejections(lib, kw, call, status):
    assert _call(A(**kw), **call) == status


def test_moe_swiglu_fusion0_with_fc3_validates(lib):
    # passes validation, then fails the workspace check (still no launch)
    st = _call(A(k=2, activation_type="swiglu", swiglu_fusion=0), with_fc3=True, ws_bytes=16)
    assert st == b.ERR_WORKSPACE_TOO_SMALL


def test_moe_workspace_and_path(lib):
    a = A(k=2, activation_type="swiglu", swiglu_fusion=0)
    n = q.moe_workspace_size((4096, 4096), (8, 14336, 4096), a)
    assert n > 0 and n % 256 == 0
    # the grouped layouts: sorted TF32 rows and FC1 output, FC2 rows by slot
    assert n >= 4 * 8192 * (4096 + 14336 + 4096)
    assert q.moe_choose_path((4096, 4096), (8, 14336, 4096), a) == b.MOE_PATH_GROUPED
    assert q.moe_choose_path((16, 48), (4, 32, 48), A(k=2)) == b.MOE_PATH_GENERIC
    a.path = b.MOE_PATH_GENERIC
    assert q.moe_choose_path((4096, 4096), (8, 14336, 4096), a) == b.MOE_PATH_GENERIC
    nh = q.moe_workspace_size((8, 4096), (8, 14336, 4096), a, hostio=True)
    assert nh >= q.moe_workspace_size((8, 4096), (8, 14336, 4096), a) + 2 * 8 * 4096 * 4
