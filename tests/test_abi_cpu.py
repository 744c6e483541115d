"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function include/qmoe.h declares;
attribute defaults must equal the QMoE manifest's `attributes`; shape and
attribute validation (manifest derive.quantContract and
attributeConstraints) must reject bad calls before anything is launched, so
these calls never touch a device.
"""
import ctypes
import os

import pytest

import __graft_entry__
import quantized_mixture_experts_gb300 as q
from quantized_mixture_experts_gb300 import binding as b


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return q.load()


def test_exports_every_declared_symbol(lib):
    names = q.declared_functions()
    assert "qmoe_forward" in names and "grouped_matmul" in names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_attr_defaults_match_manifest(lib):
    a = b.Attrs()
    lib.qmoe_attrs_default(ctypes.byref(a))
    assert a.k == 1 and a.expert_weight_bits == 4 and a.activation_type == 0
    assert a.block_size == 0 and a.swiglu_fusion == 0
    assert a.activation_alpha == 1.0 and a.activation_beta == 0.0
    assert a.has_swiglu_limit == 0 and a.normalize_routing_weights == 0
    assert a.use_sparse_mixer == 0 and a.weights_prepacked == -1 and a.quant_type_is_int == 1
    assert ctypes.sizeof(b.Attrs) == 64


def _call(attrs, T=8, H=64, I=32, E=4, bits=4, bs=0, fusion=None, scales_rank=None,
          router=None, fc2=None, s1=None, s2=None, input_shape=None, ws_bytes=1 << 30):
    fusion = fusion if fusion is not None else (2 if attrs.activation_type == 1 else 1)
    pack = 2 if bits == 4 else 1
    input_shape = input_shape or (T, H)
    router = router or (T, E)
    fc1 = (E, fusion * I, H // pack)
    fc2 = fc2 or (E, H, I // pack)
    r = scales_rank or (3 if bs else 2)
    s1 = s1 or ((E, fusion * I, H // bs) if bs else (E, fusion * I))
    s2 = s2 or ((E, H, I // bs) if bs else (E, H))
    fake = 0x1000  # never dereferenced: validation fails before any launch
    return q.load().qmoe_forward(
        fake, b._shape(input_shape), len(input_shape), fake, b._shape(router),
        fake, b._shape(fc1), fake, b._shape(s1), r, fake, b._shape(fc2), fake, b._shape(s2), r,
        fake, ctypes.byref(attrs), 0x10000, ws_bytes, None, None, None)


def A(**kw):
    return q.make_attrs(**kw)


@pytest.mark.parametrize("kw,call,status", [
    (dict(k=5), {}, b.ERR_INVALID_ARGUMENT),                       # k > E
    (dict(k=0), {}, b.ERR_INVALID_ARGUMENT),                       # k < 1
    (dict(k=2, block_size=24), {}, b.ERR_INVALID_ARGUMENT),        # not a power of two
    (dict(k=2, block_size=8), {}, b.ERR_INVALID_ARGUMENT),         # below 16
    (dict(k=2, block_size=64), dict(I=32), b.ERR_INVALID_ARGUMENT),  # does not divide inter
    (dict(k=2, activation_type="swiglu", swiglu_fusion=0), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, activation_type="relu", swiglu_fusion=1), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, activation_type="swiglu", swiglu_fusion=2), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, activation_type="gelu"), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, expert_weight_bits=2), dict(bits=4), b.ERR_NOT_SUPPORTED),
    (dict(k=2, use_sparse_mixer=1), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, weights_prepacked=1), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, weights_prepacked=3), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2, quant_type="fp4"), {}, b.ERR_NOT_SUPPORTED),
    (dict(k=2, normalize_routing_weights=2), {}, b.ERR_INVALID_ARGUMENT),
    (dict(k=2), dict(router=(7, 4)), b.ERR_INVALID_ARGUMENT),      # router rows != tokens
    (dict(k=2), dict(fc2=(4, 64, 8)), b.ERR_INVALID_ARGUMENT),     # fc2 packed cols
    (dict(k=2), dict(scales_rank=3, s1=(4, 32, 2), s2=(4, 64, 1)), b.ERR_INVALID_ARGUMENT),
    (dict(k=2, block_size=16), dict(bs=16, scales_rank=2, s1=(4, 32), s2=(4, 64)),
     b.ERR_INVALID_ARGUMENT),
    (dict(k=2, block_size=16), dict(bs=16, s1=(4, 32, 3)), b.ERR_INVALID_ARGUMENT),
    (dict(k=2), dict(input_shape=(2, 4, 64, 1)), b.ERR_INVALID_ARGUMENT),  # rank 4
    (dict(k=2), dict(ws_bytes=16), b.ERR_WORKSPACE_TOO_SMALL),
])
def test_contract_rejections(lib, kw, call, status):
    assert _call(A(**kw), **call) == status


def test_workspace_size_and_path(lib):
    a = A(k=2, expert_weight_bits=4, block_size=32, activation_type="swiglu")
    n = q.workspace_size((8, 4096), (8, 2 * 14336, 2048), a)
    assert n > 0 and n % 256 == 0
    nh = q.workspace_size((8, 4096), (8, 2 * 14336, 2048), a, hostio=True)
    assert nh >= n + 8 * 4096 * 4 * 2
    p = q.choose_path((8, 4096), (8, 2 * 14336, 2048), a)
    assert p in (q.PATH_DECODE, q.PATH_GROUPED, q.PATH_GENERIC)
    a.path = q.PATH_GENERIC
    assert q.choose_path((8, 4096), (8, 2 * 14336, 2048), a) == q.PATH_GENERIC


def test_gmm_rejections(lib):
    ws = 0x10000
    f = q.load().grouped_matmul
    assert f(0x1000, -1, 2, 0x1000, 1, 1, 0x1000, 1, 0, None, 0x1000, 0, ws, 256, None) == \
        b.ERR_INVALID_ARGUMENT
    assert f(0x1000, 1, 2, 0x1000, 1, 1, 0x1000, 1, 7, None, 0x1000, 0, ws, 256, None) == \
        b.ERR_INVALID_ARGUMENT
    assert f(0x1000, 1, 2, 0x1000, 1, 1, 0x1000, 1, 0, None, 0x1000, 9, ws, 256, None) == \
        b.ERR_INVALID_ARGUMENT
    assert f(0x1000, 1, 2, 0x1000, 1, 1, 0x1000, 1, 0, None, 0x1000, 0, ws, 8, None) == \
        b.ERR_WORKSPACE_TOO_SMALL


def test_status_strings(lib):
    assert q.binding.status_string(0) == "ok"
    assert "workspace" in q.binding.status_string(3)


@pytest.mark.parametrize("name,expected", [("tiny", "grouped"), ("decode", "decode"),
                                           ("prefill", "grouped"), ("many_small", "grouped"),
                                           ("large_e", "grouped")])
def test_auto_path_of_each_config(lib, name, expected):
    """AUTO: the decode GEMV up to 16 tokens when its shape rules hold (H and I
    multiples of 128, at least four scale blocks per 512-code chunk); the grouped
    tensor-core path when H and I are multiples of 64; the scalar path otherwise."""
    from quantized_mixture_experts_gb300.workloads import WORKLOADS
    wl = WORKLOADS[name]
    a = q.make_attrs(**wl.attrs())
    p = q.choose_path(wl.input_shape, (wl.experts, wl.fusion * wl.inter, wl.hidden // wl.pack), a)
    assert q.PATH_NAMES[p] == expected


@pytest.mark.parametrize("T,H,I,bs,expected", [
    (16, 256, 256, 32, "decode"),     # the decode rules hold at 16 tokens
    (17, 256, 256, 32, "grouped"),    # one token more
    (8, 192, 256, 32, "grouped"),     # H not a multiple of 128
    (8, 256, 256, 256, "grouped"),    # fewer than four scale blocks per 512 codes
    (8, 96, 64, 32, "generic"),       # H not a multiple of 64
    (300, 64, 96, 32, "generic"),     # I not a multiple of 64
])
def test_auto_path_boundaries(lib, T, H, I, bs, expected):
    a = A(k=2, expert_weight_bits=4, block_size=bs, activation_type="swiglu")
    assert q.PATH_NAMES[q.choose_path((T, H), (8, 2 * I, H // 2), a)] == expected


def test_profile_kernel_ids(lib):
    """Every kernel id of the header, GroupedMatMul's GEMM included, is accepted;
    ids outside the enum are rejected.  No launch is recorded, so no CUDA call."""
    for kid in (q.KERNEL_ROUTE, q.KERNEL_GROUP, q.KERNEL_FC1, q.KERNEL_FC2, q.KERNEL_COMBINE,
                q.KERNEL_GMM):
        assert lib.qmoe_profile_begin(kid) == 0
        n, ms = q.profile_end()
        assert (n, ms) == (0, 0.0)
    assert q.KERNEL_GMM == 5
    assert lib.qmoe_profile_begin(6) == 1
    assert lib.qmoe_profile_begin(-1) == 1


def _header_enums():
    """name -> value for every enumerator written `NAME = value` in include/*.h."""
    import re
    vals = {}
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    for h in ("qmoe.h", "moe.h", "qkv.h"):
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
        for body in re.findall(r"typedef enum\s*\{(.*?)\}", text, flags=re.S):
            for name, val in re.findall(r"([A-Z][A-Z0-9_]+)\s*=\s*(-?\d+)", body):
                vals[name] = int(val)
    return vals


def test_binding_constants_match_header_enums():
    """The binding's constants carry the values the C headers give their enumerators."""
    h = _header_enums()
    b = q.binding
    pairs = {
        "QMOE_OK": b.OK, "QMOE_ERR_INVALID_ARGUMENT": b.ERR_INVALID_ARGUMENT,
        "QMOE_ERR_NOT_SUPPORTED": b.ERR_NOT_SUPPORTED,
        "QMOE_ERR_WORKSPACE_TOO_SMALL": b.ERR_WORKSPACE_TOO_SMALL, "QMOE_ERR_CUDA": b.ERR_CUDA,
        "QMOE_DEVERR_NONE": b.DEVERR_NONE, "QMOE_DEVERR_INDEX": b.DEVERR_INDEX,
        "QMOE_DEVERR_NONFINITE": b.DEVERR_NONFINITE, "QMOE_DEVERR_TIMEOUT": b.DEVERR_TIMEOUT,
        "QMOE_ACT_RELU": b.ACTIVATIONS["relu"], "QMOE_ACT_SWIGLU": b.ACTIVATIONS["swiglu"],
        "QMOE_PATH_AUTO": b.PATH_AUTO, "QMOE_PATH_DECODE": b.PATH_DECODE,
        "QMOE_PATH_GROUPED": b.PATH_GROUPED, "QMOE_PATH_GENERIC": b.PATH_GENERIC,
        "QMOE_DT_F32": b.DT_F32, "QMOE_DT_F16": b.DT_F16, "QMOE_DT_BF16": b.DT_BF16,
        "QMOE_DT_F64": b.DT_F64, "QMOE_IDX_I32": b.IDX_I32, "QMOE_IDX_I64": b.IDX_I64,
        "QMOE_KERNEL_ROUTE": b.KERNEL_ROUTE, "QMOE_KERNEL_GROUP": b.KERNEL_GROUP,
        "QMOE_KERNEL_FC1": b.KERNEL_FC1, "QMOE_KERNEL_FC2": b.KERNEL_FC2,
        "QMOE_KERNEL_COMBINE": b.KERNEL_COMBINE, "QMOE_KERNEL_GMM": b.KERNEL_GMM,
        "MOE_PATH_AUTO": b.MOE_PATH_AUTO, "MOE_PATH_GROUPED": b.MOE_PATH_GROUPED,
        "MOE_PATH_GENERIC": b.MOE_PATH_GENERIC,
        "QKV_PATH_AUTO": b.QKV_PATH_AUTO, "QKV_PATH_DECODE": b.QKV_PATH_DECODE,
        "QKV_PATH_GENERIC": b.QKV_PATH_GENERIC,
    }
    pairs.update({f"MOE_ACT_{a.upper()}": v for a, v in b.MOE_ACTIVATIONS.items()})
    missing = sorted(set(pairs) - set(h))
    assert not missing, missing
    assert {k: h[k] for k in pairs} == pairs


def _header_prototypes():
    """name -> parameter count for every function prototype in include/*.h."""
    import re
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    protos = {}
    for h in ("qmoe.h", "moe.h", "qkv.h"):
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
        text = re.sub(r"typedef\s+(enum|struct)\s*\{.*?\}\s*\w+\s*;", "", text, flags=re.S)
        for name, params in re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(([^()]*)\)\s*;", text):
            params = params.strip()
            protos[name] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_argument_counts_match_prototypes(lib):
    """Every declared function is bound with as many ctypes arguments as its C
    prototype has parameters (a mismatch would pass garbage through the ABI)."""
    protos = _header_prototypes()
    assert set(protos) == set(q.declared_functions())
    for name, n in sorted(protos.items()):
        at = getattr(lib, name).argtypes
        assert at is not None and len(at) == n, (name, n, at)


@pytest.mark.parametrize("cname,pyname", [("qmoe_attrs", "Attrs"), ("moe_attrs", "MoeAttrs"),
                                          ("qkv_attrs", "QkvAttrs")])
def test_attribute_struct_layouts_match_c(tmp_path, cname, pyname):
    """The ctypes structures have the C compiler's size and field offsets for the
    attribute structs of include/*.h (compiled here with the system C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    st = getattr(b, pyname)
    fields = [f[0] for f in st._fields_]
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "qmoe.h"', '#include "moe.h"',
             '#include "qkv.h"', 'int main(void) {',
             f'  printf("%zu\\n", sizeof({cname}));']
    lines += [f'  printf("%zu\\n", offsetof({cname}, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(st)
    assert got[1:] == [getattr(st, f).offset for f in fields]


def test_hostio_direct_limit_matches_header():
    """The binding's host-IO in-place limit is the header's QMOE_HOSTIO_DIRECT_BYTES."""
    import re
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    text = open(os.path.join(inc, "qmoe.h")).read()
    m = re.search(r"#define\s+QMOE_HOSTIO_DIRECT_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "QMOE_HOSTIO_DIRECT_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == q.binding.HOSTIO_DIRECT_BYTES
