"""ctypes binding of the C ABI in include/qmoe.h, include/moe.h and include/qkv.h.

Argument marshalling only: every step of the layer runs in the CUDA library
``libqmoe_gb300.so``.  Tensors are torch CUDA tensors (torch supplies device
memory and streams); this module never computes anything itself and has no
CPU path.  If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmoe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "qmoe.h")
MOE_HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe.h")
QKV_HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "qkv.h")

# qmoe_status
OK, ERR_INVALID_ARGUMENT, ERR_NOT_SUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA = range(5)
# qmoe_device_error
DEVERR_NONE, DEVERR_INDEX, DEVERR_NONFINITE, DEVERR_TIMEOUT = range(4)
# qmoe_path
PATH_AUTO, PATH_DECODE, PATH_GROUPED, PATH_GENERIC = range(4)
PATH_NAMES = {PATH_AUTO: "auto", PATH_DECODE: "decode", PATH_GROUPED: "grouped",
              PATH_GENERIC: "generic"}
# qmoe_dtype / qmoe_index_dtype
DT_F32, DT_F16, DT_BF16, DT_F64 = range(4)
IDX_I32, IDX_I64 = range(2)
# qmoe_kernel_id
KERNEL_ROUTE, KERNEL_GROUP, KERNEL_FC1, KERNEL_FC2, KERNEL_COMBINE, KERNEL_GMM = range(6)


class QmoeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Attrs(ctypes.Structure):
    """Mirror of qmoe_attrs (same field order and C types)."""
    _fields_ = [
        ("k", ctypes.c_int64),
        ("expert_weight_bits", ctypes.c_int32),
        ("activation_type", ctypes.c_int32),
        ("block_size", ctypes.c_int64),
        ("swiglu_fusion", ctypes.c_int32),
        ("activation_alpha", ctypes.c_float),
        ("activation_beta", ctypes.c_float),
        ("has_swiglu_limit", ctypes.c_int32),
        ("swiglu_limit", ctypes.c_float),
        ("normalize_routing_weights", ctypes.c_int32),
        ("use_sparse_mixer", ctypes.c_int32),
        ("weights_prepacked", ctypes.c_int32),
        ("quant_type_is_int", ctypes.c_int32),
        ("path", ctypes.c_int32),
    ]


class MoeAttrs(ctypes.Structure):
    """Mirror of moe_attrs (same field order and C types)."""
    _fields_ = [
        ("k", ctypes.c_int64),
        ("activation_type", ctypes.c_int32),
        ("swiglu_fusion", ctypes.c_int32),
        ("activation_alpha", ctypes.c_float),
        ("activation_beta", ctypes.c_float),
        ("has_swiglu_limit", ctypes.c_int32),
        ("swiglu_limit", ctypes.c_float),
        ("normalize_routing_weights", ctypes.c_int32),
        ("use_sparse_mixer", ctypes.c_int32),
        ("path", ctypes.c_int32),
    ]


# moe_activation / moe_path
MOE_ACTIVATIONS = {"relu": 0, "gelu": 1, "silu": 2, "swiglu": 3, "identity": 4}
MOE_PATH_AUTO, MOE_PATH_GROUPED, MOE_PATH_GENERIC = 0, 2, 3

class QkvAttrs(ctypes.Structure):
    """Mirror of qkv_attrs (same field order and C types)."""
    _fields_ = [
        ("K", ctypes.c_int64),
        ("Nq", ctypes.c_int64),
        ("Nkv", ctypes.c_int64),
        ("block_size", ctypes.c_int64),
        ("bits", ctypes.c_int32),
        ("accuracy_level", ctypes.c_int32),
        ("epsilon", ctypes.c_float),
        ("path", ctypes.c_int32),
    ]


QKV_PATH_AUTO, QKV_PATH_DECODE, QKV_PATH_GENERIC = 0, 1, 3

_lib = None


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"QMoE CUDA library not built: {LIB_PATH} is missing "
                           "(run __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    PA = ctypes.POINTER(Attrs)
    PI64 = ctypes.POINTER(ctypes.c_int64)
    lib.qmoe_attrs_default.argtypes = [PA]
    lib.qmoe_attrs_default.restype = None
    lib.qmoe_status_string.argtypes = [ctypes.c_int]
    lib.qmoe_status_string.restype = ctypes.c_char_p
    lib.qmoe_workspace_size.argtypes = [PI64, I32, PI64, PA, ctypes.POINTER(SZ)]
    lib.qmoe_workspace_size.restype = ctypes.c_int
    lib.qmoe_hostio_workspace_size.argtypes = [PI64, I32, PI64, PA, ctypes.POINTER(SZ)]
    lib.qmoe_hostio_workspace_size.restype = ctypes.c_int
    lib.qmoe_choose_path.argtypes = [PI64, I32, PI64, PA, ctypes.POINTER(I32)]
    lib.qmoe_choose_path.restype = ctypes.c_int
    fwd = [P, PI64, I32, P, PI64, P, PI64, P, PI64, I32, P, PI64, P, PI64, I32, P, PA, P, SZ]
    lib.qmoe_forward.argtypes = fwd + [P, P, P]
    lib.qmoe_forward.restype = ctypes.c_int
    lib.qmoe_forward_hostio.argtypes = fwd + [P]
    lib.qmoe_forward_hostio.restype = ctypes.c_int
    lib.qmoe_noalloc_scratch_bytes.argtypes = []
    lib.qmoe_noalloc_scratch_bytes.restype = SZ
    lib.qmoe_forward_noalloc.argtypes = fwd[:-2] + [P, P, P]
    lib.qmoe_forward_noalloc.restype = ctypes.c_int
    lib.qmoe_noalloc_get_device_error.argtypes = [P, ctypes.POINTER(I32)]
    lib.qmoe_noalloc_get_device_error.restype = ctypes.c_int
    lib.grouped_matmul_workspace_size.argtypes = [ctypes.POINTER(SZ)]
    lib.grouped_matmul_workspace_size.restype = ctypes.c_int
    lib.grouped_matmul_workspace_size_for.argtypes = [I64, I64, I64, I64, I64, ctypes.c_int32,
                                                      ctypes.POINTER(SZ)]
    lib.grouped_matmul_workspace_size_for.restype = ctypes.c_int
    lib.grouped_matmul.argtypes = [P, I64, I64, P, I64, I64, P, I64, I32, P, P, I32, P, SZ, P]
    lib.grouped_matmul.restype = ctypes.c_int
    lib.qmoe_get_device_error.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.qmoe_get_device_error.restype = ctypes.c_int
    lib.qmoe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.qmoe_set_wait_limit_ns.restype = None
    lib.qmoe_debug_drop_stage.argtypes = [ctypes.c_int64]
    lib.qmoe_debug_drop_stage.restype = None
    lib.qmoe_profile_begin.argtypes = [I32]
    lib.qmoe_profile_begin.restype = ctypes.c_int
    lib.qmoe_profile_end.argtypes = [ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)]
    lib.qmoe_profile_end.restype = ctypes.c_int
    lib.qmoe_launch_count.argtypes = []
    lib.qmoe_launch_count.restype = ctypes.c_uint64
    PM = ctypes.POINTER(MoeAttrs)
    lib.moe_attrs_default.argtypes = [PM]
    lib.moe_attrs_default.restype = None
    for name in ("moe_workspace_size", "moe_hostio_workspace_size"):
        getattr(lib, name).argtypes = [PI64, I32, PI64, PM, ctypes.POINTER(SZ)]
        getattr(lib, name).restype = ctypes.c_int
    lib.moe_choose_path.argtypes = [PI64, I32, PI64, PM, ctypes.POINTER(I32)]
    lib.moe_choose_path.restype = ctypes.c_int
    mfwd = [P, PI64, I32, P, PI64, P, PI64, P, P, PI64, P, P, PI64, P, P, PM, P, SZ]
    lib.moe_forward.argtypes = mfwd + [P, P, P]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_forward_hostio.argtypes = mfwd + [P]
    lib.moe_forward_hostio.restype = ctypes.c_int
    lib.moe_get_device_error.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.moe_get_device_error.restype = ctypes.c_int
    PQ = ctypes.POINTER(QkvAttrs)
    lib.qkv_attrs_default.argtypes = [PQ]
    lib.qkv_attrs_default.restype = None
    lib.qkv_workspace_size.argtypes = [PI64, I32, PQ, I32, ctypes.POINTER(SZ)]
    lib.qkv_workspace_size.restype = ctypes.c_int
    lib.qkv_choose_path.argtypes = [PI64, I32, PQ, I32, ctypes.POINTER(I32)]
    lib.qkv_choose_path.restype = ctypes.c_int
    lib.matmul_nbits_qkv.argtypes = [P, PI64, I32, P, P, P, PI64, P, PI64, P, PI64, P, PI64,
                                     P, PI64, P, PI64, P, P, P, P, I32, PQ, P, SZ, P]
    lib.matmul_nbits_qkv.restype = ctypes.c_int
    _lib = lib
    return lib


def declared_functions() -> list:
    """Names of the functions include/qmoe.h, include/moe.h and include/qkv.h declare."""
    text = (open(HEADER_PATH).read() + open(MOE_HEADER_PATH).read() +
            open(QKV_HEADER_PATH).read())
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for", "switch")))


def status_string(status: int) -> str:
    try:
        return load().qmoe_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int, what: str):
    if status != OK:
        raise QmoeError(status, what)


def _shape(seq: Sequence[int]):
    arr = (ctypes.c_int64 * max(1, len(seq)))(*[int(v) for v in seq])
    return arr


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    p = t.data_ptr()
    return p if p != 0 else None


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


ACTIVATIONS = {"relu": 0, "swiglu": 1}
# include/qmoe.h QMOE_HOSTIO_DIRECT_BYTES: host-IO activations up to this size in mapped
# page-locked memory are read and written in place by the kernels
HOSTIO_DIRECT_BYTES = 1 << 20


def make_attrs(k: int = 1, expert_weight_bits: int = 4, block_size: int = 0,
               activation_type: str = "relu", activation_alpha: float = 1.0,
               activation_beta: float = 0.0, swiglu_limit: Optional[float] = None,
               swiglu_fusion: Optional[int] = None, normalize_routing_weights: int = 0,
               use_sparse_mixer: int = 0, weights_prepacked: int = -1,
               quant_type: str = "int", path: int = PATH_AUTO) -> Attrs:
    a = Attrs()
    load().qmoe_attrs_default(ctypes.byref(a))
    a.k = int(k)
    a.expert_weight_bits = int(expert_weight_bits)
    a.block_size = int(block_size or 0)
    a.activation_type = ACTIVATIONS.get(activation_type, 99) if isinstance(activation_type, str) \
        else int(activation_type)
    if swiglu_fusion is None:
        swiglu_fusion = 1 if activation_type == "swiglu" else 0
    a.swiglu_fusion = int(swiglu_fusion)
    a.activation_alpha = float(activation_alpha)
    a.activation_beta = float(activation_beta)
    a.has_swiglu_limit = 0 if swiglu_limit is None else 1
    a.swiglu_limit = 0.0 if swiglu_limit is None else float(swiglu_limit)
    a.normalize_routing_weights = int(normalize_routing_weights)
    a.use_sparse_mixer = int(use_sparse_mixer)
    a.weights_prepacked = int(weights_prepacked)
    a.quant_type_is_int = 1 if quant_type == "int" else 0
    a.path = int(path)
    return a


def workspace_size(input_shape, fc1_w_shape, attrs: Attrs, hostio: bool = False) -> int:
    lib = load()
    out = ctypes.c_size_t(0)
    fn = lib.qmoe_hostio_workspace_size if hostio else lib.qmoe_workspace_size
    _check(fn(_shape(input_shape), len(input_shape), _shape(fc1_w_shape), ctypes.byref(attrs),
              ctypes.byref(out)), "qmoe_workspace_size")
    return out.value


def choose_path(input_shape, fc1_w_shape, attrs: Attrs) -> int:
    out = ctypes.c_int32(0)
    _check(load().qmoe_choose_path(_shape(input_shape), len(input_shape), _shape(fc1_w_shape),
                                   ctypes.byref(attrs), ctypes.byref(out)), "qmoe_choose_path")
    return out.value


def alloc_workspace(nbytes: int, device=None):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def qmoe_forward(input, router_probs, fc1_experts_weights, fc1_scales, fc2_experts_weights,
                 fc2_scales, *, attrs: Optional[Attrs] = None, output=None, workspace=None,
                 topk_idx=None, topk_w=None, stream=None, **attr_kwargs):
    """QMoE layer (include/qmoe.h qmoe_forward) on torch CUDA tensors."""
    import torch
    if attrs is None:
        attrs = make_attrs(**attr_kwargs)
    if output is None:
        output = torch.empty_like(input)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(tuple(input.shape),
                                                   tuple(fc1_experts_weights.shape), attrs),
                                    input.device)
    st = load().qmoe_forward(
        _ptr(input), _shape(input.shape), input.dim(),
        _ptr(router_probs), _shape(router_probs.shape),
        _ptr(fc1_experts_weights), _shape(fc1_experts_weights.shape),
        _ptr(fc1_scales), _shape(fc1_scales.shape), fc1_scales.dim(),
        _ptr(fc2_experts_weights), _shape(fc2_experts_weights.shape),
        _ptr(fc2_scales), _shape(fc2_scales.shape), fc2_scales.dim(),
        _ptr(output), ctypes.byref(attrs), _ptr(workspace), workspace.numel(),
        _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(st, "qmoe_forward")
    return output


def qmoe_forward_noalloc(input, router_probs, fc1_experts_weights, fc1_scales,
                         fc2_experts_weights, fc2_scales, *, attrs: Attrs, output,
                         topk_idx=None, topk_w=None, stream=None):
    """qmoe_forward_noalloc: the layer with the library's fixed scratch array
    instead of a workspace, for callers that cannot allocate device memory."""
    st = load().qmoe_forward_noalloc(
        _ptr(input), _shape(input.shape), input.dim(),
        _ptr(router_probs), _shape(router_probs.shape),
        _ptr(fc1_experts_weights), _shape(fc1_experts_weights.shape),
        _ptr(fc1_scales), _shape(fc1_scales.shape), fc1_scales.dim(),
        _ptr(fc2_experts_weights), _shape(fc2_experts_weights.shape),
        _ptr(fc2_scales), _shape(fc2_scales.shape), fc2_scales.dim(),
        _ptr(output), ctypes.byref(attrs), _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(st, "qmoe_forward_noalloc")
    return output


def qmoe_forward_hostio(host_input, host_router_probs, fc1_experts_weights, fc1_scales,
                        fc2_experts_weights, fc2_scales, host_output, *, attrs: Attrs,
                        workspace, stream=None):
    """qmoe_forward_hostio: host (ideally pinned) activations in and out."""
    st = load().qmoe_forward_hostio(
        _ptr(host_input), _shape(host_input.shape), host_input.dim(),
        _ptr(host_router_probs), _shape(host_router_probs.shape),
        _ptr(fc1_experts_weights), _shape(fc1_experts_weights.shape),
        _ptr(fc1_scales), _shape(fc1_scales.shape), fc1_scales.dim(),
        _ptr(fc2_experts_weights), _shape(fc2_experts_weights.shape),
        _ptr(fc2_scales), _shape(fc2_scales.shape), fc2_scales.dim(),
        _ptr(host_output), ctypes.byref(attrs), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(st, "qmoe_forward_hostio")
    return host_output


_DTYPES = None


def _gmm_dtype(t):
    import torch
    global _DTYPES
    if _DTYPES is None:
        _DTYPES = {torch.float32: DT_F32, torch.float16: DT_F16, torch.bfloat16: DT_BF16,
                   torch.float64: DT_F64}
    return _DTYPES[t]


def grouped_matmul(input, weights, group_indices, bias=None, *, output=None, workspace=None,
                   stream=None):
    """GroupedMatMul-29 on torch CUDA tensors (include/qmoe.h grouped_matmul)."""
    import torch
    M, K = input.shape
    G, K2, N = weights.shape
    S = group_indices.shape[1]
    if K2 != K or group_indices.shape[0] != M:
        raise ValueError("grouped_matmul: inconsistent shapes")
    if output is None:
        output = torch.empty((M, S, N), dtype=input.dtype, device=input.device)
    if workspace is None:
        workspace = alloc_workspace(grouped_matmul_workspace_size(M, K, G, N, S, input.dtype),
                                    input.device)
    idt = IDX_I64 if group_indices.dtype == torch.int64 else IDX_I32
    st = load().grouped_matmul(_ptr(input), M, K, _ptr(weights), G, N, _ptr(group_indices), S,
                               idt, _ptr(bias) if bias is not None and bias.numel() else None,
                               _ptr(output), _gmm_dtype(input.dtype), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    _check(st, "grouped_matmul")
    return output


def grouped_matmul_workspace_size(M, K, G, N, S, dtype) -> int:
    """Workspace bytes that let grouped_matmul use the tensor cores for this shape
    (include/qmoe.h grouped_matmul_workspace_size_for); 256 when it cannot."""
    n = ctypes.c_size_t(0)
    _check(load().grouped_matmul_workspace_size_for(int(M), int(K), int(G), int(N), int(S),
                                                    _gmm_dtype(dtype), ctypes.byref(n)),
           "grouped_matmul_workspace_size_for")
    return n.value


def get_device_error(workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().qmoe_get_device_error(_ptr(workspace), _stream(stream), ctypes.byref(code)),
           "qmoe_get_device_error")
    return code.value


def noalloc_get_device_error(stream=None) -> int:
    """Device error word of the last qmoe_forward_noalloc call(s) on the current
    device (read and cleared in stream order)."""
    code = ctypes.c_int32(0)
    _check(load().qmoe_noalloc_get_device_error(_stream(stream), ctypes.byref(code)),
           "qmoe_noalloc_get_device_error")
    return code.value


def set_wait_limit_ns(ns: int):
    load().qmoe_set_wait_limit_ns(int(ns))


def debug_drop_stage(stage: int):
    """Test hook: producers skip the copies of pipeline stage `stage` (-1: off)."""
    load().qmoe_debug_drop_stage(int(stage))


def profile_begin(kernel_id: int):
    _check(load().qmoe_profile_begin(int(kernel_id)), "qmoe_profile_begin")


def profile_end():
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0)
    _check(load().qmoe_profile_end(ctypes.byref(n), ctypes.byref(ms)), "qmoe_profile_end")
    return n.value, ms.value


def launch_count() -> int:
    return int(load().qmoe_launch_count())


# --------------------------------------------------------------------------
# Float MoE (include/moe.h)
# --------------------------------------------------------------------------

def make_moe_attrs(k: int = 1, activation_type: str = "relu", swiglu_fusion: int = 0,
                   activation_alpha: float = 1.0, activation_beta: float = 0.0,
                   swiglu_limit: Optional[float] = None, normalize_routing_weights: int = 0,
                   use_sparse_mixer: int = 0, path: int = MOE_PATH_AUTO) -> MoeAttrs:
    a = MoeAttrs()
    load().moe_attrs_default(ctypes.byref(a))
    a.k = int(k)
    a.activation_type = (MOE_ACTIVATIONS.get(activation_type, 99)
                         if isinstance(activation_type, str) else int(activation_type))
    a.swiglu_fusion = int(swiglu_fusion)
    a.activation_alpha = float(activation_alpha)
    a.activation_beta = float(activation_beta)
    a.has_swiglu_limit = 0 if swiglu_limit is None else 1
    a.swiglu_limit = 0.0 if swiglu_limit is None else float(swiglu_limit)
    a.normalize_routing_weights = int(normalize_routing_weights)
    a.use_sparse_mixer = int(use_sparse_mixer)
    a.path = int(path)
    return a


def moe_workspace_size(input_shape, fc1_w_shape, attrs: MoeAttrs, hostio: bool = False) -> int:
    lib = load()
    out = ctypes.c_size_t(0)
    fn = lib.moe_hostio_workspace_size if hostio else lib.moe_workspace_size
    _check(fn(_shape(input_shape), len(input_shape), _shape(fc1_w_shape), ctypes.byref(attrs),
              ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_choose_path(input_shape, fc1_w_shape, attrs: MoeAttrs) -> int:
    out = ctypes.c_int32(0)
    _check(load().moe_choose_path(_shape(input_shape), len(input_shape), _shape(fc1_w_shape),
                                  ctypes.byref(attrs), ctypes.byref(out)), "moe_choose_path")
    return out.value


def _opt_shape(t):
    return None if t is None else _shape(t.shape)


def moe_forward(input, router_probs, fc1_experts_weights, fc2_experts_weights, *,
                fc1_experts_bias=None, fc2_experts_bias=None, fc3_experts_weights=None,
                fc3_experts_bias=None, attrs: Optional[MoeAttrs] = None, output=None,
                workspace=None, topk_idx=None, topk_w=None, stream=None, **attr_kwargs):
    """Float MoE layer (include/moe.h moe_forward) on torch CUDA tensors."""
    import torch
    if attrs is None:
        attrs = make_moe_attrs(**attr_kwargs)
    if output is None:
        output = torch.empty_like(input)
    if workspace is None:
        workspace = alloc_workspace(moe_workspace_size(tuple(input.shape),
                                                       tuple(fc1_experts_weights.shape), attrs),
                                    input.device)
    st = load().moe_forward(
        _ptr(input), _shape(input.shape), input.dim(),
        _ptr(router_probs), _shape(router_probs.shape),
        _ptr(fc1_experts_weights), _shape(fc1_experts_weights.shape), _ptr(fc1_experts_bias),
        _ptr(fc2_experts_weights), _shape(fc2_experts_weights.shape), _ptr(fc2_experts_bias),
        _ptr(fc3_experts_weights), _opt_shape(fc3_experts_weights), _ptr(fc3_experts_bias),
        _ptr(output), ctypes.byref(attrs), _ptr(workspace), workspace.numel(),
        _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(st, "moe_forward")
    return output


def moe_forward_hostio(host_input, host_router_probs, fc1_experts_weights, fc2_experts_weights,
                       host_output, *, attrs: MoeAttrs, workspace, fc1_experts_bias=None,
                       fc2_experts_bias=None, fc3_experts_weights=None, fc3_experts_bias=None,
                       stream=None):
    """moe_forward_hostio: host (ideally pinned) activations in and out."""
    st = load().moe_forward_hostio(
        _ptr(host_input), _shape(host_input.shape), host_input.dim(),
        _ptr(host_router_probs), _shape(host_router_probs.shape),
        _ptr(fc1_experts_weights), _shape(fc1_experts_weights.shape), _ptr(fc1_experts_bias),
        _ptr(fc2_experts_weights), _shape(fc2_experts_weights.shape), _ptr(fc2_experts_bias),
        _ptr(fc3_experts_weights), _opt_shape(fc3_experts_weights), _ptr(fc3_experts_bias),
        _ptr(host_output), ctypes.byref(attrs), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(st, "moe_forward_hostio")
    return host_output


def moe_get_device_error(workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().moe_get_device_error(_ptr(workspace), _stream(stream), ctypes.byref(code)),
           "moe_get_device_error")
    return code.value


# --------------------------------------------------------------------------
# RMSNorm + 4-bit Q/K/V projection (include/qkv.h)
# --------------------------------------------------------------------------

def make_qkv_attrs(K: int, Nq: int, Nkv: int, block_size: int = 32, bits: int = 4,
                   accuracy_level: int = 0, epsilon: Optional[float] = None,
                   path: int = QKV_PATH_AUTO) -> QkvAttrs:
    a = QkvAttrs()
    load().qkv_attrs_default(ctypes.byref(a))
    a.K, a.Nq, a.Nkv, a.block_size = int(K), int(Nq), int(Nkv), int(block_size)
    a.bits, a.accuracy_level = int(bits), int(accuracy_level)
    if epsilon is not None:
        a.epsilon = float(epsilon)
    a.path = int(path)
    return a


def qkv_workspace_size(a_shape, attrs: QkvAttrs, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(load().qkv_workspace_size(_shape(a_shape), len(a_shape), ctypes.byref(attrs),
                                     _gmm_dtype(dtype), ctypes.byref(out)), "qkv_workspace_size")
    return out.value


def qkv_choose_path(a_shape, attrs: QkvAttrs, dtype) -> int:
    out = ctypes.c_int32(0)
    _check(load().qkv_choose_path(_shape(a_shape), len(a_shape), ctypes.byref(attrs),
                                  _gmm_dtype(dtype), ctypes.byref(out)), "qkv_choose_path")
    return out.value


def matmul_nbits_qkv(A, norm_scale, q_B, q_scales, k_B, k_scales, v_B, v_scales, *, skip=None,
                     residual=None, attrs: Optional[QkvAttrs] = None, outputs=None,
                     workspace=None, stream=None, **attr_kwargs):
    """RMSNorm + 4-bit Q/K/V projection (include/qkv.h matmul_nbits_qkv) on torch CUDA
    tensors.  residual=True allocates the input_skip_bias_sum output (needs skip).
    Returns (Q, K, V) or (Q, K, V, residual)."""
    import torch
    Kdim = A.shape[-1]
    if attrs is None:
        attrs = make_qkv_attrs(K=Kdim, Nq=q_B.shape[0], Nkv=k_B.shape[0], **attr_kwargs)
    lead = tuple(A.shape[:-1])
    if outputs is None:
        outputs = (torch.empty(lead + (attrs.Nq,), dtype=A.dtype, device=A.device),
                   torch.empty(lead + (attrs.Nkv,), dtype=A.dtype, device=A.device),
                   torch.empty(lead + (attrs.Nkv,), dtype=A.dtype, device=A.device))
    res = None
    if residual is True:
        res = torch.empty_like(A)
    elif residual is not None and residual is not False:
        res = residual
    if workspace is None:
        workspace = alloc_workspace(qkv_workspace_size(tuple(A.shape), attrs, A.dtype), A.device)
    Q, Ko, V = outputs
    st = load().matmul_nbits_qkv(
        _ptr(A), _shape(A.shape), A.dim(), _ptr(skip), _ptr(norm_scale),
        _ptr(q_B), _shape(q_B.shape), _ptr(q_scales), _shape(q_scales.shape),
        _ptr(k_B), _shape(k_B.shape), _ptr(k_scales), _shape(k_scales.shape),
        _ptr(v_B), _shape(v_B.shape), _ptr(v_scales), _shape(v_scales.shape),
        _ptr(Q), _ptr(Ko), _ptr(V), _ptr(res), _gmm_dtype(A.dtype), ctypes.byref(attrs),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "matmul_nbits_qkv")
    return (Q, Ko, V) if res is None else (Q, Ko, V, res)
