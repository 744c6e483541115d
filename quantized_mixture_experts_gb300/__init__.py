"""GB300 (sm_103a) QMoE layer: a C-ABI CUDA library plus a thin ctypes binding.

The layer is the com.microsoft.QMoE operator (top-k routing with a softmax over
the selected logits, symmetric 4/8-bit expert weights, ReLU or interleaved
SwiGLU, weighted combine) with ONNX GroupedMatMul-29 as its core operation.
The same library carries the float com.microsoft.MoE layer (softmax over all
experts, FC1/FC3/FC2 with biases, relu/gelu/silu/swiglu/identity) and the
com.microsoft.MatMulNBitsQkv RMSNorm + 4-bit Q/K/V projection.
"""
from .binding import (  # noqa: F401
    Attrs, QmoeError, make_attrs, workspace_size, choose_path, alloc_workspace, qmoe_forward,
    qmoe_forward_hostio, grouped_matmul, get_device_error, set_wait_limit_ns, profile_begin,
    profile_end, launch_count, load, declared_functions,
    PATH_AUTO, PATH_DECODE, PATH_GROUPED, PATH_GENERIC, PATH_NAMES,
    DEVERR_NONE, DEVERR_INDEX, DEVERR_NONFINITE, DEVERR_TIMEOUT,
    KERNEL_ROUTE, KERNEL_GROUP, KERNEL_FC1, KERNEL_FC2, KERNEL_COMBINE, KERNEL_GMM,
    MoeAttrs, make_moe_attrs, moe_workspace_size, moe_choose_path, moe_forward,
    moe_forward_hostio, moe_get_device_error, MOE_PATH_AUTO, MOE_PATH_GROUPED, MOE_PATH_GENERIC,
    QkvAttrs, make_qkv_attrs, qkv_workspace_size, qkv_choose_path, matmul_nbits_qkv,
    QKV_PATH_AUTO, QKV_PATH_DECODE, QKV_PATH_GENERIC,
)
