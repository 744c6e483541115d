"""CPU reference oracle for the QMoE layer, the float MoE layer and GroupedMatMul
(test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a ctypes wrapper over the plain
double-precision C restatements in ``qmoe_oracle.c``, ``moe_oracle.c`` (the
float MoE of the [MoE README]) and ``qkv_oracle.c`` (the RMSNorm + 4-bit
Q/K/V projection of the [MatMulNBitsQkv manifest]); it shares no code with
the CUDA library and never calls it.  The wrapper only marshals arrays and
derives shapes ([QMoE manifest] derive.numTokens / derive.hiddenSize: the
token count is the product of the leading input dimensions).

Functions whose result has no independent pin say so here and in the design
notes: ``swiglu_limit`` handling (reading of [QMoE manifest]
attributeDescriptions.swiglu_limit) is "parity unpinned", in both layers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("qmoe_oracle.c", "moe_oracle.c", "qkv_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_INDEX = -1
BAD_ARG = -2


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into liboracle.so with gcc (no CUDA involved)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(f) for f in _SRCS)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, *_SRCS,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        C = ctypes.c_int
        lib.oracle_grouped_matmul.argtypes = [P, I64, I64, P, I64, I64, P, I64, P, P]
        lib.oracle_grouped_matmul.restype = C
        lib.oracle_grouped_matmul_decomposed.argtypes = [P, I64, I64, P, I64, I64, P, I64, P, P]
        lib.oracle_grouped_matmul_decomposed.restype = C
        lib.oracle_weight_code.argtypes = [P, I64, C]
        lib.oracle_weight_code.restype = C
        lib.oracle_dequant.argtypes = [P, P, I64, C, I64]
        lib.oracle_dequant.restype = D
        lib.oracle_dequant_rows.argtypes = [P, P, I64, I64, C, I64, P]
        lib.oracle_dequant_rows.restype = None
        lib.oracle_route.argtypes = [P, I64, I64, P, P]
        lib.oracle_route.restype = C
        lib.oracle_activation.argtypes = [P, I64, C, D, D, C, D, P]
        lib.oracle_activation.restype = None
        lib.oracle_qmoe.argtypes = [P, I64, P, I64, P, P, P, P, I64, C, I64, C, D, D,
                                    C, D, I64, P, I64, C, P, P, P, C]
        lib.oracle_qmoe.restype = C
        lib.oracle_moe_route.argtypes = [P, I64, I64, C, P, P]
        lib.oracle_moe_route.restype = C
        lib.oracle_moe_activation.argtypes = [P, P, I64, C, C, D, D, C, D, P]
        lib.oracle_moe_activation.restype = None
        lib.oracle_moe.argtypes = [P, I64, P, I64, P, P, P, P, P, P, I64, C, C, D, D, C, D,
                                   I64, C, P, I64, C, P, P, P, C]
        lib.oracle_moe.restype = C
        lib.oracle_qkv_code.argtypes = [P, I64, I64, I64, I64]
        lib.oracle_qkv_code.restype = C
        lib.oracle_qkv.argtypes = [P, P, P, I64, I64, P, P, I64, P, P, P, P, I64, I64, D,
                                   P, P, P, P, P]
        lib.oracle_qkv.restype = C
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# --------------------------------------------------------------------------
# GroupedMatMul  ([GroupedMatMul-29] Summary)
# --------------------------------------------------------------------------

def grouped_matmul(inp, weights, group_indices, bias=None, decomposed=False):
    """output[m, i] = input[m] @ weights[group_indices[m, i]] (+ bias[g]).

    All arithmetic in float64.  Returns (output [M,S,N] float64, status);
    status is BAD_INDEX when an index lies outside [0, G).
    """
    lib = _load()
    x = _c(inp, np.float64)
    w = _c(weights, np.float64)
    idx = _c(group_indices, np.int64)
    M, K = x.shape
    G, K2, N = w.shape
    assert K2 == K
    S = idx.shape[1] if idx.ndim == 2 else 0
    b = None if bias is None else _c(bias, np.float64)
    out = np.zeros((M, S, N), dtype=np.float64)
    fn = lib.oracle_grouped_matmul_decomposed if decomposed else lib.oracle_grouped_matmul
    st = fn(_ptr(x), M, K, _ptr(w), G, N, _ptr(idx), S,
            None if b is None else _ptr(b), _ptr(out))
    return out, st


# --------------------------------------------------------------------------
# QMoE pieces
# --------------------------------------------------------------------------

def weight_code(packed_row, j, bits):
    lib = _load()
    row = _c(packed_row, np.uint8)
    return lib.oracle_weight_code(_ptr(row), j, bits)


def dequant_rows(packed, scales, K, bits, block_size):
    """Dequantize a [rows, K/pack] packed matrix with its scales -> [rows, K]."""
    lib = _load()
    pk = _c(packed, np.uint8)
    sc = _c(scales, np.float32)
    rows = pk.shape[0]
    out = np.zeros((rows, K), dtype=np.float64)
    lib.oracle_dequant_rows(_ptr(pk), _ptr(sc), rows, K, bits, block_size, _ptr(out))
    return out


def route(logits, k):
    """Top-k selection and softmax over the selected logits, per row."""
    lib = _load()
    lg = _c(logits, np.float32)
    T, E = lg.shape
    sel = np.zeros((T, k), dtype=np.int32)
    p = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        st = lib.oracle_route(_ptr(lg[t]), E, k, _ptr(sel[t]), _ptr(p[t]))
        if st != OK:
            raise ValueError(f"oracle_route failed with {st}")
    return sel, p


def activation(h, inter, act, alpha=1.0, beta=0.0, swiglu_limit=None):
    lib = _load()
    hh = _c(h, np.float64)
    a = np.zeros(inter, dtype=np.float64)
    lib.oracle_activation(_ptr(hh), inter, 1 if act == "swiglu" else 0, alpha, beta,
                          0 if swiglu_limit is None else 1,
                          0.0 if swiglu_limit is None else float(swiglu_limit), _ptr(a))
    return a


def qmoe(x, logits, w1, s1, w2, s2, *, k, expert_weight_bits=4, block_size=0,
         activation_type="relu", activation_alpha=1.0, activation_beta=0.0,
         swiglu_limit=None, tokens=None, dense=False, nthreads=1):
    """QMoE layer output for the listed tokens (all tokens when None).

    Returns (y [ntok, H] float64, sel [ntok, k] int32, p [ntok, k] float64).
    """
    lib = _load()
    xs = _c(x, np.float32)
    H = xs.shape[-1]
    xs = xs.reshape(-1, H)
    lg = _c(logits, np.float32)
    E = lg.shape[1]
    bits = int(expert_weight_bits)
    fusion = 2 if activation_type == "swiglu" else 1
    w1a = _c(w1, np.uint8)
    w2a = _c(w2, np.uint8)
    s1a = _c(s1, np.float32)
    s2a = _c(s2, np.float32)
    I = w1a.shape[1] // fusion
    if tokens is None:
        tok = np.arange(xs.shape[0], dtype=np.int64)
    else:
        tok = _c(tokens, np.int64)
    ntok = tok.shape[0]
    y = np.zeros((ntok, H), dtype=np.float64)
    sel = np.zeros((ntok, k), dtype=np.int32)
    p = np.zeros((ntok, k), dtype=np.float64)
    st = lib.oracle_qmoe(_ptr(xs), H, _ptr(lg), E, _ptr(w1a), _ptr(s1a), _ptr(w2a),
                         _ptr(s2a), I, bits, int(block_size),
                         1 if activation_type == "swiglu" else 0,
                         float(activation_alpha), float(activation_beta),
                         0 if swiglu_limit is None else 1,
                         0.0 if swiglu_limit is None else float(swiglu_limit),
                         int(k), _ptr(tok), ntok, 1 if dense else 0,
                         _ptr(y), _ptr(sel), _ptr(p), int(nthreads))
    if st != OK:
        raise ValueError(f"oracle_qmoe failed with {st}")
    return y, sel, p


# --------------------------------------------------------------------------
# Float MoE  ([MoE README] Description, Inputs, Attributes)
# --------------------------------------------------------------------------

MOE_ACTIVATIONS = {"relu": 0, "gelu": 1, "silu": 2, "swiglu": 3, "identity": 4}


def moe_route(logits, k, normalize_routing_weights=0):
    """Softmax over all experts, the k most probable (descending), optionally
    renormalised over the selection.  Returns (sel [T,k] int32, w [T,k] f64)."""
    lib = _load()
    lg = _c(logits, np.float32)
    T, E = lg.shape
    sel = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        st = lib.oracle_moe_route(_ptr(lg[t]), E, k, int(normalize_routing_weights),
                                  _ptr(sel[t]), _ptr(w[t]))
        if st != OK:
            raise ValueError(f"oracle_moe_route failed with {st}")
    return sel, w


def moe_activation(h1, inter, act, h3=None, swiglu_fusion=0, alpha=1.0, beta=0.0,
                   swiglu_limit=None):
    """The activation of one expert row: h1 (fusion*inter values), h3 (inter or None)."""
    lib = _load()
    a1 = _c(h1, np.float64)
    a3 = None if h3 is None else _c(h3, np.float64)
    out = np.zeros(inter, dtype=np.float64)
    lib.oracle_moe_activation(_ptr(a1), None if a3 is None else _ptr(a3), inter,
                              MOE_ACTIVATIONS[act], int(swiglu_fusion), float(alpha),
                              float(beta), 0 if swiglu_limit is None else 1,
                              0.0 if swiglu_limit is None else float(swiglu_limit), _ptr(out))
    return out


def qmoe_batched(x, logits, w1, s1, w2, s2, *, k, expert_weight_bits=4, block_size=0,
                 activation_type="relu", activation_alpha=1.0, activation_beta=0.0,
                 swiglu_limit=None):
    """QMoE layer output for every token, evaluated expert by expert.

    The same steps as qmoe(), for checking whole large batches in seconds:
    routing (route), dequantisation (dequant_rows) and the activation
    (activation) are the C restatement's own functions, while the FC1 and FC2
    products of the tokens routed to one expert are fp64 matrix products
    (numpy).  A token's k weighted expert outputs are added in expert order
    rather than in selection order, which differs from qmoe() only by fp64
    rounding.  Returns (y [T, H] float64, sel [T, k] int32, p [T, k] float64).
    """
    xs = _c(x, np.float64)
    H = xs.shape[-1]
    xs = xs.reshape(-1, H)
    T = xs.shape[0]
    lg = _c(logits, np.float32)
    E = lg.shape[1]
    bits = int(expert_weight_bits)
    fusion = 2 if activation_type == "swiglu" else 1
    w1a = _c(w1, np.uint8)
    w2a = _c(w2, np.uint8)
    s1a = _c(s1, np.float32)
    s2a = _c(s2, np.float32)
    I = w1a.shape[1] // fusion
    sel, p = route(lg, k)
    y = np.zeros((T, H), dtype=np.float64)
    if I == 0:
        return y, sel, p
    for e in range(E):
        t_idx, i_idx = np.nonzero(sel == e)
        if t_idx.size == 0:
            continue
        W1 = dequant_rows(w1a[e], s1a[e].reshape(w1a.shape[1], -1), H, bits, int(block_size))
        W2 = dequant_rows(w2a[e], s2a[e].reshape(H, -1), I, bits, int(block_size))
        h = xs[t_idx] @ W1.T
        a = np.empty((t_idx.size, I), dtype=np.float64)
        for r in range(t_idx.size):
            a[r] = activation(h[r], I, activation_type, activation_alpha, activation_beta,
                              swiglu_limit)
        y[t_idx] += p[t_idx, i_idx][:, None] * (a @ W2.T)
    return y, sel, p


def moe(x, logits, fc1_w, fc2_w, *, k, fc1_bias=None, fc2_bias=None, fc3_w=None,
        fc3_bias=None, activation_type="relu", swiglu_fusion=0, activation_alpha=1.0,
        activation_beta=0.0, swiglu_limit=None, normalize_routing_weights=0,
        tokens=None, dense=False, nthreads=1):
    """Float MoE layer output for the listed tokens (all tokens when None).

    Returns (y [ntok, H] float64, sel [ntok, k] int32, w [ntok, k] float64).
    """
    lib = _load()
    xs = _c(x, np.float32)
    H = xs.shape[-1]
    xs = xs.reshape(-1, H)
    lg = _c(logits, np.float32)
    E = lg.shape[1]
    w1 = _c(fc1_w, np.float32)
    w2 = _c(fc2_w, np.float32)
    I = w2.shape[2]
    opt = [None if a is None else _c(a, np.float32) for a in (fc1_bias, fc2_bias, fc3_w, fc3_bias)]
    tok = (np.arange(xs.shape[0], dtype=np.int64) if tokens is None
           else _c(tokens, np.int64))
    ntok = tok.shape[0]
    y = np.zeros((ntok, H), dtype=np.float64)
    sel = np.zeros((ntok, k), dtype=np.int32)
    w = np.zeros((ntok, k), dtype=np.float64)
    b1, b2, w3, b3 = [None if a is None else _ptr(a) for a in opt]
    st = lib.oracle_moe(_ptr(xs), H, _ptr(lg), E, _ptr(w1), b1, _ptr(w2), b2, w3, b3, I,
                        MOE_ACTIVATIONS[activation_type], int(swiglu_fusion),
                        float(activation_alpha), float(activation_beta),
                        0 if swiglu_limit is None else 1,
                        0.0 if swiglu_limit is None else float(swiglu_limit), int(k),
                        int(normalize_routing_weights), _ptr(tok), ntok, 1 if dense else 0,
                        _ptr(y), _ptr(sel), _ptr(w), int(nthreads))
    if st != OK:
        raise ValueError(f"oracle_moe failed with {st}")
    return y, sel, w


# --------------------------------------------------------------------------
# RMSNorm + 4-bit Q/K/V projection  ([MatMulNBitsQkv manifest])
# --------------------------------------------------------------------------

QKV_EPSILON = 9.999999974752427e-7   # attributes.epsilon default


def qkv_code(packed, n, k, K, block_size=32):
    """Code of element (n, k) of a [N, kBlocks, blob] packed weight."""
    lib = _load()
    pk = _c(packed, np.uint8)
    kblocks = (K + block_size - 1) // block_size
    return lib.oracle_qkv_code(_ptr(pk), int(n), int(k), kblocks, block_size)


def qkv(A, norm_scale, q_B, q_scales, k_B, k_scales, v_B, v_scales, *, skip=None,
        block_size=32, epsilon=QKV_EPSILON, residual=False, normed=False):
    """Q, K, V [rows, N] float64 for A [..., K] (leading dims flattened); with
    residual=True also x = A + skip, with normed=True also the normalised rows."""
    lib = _load()
    a = _c(A, np.float64)
    K = a.shape[-1]
    a = a.reshape(-1, K)
    rows = a.shape[0]
    sk = None if skip is None else _c(skip, np.float64).reshape(-1, K)
    g = _c(norm_scale, np.float64)
    qb, kb, vb = (_c(t, np.uint8) for t in (q_B, k_B, v_B))
    qs, ks, vs = (_c(t, np.float64) for t in (q_scales, k_scales, v_scales))
    Nq, Nkv = qb.shape[0], kb.shape[0]
    Q = np.zeros((rows, Nq))
    Ko = np.zeros((rows, Nkv))
    V = np.zeros((rows, Nkv))
    res = np.zeros((rows, K)) if residual else None
    nrm = np.zeros((rows, K)) if normed else None
    st = lib.oracle_qkv(_ptr(a), None if sk is None else _ptr(sk), _ptr(g), rows, K,
                        _ptr(qb), _ptr(qs), Nq, _ptr(kb), _ptr(ks), _ptr(vb), _ptr(vs), Nkv,
                        int(block_size), float(epsilon), _ptr(Q), _ptr(Ko), _ptr(V),
                        None if res is None else _ptr(res), None if nrm is None else _ptr(nrm))
    if st != OK:
        raise ValueError(f"oracle_qkv failed with {st}")
    out = [Q, Ko, V]
    if residual:
        out.append(res)
    if normed:
        out.append(nrm)
    return tuple(out)
