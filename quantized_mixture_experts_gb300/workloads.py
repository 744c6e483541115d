"""Seeded synthetic inputs for the QMoE layer.

This module only draws random numbers with the shapes, value distributions and
load skew of the five benchmark workloads; it holds none of the layer's
arithmetic.  Both the CUDA path and the CPU oracle receive the arrays it
returns, so neither side generates its own inputs.

Recipe (every workload):
  * activations  fp32 ~ N(0, 1), shaped like the workload's input
    (rank 2 ``[T, H]`` or rank 3 ``[B, S, H]``);
  * router logits fp32 ~ N(0, sigma^2) with sigma = 1 or 2 (the workload
    text writes "N(0,2)", read as a standard deviation of 2);
  * the many-small-experts workload adds a per-expert bias
    ``-1.1 * ln(1 + pi(e))`` (pi a seeded permutation) to skew load like a
    Zipf(s=1.1) popularity law;
  * any logit row whose k+1 largest values contain a repeated value is
    redrawn, so the top-k set is unique;
  * packed expert weights are uniform random bytes (4-bit codes uniform on
    0..15, 8-bit codes on 0..255);
  * scales fp32 ~ U[lo, hi] (U[0.005, 0.02] for the tiny workload,
    U[0.002, 0.01] otherwise).
Seeds are ``workload_index * 1000 + tensor_id`` with numpy's PCG64.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    input_shape: Tuple[int, ...]
    hidden: int
    inter: int
    experts: int
    k: int
    bits: int
    block_size: int          # 0 = column-wise scales
    activation: str          # "relu" | "swiglu"
    logit_sigma: float = 1.0
    scale_lo: float = 0.002
    scale_hi: float = 0.01
    zipf_s: float = 0.0      # 0 = no skew bias
    alpha: float = 1.0
    beta: float = 0.0
    swiglu_limit: Optional[float] = None

    @property
    def tokens(self) -> int:
        n = 1
        for d in self.input_shape[:-1]:
            n *= d
        return n

    @property
    def fusion(self) -> int:
        return 2 if self.activation == "swiglu" else 1

    @property
    def pack(self) -> int:
        return 2 if self.bits == 4 else 1

    def attrs(self) -> dict:
        return dict(k=self.k, expert_weight_bits=self.bits, block_size=self.block_size,
                    activation_type=self.activation, activation_alpha=self.alpha,
                    activation_beta=self.beta, swiglu_limit=self.swiglu_limit)

    def with_tokens(self, T: int, name: Optional[str] = None) -> "Workload":
        return dataclasses.replace(self, name=name or f"{self.name}_T{T}",
                                   input_shape=(T, self.hidden))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 0, (16, 64), 64, 128, 4, 2, 4, 0, "relu",
                     logit_sigma=1.0, scale_lo=0.005, scale_hi=0.02),
    "decode": Workload("decode", 1, (8, 4096), 4096, 14336, 8, 2, 4, 32, "swiglu",
                       logit_sigma=2.0),
    "prefill": Workload("prefill", 2, (2, 2048, 4096), 4096, 14336, 8, 2, 4, 128,
                        "swiglu", logit_sigma=2.0),
    "many_small": Workload("many_small", 3, (2048, 2048), 2048, 1024, 64, 8, 8, 0,
                           "swiglu", logit_sigma=1.0, zipf_s=1.1),
    "large_e": Workload("large_e", 4, (4, 4096, 2048), 2048, 768, 128, 8, 4, 64,
                        "swiglu", logit_sigma=1.0),
}


def _rng(wl: Workload, tensor_id: int, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng(wl.index * 1000 + tensor_id + 100000 * salt)


def _logits(wl: Workload, T: int, salt: int) -> np.ndarray:
    E, k = wl.experts, wl.k
    rng = _rng(wl, 2, salt)
    lg = (rng.standard_normal((T, E), dtype=np.float32) * np.float32(wl.logit_sigma))
    bias = None
    if wl.zipf_s > 0:
        perm = _rng(wl, 7, salt).permutation(E)
        bias = (-wl.zipf_s * np.log1p(perm.astype(np.float64))).astype(np.float32)
        lg = lg + bias[None, :]
    redraw = _rng(wl, 8, salt)
    m = min(k + 1, E)
    for _ in range(100):
        top = -np.sort(-lg, axis=1)[:, :m]
        bad = np.nonzero(np.any(top[:, 1:] == top[:, :-1], axis=1))[0]
        if bad.size == 0:
            break
        fresh = redraw.standard_normal((bad.size, E), dtype=np.float32) * np.float32(wl.logit_sigma)
        if bias is not None:
            fresh = fresh + bias[None, :]
        lg[bad] = fresh
    return np.ascontiguousarray(lg, dtype=np.float32)


def make_inputs(wl: Workload, salt: int = 0) -> dict:
    """Draw every input tensor of one QMoE call for workload ``wl``."""
    T, H, I, E = wl.tokens, wl.hidden, wl.inter, wl.experts
    f, pk = wl.fusion, wl.pack
    x = _rng(wl, 1, salt).standard_normal(wl.input_shape, dtype=np.float32)
    logits = _logits(wl, T, salt)
    w1 = _rng(wl, 3, salt).integers(0, 256, (E, f * I, H // pk), dtype=np.uint8)
    w2 = _rng(wl, 5, salt).integers(0, 256, (E, H, I // pk), dtype=np.uint8)
    if wl.block_size:
        s1_shape = (E, f * I, H // wl.block_size)
        s2_shape = (E, H, I // wl.block_size)
    else:
        s1_shape = (E, f * I)
        s2_shape = (E, H)
    s1 = _rng(wl, 4, salt).uniform(wl.scale_lo, wl.scale_hi, s1_shape).astype(np.float32)
    s2 = _rng(wl, 6, salt).uniform(wl.scale_lo, wl.scale_hi, s2_shape).astype(np.float32)
    return dict(input=x, router_probs=logits, fc1_experts_weights=w1, fc1_scales=s1,
                fc2_experts_weights=w2, fc2_scales=s2)


def tied_logits(T: int, E: int, seed: int, levels: int = 4, scale: float = 0.5) -> np.ndarray:
    """Router logits with exact ties in almost every row, for the tie-order cases.

    Each logit is ``scale * j`` with j drawn uniformly from ``0 .. levels - 1``,
    so a row of E > levels experts holds repeated values, and with E much
    larger than ``levels`` the k-th and (k+1)-th largest values are usually
    equal.  A fraction of the rows gets one draw shifted by -0.0 or a large
    margin to vary the pattern.  The values are exact in fp32.
    """
    rng = np.random.default_rng(seed)
    lg = (rng.integers(0, levels, (T, E)).astype(np.float32) * np.float32(scale))
    flip = rng.random(T) < 0.25
    cols = rng.integers(0, E, T)
    lg[flip, cols[flip]] = np.float32(scale * (levels + 2))   # one clear winner
    zero = lg == 0
    neg = zero & (rng.random((T, E)) < 0.5)
    lg[neg] = np.float32(-0.0)                                 # -0 ties with +0
    return np.ascontiguousarray(lg, dtype=np.float32)


def sample_tokens(logits_sel: np.ndarray, T: int, n: int, seed: int) -> np.ndarray:
    """Seeded token subset of size >= n that touches every selected expert.

    ``logits_sel`` is the [T, k] selected-expert table of the workload (the
    oracle's routing), used only to add one token per touched expert.
    """
    rng = np.random.default_rng(seed)
    n = min(n, T)
    chosen = set(rng.choice(T, size=n, replace=False).tolist())
    first = {}
    for t in range(T):
        for e in logits_sel[t].tolist():
            first.setdefault(e, t)
    chosen.update(first.values())
    return np.array(sorted(chosen), dtype=np.int64)


# ---------------------------------------------------------------------------
# Float (unquantized) MoE layer inputs
# ---------------------------------------------------------------------------
#
# Recipe: activations fp32 ~ N(0, 1); router logits fp32 ~ N(0, sigma^2) with
# the same tie redraw as above; expert weights fp32 ~ N(0, 1/fan_in) (fan_in =
# H for FC1/FC3, I for FC2), so that every projection keeps unit scale; biases
# fp32 ~ N(0, 0.1^2) when the workload has them.  Seeds are
# ``workload_index * 1000 + tensor_id``.  The README names no benchmark shape;
# the decode and prefill workloads reuse the QMoE layer's shapes with SwiGLU
# from a separate FC3 (the README's default swiglu_fusion 0).


@dataclasses.dataclass(frozen=True)
class FloatWorkload:
    name: str
    index: int
    input_shape: Tuple[int, ...]
    hidden: int
    inter: int
    experts: int
    k: int
    activation: str              # relu | gelu | silu | swiglu | identity
    swiglu_fusion: int = 0
    fc3: bool = False            # FC3 weights present (needed by swiglu_fusion 0)
    biases: bool = False
    normalize: int = 0
    logit_sigma: float = 1.0
    alpha: float = 1.0
    beta: float = 0.0
    swiglu_limit: Optional[float] = None

    @property
    def tokens(self) -> int:
        n = 1
        for d in self.input_shape[:-1]:
            n *= d
        return n

    @property
    def fc1_rows(self) -> int:
        fused = self.activation == "swiglu" and self.swiglu_fusion != 0
        return (2 if fused else 1) * self.inter

    def attrs(self) -> dict:
        return dict(k=self.k, activation_type=self.activation, swiglu_fusion=self.swiglu_fusion,
                    activation_alpha=self.alpha, activation_beta=self.beta,
                    swiglu_limit=self.swiglu_limit,
                    normalize_routing_weights=self.normalize)

    def replace(self, **kw) -> "FloatWorkload":
        return dataclasses.replace(self, **kw)


FLOAT_WORKLOADS = {
    "float_tiny": FloatWorkload("float_tiny", 40, (16, 64), 64, 128, 4, 2, "relu", biases=True),
    "float_decode": FloatWorkload("float_decode", 41, (8, 4096), 4096, 14336, 8, 2, "swiglu",
                                  swiglu_fusion=0, fc3=True, logit_sigma=2.0),
    "float_prefill": FloatWorkload("float_prefill", 42, (2, 2048, 4096), 4096, 14336, 8, 2,
                                   "swiglu", swiglu_fusion=0, fc3=True, logit_sigma=2.0),
    # prefill-like load per expert (about 1024 routed rows) with 1.4 GB of weights, for
    # counter captures that must stay small
    "float_prefill_e4": FloatWorkload("float_prefill_e4", 43, (2048, 4096), 4096, 7168, 4, 2,
                                      "swiglu", swiglu_fusion=0, fc3=True, logit_sigma=2.0),
}


def make_float_inputs(wl: FloatWorkload, salt: int = 0) -> dict:
    """Draw every input tensor of one float MoE call for workload ``wl``."""
    T, H, I, E = wl.tokens, wl.hidden, wl.inter, wl.experts
    fake = Workload(wl.name, wl.index, wl.input_shape, H, I, E, wl.k, 4, 0, "relu",
                    logit_sigma=wl.logit_sigma)

    def normal(tid, shape, sd):
        g = _rng(fake, tid, salt)
        return (g.standard_normal(shape, dtype=np.float32) * np.float32(sd))

    out = dict(
        input=_rng(fake, 1, salt).standard_normal(wl.input_shape, dtype=np.float32),
        router_probs=_logits(fake, T, salt),
        fc1_experts_weights=normal(3, (E, wl.fc1_rows, H), 1.0 / np.sqrt(H)),
        fc2_experts_weights=normal(5, (E, H, I), 1.0 / np.sqrt(max(I, 1))))
    if wl.fc3:
        out["fc3_experts_weights"] = normal(9, (E, I, H), 1.0 / np.sqrt(H))
    if wl.biases:
        out["fc1_experts_bias"] = normal(4, (E, wl.fc1_rows), 0.1)
        out["fc2_experts_bias"] = normal(6, (E, H), 0.1)
        if wl.fc3:
            out["fc3_experts_bias"] = normal(10, (E, I), 0.1)
    return out


# ---------------------------------------------------------------------------
# RMSNorm + 4-bit Q/K/V projection inputs
# ---------------------------------------------------------------------------
#
# Recipe: A ~ N(0, 1) and skip ~ N(0, 0.5^2) in T1; norm_scale ~ U[0.5, 1.5];
# packed weights uniform random bytes [N, kBlocks, 16]; block scales
# ~ U[0.002, 0.01] in T1.  The manifest names no benchmark shape: the decode
# workloads take grouped-query attention projections (K 8192 with 64 query
# heads and 8 key/value heads of 128: Nq 8192, Nkv 1024; and K 16384 with 128
# query heads) for 8 rows.


@dataclasses.dataclass(frozen=True)
class QkvWorkload:
    name: str
    index: int
    input_shape: Tuple[int, ...]
    K: int
    Nq: int
    Nkv: int
    dtype: str = "float32"       # T1: float32 | float16
    skip: bool = False
    residual: bool = False

    @property
    def rows(self) -> int:
        n = 1
        for d in self.input_shape[:-1]:
            n *= d
        return n

    @property
    def kblocks(self) -> int:
        return (self.K + 31) // 32


QKV_WORKLOADS = {
    "qkv_tiny": QkvWorkload("qkv_tiny", 70, (4, 256), 256, 128, 64, "float32", True, True),
    "qkv_decode": QkvWorkload("qkv_decode", 71, (8, 8192), 8192, 8192, 1024, "float16"),
    "qkv_decode_f32": QkvWorkload("qkv_decode_f32", 72, (8, 8192), 8192, 8192, 1024, "float32",
                                  True, True),
    # a wider model: K 16384, 128 query heads and 8 key/value heads of 128 (170 MB of codes
    # and fp16 scales, larger than L2)
    "qkv_decode_wide": QkvWorkload("qkv_decode_wide", 73, (8, 16384), 16384, 16384, 1024,
                                   "float16"),
}


def make_qkv_inputs(wl: QkvWorkload, salt: int = 0) -> dict:
    """Draw every input tensor of one Q/K/V projection call for workload ``wl``."""
    fake = Workload(wl.name, wl.index, wl.input_shape, wl.K, 1, 1, 1, 4, 0, "relu")
    dt = np.float16 if wl.dtype == "float16" else np.float32

    def g(tid):
        return _rng(fake, tid, salt)

    out = dict(A=g(1).standard_normal(wl.input_shape, dtype=np.float32).astype(dt),
               norm_scale=g(2).uniform(0.5, 1.5, wl.K).astype(dt))
    for i, (name, n) in enumerate((("q", wl.Nq), ("k", wl.Nkv), ("v", wl.Nkv))):
        out[f"{name}_B"] = g(10 + i).integers(0, 256, (n, wl.kblocks, 16), dtype=np.uint8)
        out[f"{name}_scales"] = g(20 + i).uniform(0.002, 0.01, (n, wl.kblocks)).astype(dt)
    if wl.skip:
        out["skip"] = (g(3).standard_normal(wl.input_shape, dtype=np.float32) * 0.5).astype(dt)
    return out


# ---------------------------------------------------------------------------
# GroupedMatMul-29 on 16-bit operands.  input ~ U[-sqrt 3, sqrt 3] (unit
# variance); weights ~ U[-sqrt(3/K), sqrt(3/K)] (variance 1/K) so the outputs
# stay near unit scale in f16 (uniform rather than normal draws: a billion
# weights take seconds that way); group_indices int64: each row draws
# S distinct groups uniformly (the QMoE layer's k distinct experts per token).
# The prefill workload is the prefill layer's FC1 as a dense grouped product:
# 4096 tokens, k 2 of 8 experts, hidden 4096 -> 2 x 14336 (gate and linear).
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class GmmWorkload:
    name: str
    index: int
    M: int
    K: int
    G: int
    N: int
    S: int
    dtype: str = "float16"       # float16 | bfloat16 | float32 | float64

    @property
    def flops(self) -> int:
        return 2 * self.M * self.S * self.K * self.N


GMM_WORKLOADS = {
    "gmm_tiny": GmmWorkload("gmm_tiny", 80, 300, 128, 5, 200, 2),
    "gmm_prefill": GmmWorkload("gmm_prefill", 81, 4096, 4096, 8, 28672, 2),
    "gmm_prefill_bf16": GmmWorkload("gmm_prefill_bf16", 82, 4096, 4096, 8, 28672, 2,
                                    "bfloat16"),
    "gmm_prefill_f32": GmmWorkload("gmm_prefill_f32", 83, 4096, 4096, 8, 28672, 2, "float32"),
    "gmm_prefill_f64": GmmWorkload("gmm_prefill_f64", 84, 4096, 4096, 8, 28672, 2, "float64"),
}


def make_gmm_inputs(wl: GmmWorkload, salt: int = 0) -> dict:
    """Draw input [M, K], weights [G, K, N] (float32, to be cast to the workload's
    16-bit type by the caller) and group_indices [M, S] (int64) for ``wl``."""
    fake = Workload(wl.name, wl.index, (wl.M, wl.K), wl.K, 1, 1, 1, 4, 0, "relu")

    def g(tid):
        return _rng(fake, tid, salt)

    def uniform(tid, shape, half_width):
        a = g(tid).random(shape, dtype=np.float32)
        a *= np.float32(2.0 * half_width)
        a -= np.float32(half_width)
        return a

    x = uniform(1, (wl.M, wl.K), np.sqrt(3.0))
    w = uniform(2, (wl.G, wl.K, wl.N), np.sqrt(3.0 / wl.K))
    keys = g(3).random((wl.M, wl.G))
    idx = np.argsort(keys, axis=1, kind="stable")[:, :wl.S].astype(np.int64)
    return dict(input=x, weights=w, group_indices=idx)
