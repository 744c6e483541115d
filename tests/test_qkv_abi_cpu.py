"""Host-side checks of the Q/K/V projection C ABI (include/qkv.h) that need no GPU.

Defaults must equal the MatMulNBitsQkv manifest's attributes, and validation
(attributeConstraints, typeConstraints, derive.weightShapeOk, scaleShapeOk,
ioShapeOk, normContractOk) must reject bad calls before anything launches.
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


def test_qkv_exports(lib):
    for n in ("qkv_attrs_default", "qkv_workspace_size", "qkv_choose_path", "matmul_nbits_qkv"):
        assert n in q.declared_functions() and hasattr(lib, n)


def test_qkv_defaults_match_manifest(lib):
    a = b.QkvAttrs()
    lib.qkv_attrs_default(ctypes.byref(a))
    assert a.bits == 4 and a.accuracy_level == 0 and a.path == b.QKV_PATH_AUTO
    assert a.epsilon == pytest.approx(9.999999974752427e-7, rel=1e-7)
    assert a.K == 0 and a.Nq == 0 and a.Nkv == 0 and a.block_size == 0   # required
    assert ctypes.sizeof(b.QkvAttrs) == 48


def _call(attrs=None, K=256, Nq=128, Nkv=64, rows=4, a_shape=None, qb=None, ks=None, skip=True,
          residual=False, dtype=b.DT_F32, ws=1 << 30):
    attrs = attrs or q.make_qkv_attrs(K=K, Nq=Nq, Nkv=Nkv)
    kb = (K + 31) // 32
    a_shape = a_shape or (rows, K)
    qb = qb or (Nq, kb, 16)
    ks = ks or (Nkv, kb)
    fake = 0x1000  # never dereferenced: validation fails before any launch
    sh = b._shape
    return q.load().matmul_nbits_qkv(
        fake, sh(a_shape), len(a_shape), fake if skip else None, fake,
        fake, sh(qb), fake, sh((Nq, kb)), fake, sh((Nkv, kb, 16)), fake, sh(ks),
        fake, sh((Nkv, kb, 16)), fake, sh((Nkv, kb)), fake, fake, fake,
        fake if residual else None, dtype, ctypes.byref(attrs), 0x10000, ws, None)


def A(**kw):
    base = dict(K=256, Nq=128, Nkv=64)
    base.update(kw)
    return q.make_qkv_attrs(**base)


@pytest.mark.parametrize("attrs,call,status", [
    (A(bits=8), {}, b.ERR_NOT_SUPPORTED),
    (A(block_size=64), {}, b.ERR_NOT_SUPPORTED),
    (A(block_size=0), {}, b.ERR_INVALID_ARGUMENT),                 # required
    (A(accuracy_level=4), {}, b.ERR_NOT_SUPPORTED),
    (A(K=0), dict(K=0), b.ERR_INVALID_ARGUMENT),
    (A(Nq=0), {}, b.ERR_INVALID_ARGUMENT),
    (None, dict(dtype=b.DT_BF16), b.ERR_NOT_SUPPORTED),            # T1 float32/float16
    (None, dict(a_shape=(4, 255)), b.ERR_INVALID_ARGUMENT),        # last dim != K
    (None, dict(a_shape=(2, 2, 2, 256)), b.ERR_INVALID_ARGUMENT),  # rank 4
    (None, dict(qb=(128, 7, 16)), b.ERR_INVALID_ARGUMENT),         # kBlocks
    (None, dict(qb=(128, 8, 32)), b.ERR_INVALID_ARGUMENT),         # blobSize
    (None, dict(ks=(64, 9)), b.ERR_INVALID_ARGUMENT),              # scale shape
    (None, dict(skip=False, residual=True), b.ERR_INVALID_ARGUMENT),   # residual needs skip
    (None, dict(ws=16), b.ERR_WORKSPACE_TOO_SMALL),
    (A(path=b.QKV_PATH_DECODE), dict(K=200), b.ERR_NOT_SUPPORTED),   # K % 128
    (A(path=b.QKV_PATH_DECODE), dict(rows=17), b.ERR_NOT_SUPPORTED),
    (A(path=2), {}, b.ERR_INVALID_ARGUMENT),
])
def test_qkv_contract_rejections(lib, attrs, call, status):
    if attrs is not None and "K" in call:
        attrs.K = call["K"]
    assert _call(attrs, **call) == status


def test_qkv_workspace_and_path(lib):
    import torch
    a = A(K=8192, Nq=8192, Nkv=1024)
    n = q.qkv_workspace_size((8, 8192), a, torch.float16)
    assert n > 0 and n % 256 == 0
    assert q.qkv_choose_path((8, 8192), a, torch.float16) == b.QKV_PATH_DECODE
    assert q.qkv_choose_path((17, 8192), a, torch.float16) == b.QKV_PATH_GENERIC
    a200 = A(K=200)
    assert q.qkv_choose_path((4, 200), a200, torch.float32) == b.QKV_PATH_GENERIC
    # fp16 scales need 16-byte scale rows on the GEMV path: K a multiple of 256
    a384 = A(K=384)
    assert q.qkv_choose_path((4, 384), a384, torch.float32) == b.QKV_PATH_DECODE
    assert q.qkv_choose_path((4, 384), a384, torch.float16) == b.QKV_PATH_GENERIC


def _qkv_plan_bytes(rows, K, Nq, Nkv, sms=152):
    """The GEMV path's workspace, restated: the error word, the fp32 normalised rows
    (scalar-path fallback), the fp16 operand rows, fp32 partial sums for every slot
    of a shared row block and a 64-bit completion flag per slot and row block; each
    region rounded up to 256 bytes.  The flat (128-row block, 512-wide K chunk)
    range is cut into min(total, sms) equal pieces."""
    def up(x):
        return (max(x, 1) + 255) // 256 * 256
    N = (Nq, Nkv, Nkv)
    nkc = -(-K // 512)
    n_rb = sum(-(-n // 128) for n in N)
    total = n_rb * nkc
    G = max(1, min(total, sms))
    cta = lambda f: ((f + 1) * G - 1) // total
    splits = max(cta(rb * nkc + nkc - 1) - cta(rb * nkc) + 1 for rb in range(n_rb))
    off = 256
    off += up(4 * rows * K)
    off += up(2 * rows * K)
    off += up(4 * splits * rows * sum(N))
    off += up(8 * splits * n_rb)
    return off, splits


@pytest.mark.parametrize("rows,K,Nq,Nkv,splits", [
    (8, 8192, 8192, 1024, 3),      # 1280 chunks over 152 CTAs: 8-9 each, 16 per row block
    (4, 4096, 128, 64, 8),         # 24 chunks, one per CTA: eight CTAs share each row block
    (11, 2048, 200, 72, 4),        # 16 chunks: four CTAs a row block
    (16, 768, 256, 256, 2),
])
def test_qkv_workspace_covers_partials_and_flags(lib, rows, K, Nq, Nkv, splits):
    import torch
    a = A(K=K, Nq=Nq, Nkv=Nkv)
    assert q.qkv_choose_path((rows, K), a, torch.float16) == b.QKV_PATH_DECODE
    want, got_splits = _qkv_plan_bytes(rows, K, Nq, Nkv)
    assert got_splits == splits
    assert q.qkv_workspace_size((rows, K), a, torch.float16) == want
