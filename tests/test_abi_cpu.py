"""Host-side checks of the C ABI: the library loads, exports every symbol that
include/rq.h declares, and rejects bad arguments before enqueuing anything
(these calls never touch a GPU)."""
import ctypes
import os
import re

import pytest
import torch

import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import build as rq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rq_build.build()
    return rq.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "rq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"rq_fwht_quant", "rq_w4a4_gemm", "rq_kv_rotate_quant"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.rq_status_string(0) == b"RQ_OK"
    assert lib.rq_status_string(3) == b"RQ_ERR_MISALIGNED"
    assert lib.rq_status_string(99) == b"RQ_ERR_UNKNOWN"
    assert lib.rq_version() >> 16 == 1


# Fake device addresses: validation must fail before anything dereferences them.
A16 = ctypes.c_void_p(0x10000)
A1 = ctypes.c_void_p(0x10001)
NULL = None


def fq(lib, x=A16, dtype=1, rows=4, n=128, ld=128, flags=1, q=A16, s=A16, y=NULL):
    return lib.rq_fwht_quant(x, dtype, rows, n, ld, 7, flags, q, s, y, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(rows=-1), 1),
    (dict(n=0), 1),
    (dict(n=48, ld=48), 2),          # not a power of two
    (dict(n=16, ld=16), 2),          # below the smallest size
    (dict(n=16384, ld=16384), 2),    # above the largest size
    (dict(n=12 * 16, ld=12 * 16), 2),        # 12 x 16: the power-of-two factor is below 32
    (dict(n=36 * 64, ld=36 * 64), 2),        # 36 is not one of the Hadamard blocks 12, 20, 28
    (dict(n=28 * 2048, ld=28 * 2048), 2),    # 28 x 2048: the power-of-two factor is above 1024
    (dict(n=28 * 512, ld=28 * 512, rows=0), 0),   # 14336 = 28 x 512: accepted
    (dict(n=12 * 256, ld=12 * 256, rows=0), 0),   # 3072 = 12 x 256: accepted
    (dict(n=20 * 1024, ld=20 * 1024 - 1, rows=0), 1),   # stride shorter than the row
    (dict(ld=64), 1),                # stride shorter than the row
    (dict(flags=2), 1),
    (dict(dtype=3), 2),              # int32 input
    (dict(x=NULL), 1),
    (dict(q=NULL), 1),
    (dict(x=A1), 3),
    (dict(y=A1), 3),
    (dict(ld=132), 3),               # 264-byte bf16 stride is not a multiple of 16
    (dict(rows=0, x=NULL), 0),       # empty: nothing to do
])
def test_fwht_quant_argument_checks(lib, kw, expect):
    assert fq(lib, **kw) == expect


def gemm(lib, M=16, N=64, K=256, a=A16, w=A16, sa=A16, sw=A16, y=A16, ydt=2, flags=0):
    return lib.rq_w4a4_gemm(a, sa, w, sw, M, N, K, 0, flags, y, ydt, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), 1),
    (dict(K=0), 1),
    (dict(K=200), 2),                 # not a multiple of 128
    (dict(K=131072), 2),
    (dict(flags=1), 1),
    (dict(flags=32), 1),
    (dict(flags=16), 2),              # operand-form activations feed the M > 64 kernel only
    (dict(flags=16, M=0, a=NULL), 0),  # empty: nothing to do
    (dict(flags=16, M=128, ydt=3, sa=NULL, sw=NULL), 1),   # operand form: the row code sums are read for int32 too
    (dict(flags=16, M=128, ydt=3, sa=A1, sw=NULL), 3),
    (dict(flags=8, M=128, N=128), 2),                     # per-group scales need operand-form activations
    (dict(flags=24, M=16, N=128), 2),                     # ... and more than 64 rows
    (dict(flags=24, M=128, N=128, ydt=3), 2),             # ... and fp16 / fp32 output
    (dict(flags=24, M=128, N=192), 2),                    # ... and N a multiple of 128
    (dict(flags=24, M=128, N=128, K=8320), 2),            # ... and at most 64 groups
    (dict(flags=24, M=0, N=128, a=NULL), 0),              # empty: nothing to do
    (dict(ydt=1), 2),                 # bf16 output not offered
    (dict(a=NULL), 1),
    (dict(sa=NULL), 1),
    (dict(w=A1), 3),
    (dict(N=4), 3),                   # 8-byte fp16 rows are not 16-byte multiples
    (dict(M=0, a=NULL), 0),
])
def test_gemm_argument_checks(lib, kw, expect):
    assert gemm(lib, **kw) == expect


def kv(lib, k=A16, v=A16, dtype=1, T=4, H=2, D=128, kq=A16, ks=A16, vq=A16, vs=A16):
    return lib.rq_kv_rotate_quant(k, v, dtype, T, H, D, 1, 1, kq, ks, vq, vs, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(T=-1), 1),
    (dict(H=0), 1),
    (dict(k=NULL, v=NULL), 1),
    (dict(D=96), 2),
    (dict(D=512), 2),
    (dict(kq=NULL), 1),
    (dict(vs=A1), 3),
    (dict(T=0), 0),
])
def test_kv_argument_checks(lib, kw, expect):
    assert kv(lib, **kw) == expect


def test_binding_raises_without_library(monkeypatch, tmp_path):
    from rotational_w4a4_quantization_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _binding.load_library()


def fused(lib, x=A16, dt=1, M=16, K=4096, ld=4096, flags=1, w=A16, ws=A16, N=4096, y=A16, ydt=2,
          aq=NULL, asc=NULL):
    return lib.rq_fwht_quant_gemm(x, dt, M, K, ld, 7, flags, w, ws, N, y, ydt, aq, asc, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), 1),
    (dict(K=0), 1),
    (dict(flags=2), 1),
    (dict(ld=4000), 1),               # stride shorter than the row
    (dict(dt=0), 2),                  # fp32 activations not offered by the fused path
    (dict(ydt=1), 2),                 # bf16 output not offered
    (dict(M=17), 2),                  # more than one m16 tile of tokens
    (dict(K=512, ld=512), 2),         # the fused rotation takes K = 1024, 2048, 4096, 8192
    (dict(K=3072, ld=3072), 2),
    (dict(K=16384, ld=16384), 2),
    (dict(N=4000), 2),                # N not a multiple of 128
    (dict(x=NULL), 1),
    (dict(ws=NULL), 1),
    (dict(y=A1), 3),
    (dict(aq=A1), 3),
    (dict(ld=4100), 3),               # 8200-byte stride is not a multiple of 16
    (dict(M=0, x=NULL), 0),           # empty: nothing to do
])
def test_fused_argument_checks(lib, kw, expect):
    assert fused(lib, **kw) == expect


def attn(lib, q=A16, dt=1, M=1, H=32, D=128, kq=A16, ks=A16, vq=A16, vs=A16, T=8192, flags=1, out=A16):
    return lib.rq_attn_decode(q, dt, M, H, D, kq, ks, vq, vs, T, 7, flags, 0.088, out, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), 1),
    (dict(T=-1), 1),
    (dict(flags=4), 1),               # unknown flag bit
    (dict(dt=3), 2),                  # int32 queries
    (dict(D=96), 2),
    (dict(D=512), 2),
    (dict(T=0), 1),                   # a softmax over no tokens
    (dict(kq=NULL), 1),
    (dict(out=NULL), 1),
    (dict(q=A1), 3),
    (dict(vq=A1), 3),
    (dict(ks=A1), 3),                 # scales need 4-byte alignment
    (dict(M=0, q=NULL), 0),           # empty: nothing to do
    (dict(H=0), 0),
])
def test_attn_argument_checks(lib, kw, expect):
    assert attn(lib, **kw) == expect


def w8(lib, a=A16, sa=A16, w=A16, sw=A16, M=16, N=4096, K=4096, group=128, y=A16, ydt=2):
    return lib.rq_w4a8_gemm(a, sa, w, sw, M, N, K, group, y, ydt, NULL)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), 1),
    (dict(K=0), 1),
    (dict(group=0), 1),
    (dict(K=4000), 2),                # K not a multiple of 128
    (dict(group=64), 2),              # groups of 128 or one per channel only
    (dict(ydt=3), 2),                 # raw int32 sums need per-channel scales
    (dict(ydt=1), 2),                 # bf16 output not offered
    (dict(a=NULL), 1),
    (dict(sw=NULL), 1),
    (dict(w=A1), 3),
    (dict(sa=A1), 3),                 # scales need 4-byte alignment
    (dict(M=0, a=NULL), 0),
    (dict(N=0), 0),
])
def test_w4a8_argument_checks(lib, kw, expect):
    assert w8(lib, **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(n=4096, ld=4096, flags=1 | 4, rows=0), 0),     # INT8 codes at n = 4096
    (dict(n=4096, ld=4096, flags=8, rows=0), 0),         # per-group scales at n = 4096
    (dict(n=2048, ld=2048, flags=4, rows=0), 0),         # INT8 codes at n = 2048
    (dict(n=256, ld=256, flags=8, rows=0), 0),           # per-group scales from n = 256 on
    (dict(n=128, ld=128, flags=4, rows=0), 0),           # n = 128: the head-sized kernel
    (dict(n=128, ld=128, flags=8, rows=0), 0),
    (dict(n=64, ld=64, flags=4, rows=0), 2),             # not below 128
    (dict(n=14336, ld=14336, flags=4, rows=0), 0),       # and for n = m 2^k (Paley blocks)
    (dict(n=12 * 32, ld=12 * 32, flags=8, rows=0), 0),
    (dict(n=4096, ld=4096, flags=4 | 8, rows=0), 1),     # one mode at a time
    (dict(n=4096, ld=4096, flags=64, rows=0), 1),        # unknown flag bit
    (dict(n=4096, ld=4096, flags=1 | 32, rows=0), 0),    # INT4 codes one per byte at n = 4096
    (dict(n=14336, ld=14336, flags=32, rows=0), 0),      # and for n = m 2^k
    (dict(n=128, ld=128, flags=32, rows=0), 0),          # n = 128 too
    (dict(n=32, ld=32, flags=32, rows=0), 2),            # not below 128
    (dict(n=4096, ld=4096, flags=4 | 32, rows=0), 1),    # one mode at a time
    (dict(n=8192, ld=8192, flags=1 | 16, rows=0), 0),    # E4M3 operand codes at n = 8192
    (dict(n=256, ld=256, flags=16, rows=0), 0),          # and from n = 256 on
    (dict(n=128, ld=128, flags=16, rows=0), 0),          # and at n = 128
    (dict(n=64, ld=64, flags=16, rows=0), 2),            # not below
    (dict(n=14336, ld=14336, flags=16, rows=0), 2),      # nor for n = m 2^k
    (dict(n=4096, ld=4096, flags=4 | 16, rows=0), 1),    # one mode at a time
])
def test_fwht_code_mode_checks(lib, kw, expect):
    assert fq(lib, **kw) == expect


@pytest.mark.parametrize("limit,expect", [(0, 1), (999, 1), (4_000_000_001, 1), (-5, 1)])
def test_selftest_limit_checks(lib, limit, expect):
    """The failure-detection self-test rejects limits outside 1000 .. 4e9 cycles
    before it launches anything."""
    lib.rq_selftest_wait_timeout.restype = ctypes.c_int32
    lib.rq_selftest_wait_timeout.argtypes = [ctypes.c_int64, ctypes.c_void_p]
    assert lib.rq_selftest_wait_timeout(limit, NULL) == expect


# --------------------------------------------------------------------------
# The Python binding checks every buffer the caller passes in (shape, dtype,
# contiguity) before it reaches the C side, which cannot size-check a pointer.
# These run on CPU tensors: the buffer checks come before the device check.
# --------------------------------------------------------------------------

def _t(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("kw,match", [
    (dict(q=("rows", "half", torch.uint8, -1)), "q: expected shape"),
    (dict(q=("rows", "half", torch.int8, 0)), "q: expected dtype"),
    (dict(scales=("rows+1", torch.float32)), "scales: expected shape"),
    (dict(scales=("rows", torch.float16)), "scales: expected dtype"),
    (dict(y=("rows", "n", torch.float16)), "y: expected dtype"),
])
def test_binding_checks_fwht_quant_buffers(lib, kw, match):
    rows, n = 8, 256
    x = _t((rows, n), torch.bfloat16)
    args = {}
    if "q" in kw:
        _, _, dt, extra = kw["q"]
        args["q"] = _t((rows, n // 2 + extra), dt)
    if "scales" in kw:
        r, dt = kw["scales"]
        args["scales"] = _t((rows + (1 if r == "rows+1" else 0),), dt)
    if "y" in kw:
        args["y"] = _t((rows, n), kw["y"][2])
    with pytest.raises(ValueError, match=match):
        rq.fwht_quant(x, 1, rq.RQ_SIGNS_FIRST, **args)


def test_binding_checks_fwht_quant_code_modes(lib):
    x = _t((4, 512), torch.bfloat16)
    with pytest.raises(ValueError, match="q: expected shape"):     # INT8 codes take n bytes per row
        rq.fwht_quant(x, 1, rq.RQ_INT8_CODES, q=_t((4, 256), torch.int8))
    with pytest.raises(ValueError, match="scales: expected shape"):  # one scale per group of 128
        rq.fwht_quant(x, 1, rq.RQ_GROUP_SCALES, scales=_t((4,), torch.float32))
    with pytest.raises(ValueError, match="scales: expected shape"):  # operand form: (scale, code sum) per row
        rq.fwht_quant(x, 1, rq.RQ_E4M3_CODES, scales=_t((4,), torch.float32))
    with pytest.raises(ValueError, match="q: expected shape"):       # operand form: n bytes per row
        rq.fwht_quant(x, 1, rq.RQ_E4M3_CODES, q=_t((4, 256), torch.uint8))
    with pytest.raises(ValueError, match="q must be contiguous"):
        rq.fwht_quant(x, 1, 1, q=_t((4, 512), torch.uint8)[:, ::2])


@pytest.mark.parametrize("which,bad,match", [
    ("a_scales", _t((15,), torch.float32), "a_scales: expected shape"),
    ("a_scales", _t((16,), torch.float16), "a_scales: expected dtype"),
    ("w_scales", _t((64, 2), torch.float32)[:, 0], "w_scales must be contiguous"),
    ("w_scales", None, "w_scales is required"),
    ("out", _t((16, 63), torch.float16), "out: expected shape"),
    ("out", _t((16, 64), torch.bfloat16), "out: expected dtype"),
])
def test_binding_checks_gemm_buffers(lib, which, bad, match):
    M, N, K = 16, 64, 256
    args = dict(a_q=_t((M, K // 2), torch.uint8), a_scales=_t((M,), torch.float32),
                w_q=_t((N, K // 2), torch.uint8), w_scales=_t((N,), torch.float32))
    out = None
    if which == "out":
        out = bad
    else:
        args[which] = bad
    with pytest.raises(ValueError, match=match):
        rq.w4a4_gemm(args["a_q"], args["a_scales"], args["w_q"], args["w_scales"], out=out)


@pytest.mark.parametrize("sa,match", [
    (_t((128,), torch.float32), "a_scales: expected shape"),   # operand form: (scale, code sum) per row
    (None, "a_scales is required"),                            # read for int32 output too
])
def test_binding_checks_operand_form_scales(lib, sa, match):
    M, N, K = 128, 64, 256
    with pytest.raises(ValueError, match=match):
        rq.w4a4_gemm(_t((M, K), torch.uint8), sa, _t((N, K // 2), torch.uint8), None, out=_t((M, N), torch.int32))


@pytest.mark.parametrize("a_cols,sw_shape,out_dtype,match", [
    (128, (64, 2), torch.float16, "per-group w_scales need the operand-form activations"),
    (256, (64, 2), torch.int32, "per-group scales give fp16 or fp32 output"),
    (256, (64, 3), torch.float16, "w_scales: expected shape"),
])
def test_binding_checks_per_group_product(lib, a_cols, sw_shape, out_dtype, match):
    M, N, K = 128, 64, 256
    with pytest.raises(ValueError, match=match):
        rq.w4a4_gemm(_t((M, a_cols), torch.uint8), _t((M, 2), torch.float32), _t((N, K // 2), torch.uint8),
                      _t(sw_shape, torch.float32), out=_t((M, N), out_dtype))


def test_binding_gemm_raw_mode_needs_no_scales(lib):
    # int32 accumulators do not read the scales: None passes the buffer checks
    # and stops at the device check (CPU tensors)
    with pytest.raises(ValueError, match="CUDA"):
        rq.w4a4_gemm(_t((16, 128), torch.uint8), None, _t((64, 128), torch.uint8), None,
                     out=_t((16, 64), torch.int32))


@pytest.mark.parametrize("key,shape,dtype,match", [
    ("kq", (4, 2, 63), torch.uint8, "out\\['kq'\\]: expected shape"),
    ("ks", (4, 2), torch.float64, "out\\['ks'\\]: expected dtype"),
    ("vq", (4, 2, 64), torch.int8, "out\\['vq'\\]: expected dtype"),
    ("vs", (4, 3), torch.float32, "out\\['vs'\\]: expected shape"),
])
def test_binding_checks_kv_buffers(lib, key, shape, dtype, match):
    T, H, D = 4, 2, 128
    k, v = _t((T, H, D), torch.bfloat16), _t((T, H, D), torch.bfloat16)
    out = {"kq": _t((T, H, D // 2), torch.uint8), "ks": _t((T, H), torch.float32),
           "vq": _t((T, H, D // 2), torch.uint8), "vs": _t((T, H), torch.float32)}
    out[key] = _t(shape, dtype)
    with pytest.raises(ValueError, match=match):
        rq.kv_rotate_quant(k, v, 1, out=out)
    del out["kq"]
    with pytest.raises(ValueError, match="is required"):
        rq.kv_rotate_quant(k, None if key.startswith("v") else v, 1, out=out)


@pytest.mark.parametrize("which,bad,match", [
    ("out", _t((4, 127), torch.float16), "out: expected shape"),
    ("a_q", _t((4, 2047), torch.uint8), "a_q: expected shape"),
    ("a_scales", _t((4,), torch.int32), "a_scales: expected dtype"),
    ("w_scales", _t((129,), torch.float32), "w_scales: expected shape"),
])
def test_binding_checks_fused_buffers(lib, which, bad, match):
    M, K, N = 4, 4096, 128
    kw = dict(out=None, a_q=None, a_scales=None)
    ws = _t((N,), torch.float32)
    if which == "w_scales":
        ws = bad
    else:
        kw[which] = bad
    with pytest.raises(ValueError, match=match):
        rq.fwht_quant_gemm(_t((M, K), torch.bfloat16), 1, 1, _t((N, K // 2), torch.uint8), ws, **kw)


def test_binding_checks_attn_and_w4a8_buffers(lib):
    M, H, D, T = 2, 4, 128, 16
    cache = {"kq": _t((T, H, D // 2), torch.uint8), "ks": _t((T, H), torch.float32),
             "vq": _t((T, H, D // 2), torch.uint8), "vs": _t((T, H), torch.float32)}
    with pytest.raises(ValueError, match="out: expected shape"):
        rq.attn_decode(_t((M, H, D), torch.bfloat16), cache, 1, out=_t((M, H, D - 1), torch.float32))
    Mw, N, K = 8, 256, 512
    aq, wq = _t((Mw, K), torch.int8), _t((N, K // 2), torch.uint8)
    with pytest.raises(ValueError, match="w_scales: expected shape"):      # per-group: (N, K/128)
        rq.w4a8_gemm(aq, _t((Mw,), torch.float32), wq, _t((N, K // 128 + 1), torch.float32))
    with pytest.raises(ValueError, match="a_scales: expected shape"):
        rq.w4a8_gemm(aq, _t((Mw + 1,), torch.float32), wq, _t((N,), torch.float32))
    with pytest.raises(ValueError, match="out: expected dtype"):
        rq.w4a8_gemm(aq, _t((Mw,), torch.float32), wq, _t((N,), torch.float32), out=_t((Mw, N), torch.int64))


@pytest.mark.parametrize("count,expect", [(0, 1), (-5, 1), ((1 << 30) + 1, 1)])
def test_probe_argument_checks(lib, count, expect):
    ctas = ctypes.c_int32(-1)
    assert lib.rq_probe_f8_mma(count, ctypes.byref(ctas), NULL) == expect
