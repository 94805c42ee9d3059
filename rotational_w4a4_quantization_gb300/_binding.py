"""ctypes binding of librq.so: argument marshalling only.

Each function checks that tensors live on the current CUDA device with the
expected dtype and contiguity, then passes raw device pointers, sizes and the
current stream to the C entry point of the same name.  All compute runs in the
library's kernels; a non-OK status raises :class:`RQError`.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librq.so")

RQ_SIGNS_FIRST = 1
RQ_ATTN_ROTATED_OUT = 2
RQ_INT8_CODES = 4
RQ_GROUP_SCALES = 8
RQ_E4M3_CODES = 16      # rq_fwht_quant: INT4 codes as the product's E4M3 operand bytes
RQ_INT4_BYTES = 32      # rq_fwht_quant: INT4 codes, one int8 byte each (the W4A8 product's A operand)
RQ_A_E4M3 = 16          # rq_w4a4_gemm: a_q holds those bytes

_STATUS = {0: "RQ_OK", 1: "RQ_ERR_INVALID_ARG", 2: "RQ_ERR_UNSUPPORTED", 3: "RQ_ERR_MISALIGNED",
           4: "RQ_ERR_CUDA", 5: "RQ_ERR_TIMEOUT"}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.int32: 3}

_lib = None


class RQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load librq.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"librq.so not found at {_LIB_PATH}: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i64, u64, u32, i32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                             ctypes.c_int)
    lib.rq_fwht_quant.restype = i32
    lib.rq_fwht_quant.argtypes = [P, i32, i64, i64, i64, u64, u32, P, P, P, P]
    lib.rq_w4a4_gemm.restype = i32
    lib.rq_w4a4_gemm.argtypes = [P, P, P, P, i64, i64, i64, u64, u32, P, i32, P]
    lib.rq_kv_rotate_quant.restype = i32
    lib.rq_kv_rotate_quant.argtypes = [P, P, i32, i64, i64, i64, u64, u32, P, P, P, P, P]
    lib.rq_fwht_quant_gemm.restype = i32
    lib.rq_fwht_quant_gemm.argtypes = [P, i32, i64, i64, i64, u64, u32, P, P, i64, P, i32, P, P, P]
    lib.rq_w4a8_gemm.restype = i32
    lib.rq_w4a8_gemm.argtypes = [P, P, P, P, i64, i64, i64, i64, P, i32, P]
    lib.rq_attn_decode.restype = i32
    lib.rq_attn_decode.argtypes = [P, i32, i64, i64, i64, P, P, P, P, i64, u64, u32, ctypes.c_float, P, P]
    lib.rq_sync_status.restype = i32
    lib.rq_sync_status.argtypes = [P]
    lib.rq_selftest_wait_timeout.restype = i32
    lib.rq_selftest_wait_timeout.argtypes = [i64, P]
    lib.rq_probe_f8_mma.restype = i32
    lib.rq_probe_f8_mma.argtypes = [i64, P, P]
    lib.rq_status_string.restype = ctypes.c_char_p
    lib.rq_status_string.argtypes = [i32]
    lib.rq_version.restype = u32
    lib.rq_version.argtypes = []
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, st):
    if st != 0:
        raise RQError(fn, st)


def _dev(*tensors):
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors must be on one device")
    return dev


def _expect(t, name: str, shape, dtypes, *, optional: bool = False):
    """Check a tensor the caller passes in (an output buffer, a scale vector):
    exact shape, dtype and contiguity, so that no kernel reads or writes past the
    end of a buffer the C side cannot size-check."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    dtypes = dtypes if isinstance(dtypes, (tuple, list)) else (dtypes,)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: expected dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_OUT_DTYPES = (torch.float16, torch.float32, torch.int32)


def fwht_quant(x: torch.Tensor, seed: int, flags: int = RQ_SIGNS_FIRST, *, q=None, scales=None,
               y=None, want_y: bool = False, stream=None):
    """Rotate each row of ``x`` (rows x n; row stride may exceed n) by the
    randomized Hadamard R and quantize it to packed INT4.

    Returns ``(q, scales)`` or ``(q, scales, y)`` when ``want_y``: q is
    (rows x n/2) uint8, scales (rows,) fp32, y (rows x n) fp32 = x R.  With
    RQ_INT8_CODES in flags q is (rows x n) int8; with RQ_GROUP_SCALES scales is
    (rows x n/128); with RQ_E4M3_CODES q is (rows x n) uint8, the same INT4 codes
    as the product's operand bytes (see include/rq.h), and scales (rows x 2)
    holds each row's scale and code sum; with RQ_INT4_BYTES q is
    (rows x n) int8, the INT4 codes one per byte (for w4a8_gemm: a W4A4 product
    with per-group weight scales)."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit stride in the last dimension")
    if x.dtype not in (torch.float32, torch.bfloat16, torch.float16):
        raise ValueError("x must be float32, bfloat16 or float16")
    rows, n = x.shape
    if flags & (RQ_INT8_CODES | RQ_INT4_BYTES):
        q_shape, q_dtype = (rows, n), torch.int8
    elif flags & RQ_E4M3_CODES:
        q_shape, q_dtype = (rows, n), torch.uint8
    else:
        q_shape, q_dtype = (rows, n // 2), torch.uint8
    s_shape = (rows, n // 128) if flags & RQ_GROUP_SCALES else ((rows, 2) if flags & RQ_E4M3_CODES else (rows,))
    if q is None:
        q = torch.empty(q_shape, dtype=q_dtype, device=x.device)
    if scales is None:
        scales = torch.empty(s_shape, dtype=torch.float32, device=x.device)
    if want_y and y is None:
        y = torch.empty(rows, n, dtype=torch.float32, device=x.device)
    _expect(q, "q", q_shape, q_dtype)
    _expect(scales, "scales", s_shape, torch.float32)
    _expect(y, "y", (rows, n), torch.float32, optional=True)
    _dev(x, q, scales, y)
    with torch.cuda.device(x.device):
        st = lib.rq_fwht_quant(_ptr(x), _DTYPES[x.dtype], rows, n, x.stride(0), seed, flags,
                               _ptr(q), _ptr(scales), _ptr(y), _stream(stream))
    _check("rq_fwht_quant", st)
    return (q, scales, y) if y is not None else (q, scales)


def w4a4_gemm(a_q: torch.Tensor, a_scales, w_q: torch.Tensor, w_scales, *, out_dtype=torch.float16,
              seed: int = 0, out=None, stream=None):
    """y = dequant(Q(XR) . Q(R^T W)): a_q (M x K/2), w_q (N x K/2) packed codes,
    a_scales (M,), w_scales (N,).  out_dtype float16 / float32, or int32 for the
    raw accumulators.  a_q of shape (M x K) holds the activation codes in the
    operand form of fwht_quant(..., RQ_E4M3_CODES) (more than 64 rows); a_scales
    is then the (M x 2) scales-and-code-sums it returns, needed for int32 too.
    With operand-form activations, w_scales of shape (N x K/128) are per-group
    weight scales (fwht_quant(..., RQ_GROUP_SCALES) on the rows of W^T): fp16
    or fp32 output, N a multiple of 128, K <= 8192."""
    lib = load_library()
    M, ka = a_q.shape
    N, kb2 = w_q.shape
    if a_q.dtype != torch.uint8 or w_q.dtype != torch.uint8 or ka not in (kb2, 2 * kb2):
        raise ValueError("a_q (M x K/2, or M x K operand bytes) and w_q (N x K/2) must be uint8")
    if not (a_q.is_contiguous() and w_q.is_contiguous()):
        raise ValueError("packed operands must be contiguous")
    K = 2 * kb2
    flags = RQ_A_E4M3 if ka == K else 0
    if isinstance(w_scales, torch.Tensor) and w_scales.dim() == 2:
        if not flags:
            raise ValueError("per-group w_scales need the operand-form activations (a_q of shape M x K)")
        flags |= RQ_GROUP_SCALES
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=a_q.device)
    _expect(out, "out", (M, N), _OUT_DTYPES)
    raw = out.dtype == torch.int32       # raw accumulators: the scales are not read
    if flags & RQ_A_E4M3:
        _expect(a_scales, "a_scales", (M, 2), torch.float32)   # (scale, code sum) per row
    else:
        _expect(a_scales, "a_scales", (M,), torch.float32, optional=raw)
    if flags & RQ_GROUP_SCALES:
        if raw:
            raise ValueError("per-group scales give fp16 or fp32 output, not raw int32 accumulators")
        _expect(w_scales, "w_scales", (N, K // 128), torch.float32)
    else:
        _expect(w_scales, "w_scales", (N,), torch.float32, optional=raw)
    _dev(a_q, w_q, a_scales, w_scales, out)
    with torch.cuda.device(a_q.device):
        st = lib.rq_w4a4_gemm(_ptr(a_q), _ptr(a_scales), _ptr(w_q), _ptr(w_scales), M, N, K, seed, flags,
                              _ptr(out), _DTYPES[out.dtype], _stream(stream))
    _check("rq_w4a4_gemm", st)
    return out


def kv_rotate_quant(k, v, seed: int, flags: int = RQ_SIGNS_FIRST, *, out=None, stream=None):
    """K, V ([tokens][heads][head_dim], contiguous; either may be None) ->
    dict(kq, ks, vq, vs): packed codes [T][H][D/2] uint8 and scales [T][H] fp32."""
    lib = load_library()
    ref = k if k is not None else v
    if ref is None:
        raise ValueError("k and v cannot both be None")
    T, H, D = ref.shape
    for t in (k, v):
        if t is not None and (t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous()):
            raise ValueError("k and v must be contiguous with the same shape and dtype")
    if out is None:
        out = {}
        if k is not None:
            out["kq"] = torch.empty(T, H, D // 2, dtype=torch.uint8, device=ref.device)
            out["ks"] = torch.empty(T, H, dtype=torch.float32, device=ref.device)
        if v is not None:
            out["vq"] = torch.empty(T, H, D // 2, dtype=torch.uint8, device=ref.device)
            out["vs"] = torch.empty(T, H, dtype=torch.float32, device=ref.device)
    for src, qk, sk in ((k, "kq", "ks"), (v, "vq", "vs")):
        if src is not None:
            _expect(out.get(qk), f"out[{qk!r}]", (T, H, D // 2), torch.uint8)
            _expect(out.get(sk), f"out[{sk!r}]", (T, H), torch.float32)
    _dev(k, v, *out.values())
    with torch.cuda.device(ref.device):
        st = lib.rq_kv_rotate_quant(_ptr(k), _ptr(v), _DTYPES[ref.dtype], T, H, D, seed, flags,
                                    _ptr(out.get("kq")), _ptr(out.get("ks")), _ptr(out.get("vq")),
                                    _ptr(out.get("vs")), _stream(stream))
    _check("rq_kv_rotate_quant", st)
    return out


def fwht_quant_gemm(x: torch.Tensor, seed: int, flags: int, w_q: torch.Tensor, w_scales, *,
                    out_dtype=torch.float16, out=None, a_q=None, a_scales=None, stream=None):
    """Decode-sized fusion of :func:`fwht_quant` and :func:`w4a4_gemm`: x (M x K,
    bf16/fp16, unit stride in the last dimension; M <= 16, K = 1024, 2048, 4096 or
    8192) is rotated,
    quantized and multiplied by w_q (N x K/2 packed codes, N a multiple of 128)
    in one launch.  Returns y (M x N, out_dtype float16 / float32 / int32 raw
    accumulators); a_q (M x K/2) and a_scales (M,), when given, receive the
    activation codes and scales."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit stride in the last dimension")
    M, K = x.shape
    N, kb = w_q.shape
    if kb * 2 != K or w_q.dtype != torch.uint8 or not w_q.is_contiguous():
        raise ValueError("w_q must be contiguous uint8 with K/2 columns")
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be bfloat16 or float16")
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _expect(out, "out", (M, N), _OUT_DTYPES)
    _expect(w_scales, "w_scales", (N,), torch.float32, optional=out.dtype == torch.int32)
    _expect(a_q, "a_q", (M, K // 2), torch.uint8, optional=True)
    _expect(a_scales, "a_scales", (M,), torch.float32, optional=True)
    _dev(x, w_q, w_scales, out, a_q, a_scales)
    with torch.cuda.device(x.device):
        st = lib.rq_fwht_quant_gemm(_ptr(x), _DTYPES[x.dtype], M, K, x.stride(0), seed, flags, _ptr(w_q),
                                    _ptr(w_scales), N, _ptr(out), _DTYPES[out.dtype], _ptr(a_q), _ptr(a_scales),
                                    _stream(stream))
    _check("rq_fwht_quant_gemm", st)
    return out


def attn_decode(q: torch.Tensor, cache: dict, seed: int, flags: int = RQ_SIGNS_FIRST, softmax_scale=None, *,
                out=None, stream=None):
    """Attention of query rows q ([M][heads][head_dim], contiguous fp32/bf16/fp16)
    over the rotated INT4 cache that :func:`kv_rotate_quant` wrote (a dict with kq,
    ks, vq, vs).  Returns out [M][heads][head_dim] fp32: (sum_t p_t v^_t) R^T, or the
    rotated sum with RQ_ATTN_ROTATED_OUT in flags.  softmax_scale defaults to
    1/sqrt(head_dim)."""
    lib = load_library()
    if q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be a contiguous [M][heads][head_dim] tensor")
    M, H, D = q.shape
    kq, ks, vq, vs = cache["kq"], cache["ks"], cache["vq"], cache["vs"]
    T = kq.shape[0]
    for t, shape, dt in ((kq, (T, H, D // 2), torch.uint8), (vq, (T, H, D // 2), torch.uint8),
                         (ks, (T, H), torch.float32), (vs, (T, H), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous():
            raise ValueError("cache tensors must be contiguous with the kv_rotate_quant layout")
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if q.dtype not in (torch.float32, torch.bfloat16, torch.float16):
        raise ValueError("q must be float32, bfloat16 or float16")
    if out is None:
        out = torch.empty(M, H, D, dtype=torch.float32, device=q.device)
    _expect(out, "out", (M, H, D), torch.float32)
    _dev(q, kq, ks, vq, vs, out)
    with torch.cuda.device(q.device):
        st = lib.rq_attn_decode(_ptr(q), _DTYPES[q.dtype], M, H, D, _ptr(kq), _ptr(ks), _ptr(vq), _ptr(vs), T,
                                seed, flags, float(softmax_scale), _ptr(out), _stream(stream))
    _check("rq_attn_decode", st)
    return out


def w4a8_gemm(a_q: torch.Tensor, a_scales, w_q: torch.Tensor, w_scales, *, out_dtype=torch.float16, out=None,
              stream=None):
    """a_q (M x K int8) x w_q (N x K/2 packed INT4): y (M x N).  w_scales of shape (N,)
    are per channel, (N, K/128) per group of 128; out_dtype float16 / float32, or
    int32 (raw exact sums, per-channel scales only)."""
    lib = load_library()
    M, K = a_q.shape
    N, kb = w_q.shape
    if kb * 2 != K or a_q.dtype != torch.int8 or w_q.dtype != torch.uint8:
        raise ValueError("a_q must be int8 (M x K), w_q uint8 (N x K/2)")
    if not (a_q.is_contiguous() and w_q.is_contiguous()):
        raise ValueError("a_q and w_q must be contiguous")
    per_group = w_scales is not None and w_scales.dim() == 2 and w_scales.shape[1] != 1
    group = 128 if per_group else K
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=a_q.device)
    _expect(out, "out", (M, N), _OUT_DTYPES)
    raw = out.dtype == torch.int32
    _expect(a_scales, "a_scales", (M,), torch.float32, optional=raw)
    sw_shape = (N, K // 128) if per_group else ((N, 1) if w_scales is not None and w_scales.dim() == 2 else (N,))
    _expect(w_scales, "w_scales", sw_shape, torch.float32, optional=raw)
    _dev(a_q, a_scales, w_q, w_scales, out)
    with torch.cuda.device(a_q.device):
        st = lib.rq_w4a8_gemm(_ptr(a_q), _ptr(a_scales), _ptr(w_q), _ptr(w_scales), M, N, K, group, _ptr(out),
                              _DTYPES[out.dtype], _stream(stream))
    _check("rq_w4a8_gemm", st)
    return out


def sync_status(stream=None) -> int:
    """Drain the stream and return the library's status word (0 = OK)."""
    return int(load_library().rq_sync_status(_stream(stream)))


def selftest_wait_timeout(limit_cycles: int, stream=None) -> None:
    """Launch the failure-detection self-test: a bounded device wait on a barrier
    that nothing arrives on.  The next :func:`sync_status` returns RQ_ERR_TIMEOUT."""
    _check("rq_selftest_wait_timeout", load_library().rq_selftest_wait_timeout(int(limit_cycles), _stream(stream)))


def probe_f8_mma(mmas_per_sm: int, stream=None) -> int:
    """Enqueue the tensor-pipe probe (back-to-back M128 N256 K32 FP8 MMAs, one CTA
    per SM); returns the number of CTAs.  Each MMA is 2,097,152 operations."""
    ctas = ctypes.c_int32(0)
    _check("rq_probe_f8_mma", load_library().rq_probe_f8_mma(int(mmas_per_sm), ctypes.byref(ctas), _stream(stream)))
    return int(ctas.value)
