"""CPU oracle for the rotation-based W4A4 hot path (fp64, single-threaded C).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use this module;
the product library never does.  The C source ``rq_oracle.c`` shares no code with
the CUDA path and cites, per function, the page passage it follows.

``build()`` compiles ``rq_oracle.c`` with gcc into ``liboracle.so`` next to it.
Arrays are numpy; floating-point inputs are fp64 (exact widenings of the bf16 /
fp32 tensors the CUDA path reads).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

SIGNS_FIRST = 1  # flags bit 0, same meaning as the C oracle's RQO_SIGNS_FIRST

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (no fused multiply-add, so x86-64 and aarch64 agree)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    u64 = ctypes.c_uint64
    u32 = ctypes.c_uint32
    lib.rqo_splitmix64.restype = u64
    lib.rqo_splitmix64.argtypes = [u64, u64]
    lib.rqo_signs.restype = None
    lib.rqo_signs.argtypes = [u64, i64, P]
    lib.rqo_hadamard.restype = ctypes.c_int
    lib.rqo_hadamard.argtypes = [P, i64]
    lib.rqo_rotate_row.restype = ctypes.c_int
    lib.rqo_rotate_row.argtypes = [P, i64, P, u32, P]
    lib.rqo_quant_row.restype = None
    lib.rqo_quant_row.argtypes = [P, i64, P, P, P]
    lib.rqo_pack_row.restype = None
    lib.rqo_pack_row.argtypes = [P, i64, P]
    lib.rqo_unpack_row.restype = None
    lib.rqo_unpack_row.argtypes = [P, i64, P]
    lib.rqo_fwht_quant.restype = ctypes.c_int
    lib.rqo_fwht_quant.argtypes = [P, i64, i64, i64, u64, u32, P, P, P, P]
    lib.rqo_w4a4_gemm.restype = ctypes.c_int
    lib.rqo_w4a4_gemm.argtypes = [P, P, P, P, i64, i64, i64, P, P]
    lib.rqo_w4a4_gemm_entries.restype = ctypes.c_int
    lib.rqo_w4a4_gemm_entries.argtypes = [P, P, P, P, i64, i64, P, P, P, P]
    lib.rqo_kv_rotate_quant.restype = ctypes.c_int
    lib.rqo_kv_rotate_quant.argtypes = [P, P, i64, i64, i64, u64, u32, P, P, P, P]
    lib.rqo_quant_row8.restype = None
    lib.rqo_quant_row8.argtypes = [P, i64, P, P, P]
    lib.rqo_fwht_quant8.restype = ctypes.c_int
    lib.rqo_fwht_quant8.argtypes = [P, i64, i64, i64, u64, u32, P, P, P]
    lib.rqo_fwht_quant_groups.restype = ctypes.c_int
    lib.rqo_fwht_quant_groups.argtypes = [P, i64, i64, i64, u64, u32, i64, P, P, P]
    lib.rqo_w4a8_gemm.restype = ctypes.c_int
    lib.rqo_w4a8_gemm.argtypes = [P, P, P, P, i64, i64, i64, i64, P, P]
    lib.rqo_paley.restype = ctypes.c_int
    lib.rqo_paley.argtypes = [ctypes.c_int, P]
    lib.rqo_attn_decode.restype = ctypes.c_int
    lib.rqo_attn_decode.argtypes = [P, i64, i64, i64, P, P, P, P, i64, u64, u32, ctypes.c_double, ctypes.c_int, P]
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _check(st, what):
    if st == 2:
        raise OverflowError(f"{what}: an accumulator left the int32 range")
    if st != 0:
        raise ValueError(f"{what}: oracle status {st}")


def splitmix64(seed: int, i: int) -> int:
    return int(_load().rqo_splitmix64(seed, i))


def signs(seed: int, n: int) -> np.ndarray:
    s = np.empty(n, dtype=np.int8)
    _load().rqo_signs(seed, n, _ptr(s))
    return s


def hadamard(x) -> np.ndarray:
    """H_n applied to each row of x (last axis, length a power of two)."""
    y = _f64(x).copy()
    n = y.shape[-1]
    flat = y.reshape(-1, n)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        _check(lib.rqo_hadamard(_ptr(row), n), "hadamard")
        flat[r] = row
    return flat.reshape(y.shape)


def paley(m: int) -> np.ndarray:
    """The Hadamard block H_m (m in {12, 20, 28}) of rotations of size n = m 2^k."""
    H = np.empty((m, m), dtype=np.int8)
    _check(_load().rqo_paley(m, _ptr(H)), "paley")
    return H


def rotate(x, seed: int, flags: int) -> np.ndarray:
    """y = x R for each row of x, R the randomized Hadamard selected by flags."""
    xs = _f64(x)
    n = xs.shape[-1]
    flat = xs.reshape(-1, n)
    out = np.empty_like(flat)
    s = signs(seed, n)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        o = np.empty(n, dtype=np.float64)
        _check(lib.rqo_rotate_row(_ptr(row), n, _ptr(s), flags, _ptr(o)), "rotate")
        out[r] = o
    return out.reshape(xs.shape)


def quant_rows(y):
    """Per-row symmetric INT4: returns (codes int8, scales fp64, ratios y/scale)."""
    ys = _f64(y)
    n = ys.shape[-1]
    flat = ys.reshape(-1, n)
    codes = np.empty(flat.shape, dtype=np.int8)
    ratio = np.empty(flat.shape, dtype=np.float64)
    scales = np.empty(flat.shape[0], dtype=np.float64)
    lib = _load()
    sc = ctypes.c_double()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        c = np.empty(n, dtype=np.int8)
        rt = np.empty(n, dtype=np.float64)
        lib.rqo_quant_row(_ptr(row), n, _ptr(c), ctypes.byref(sc), _ptr(rt))
        codes[r], ratio[r], scales[r] = c, rt, sc.value
    return (codes.reshape(ys.shape), scales.reshape(ys.shape[:-1]), ratio.reshape(ys.shape))


def pack(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.int8))
    n = c.shape[-1]
    flat = c.reshape(-1, n)
    out = np.empty((flat.shape[0], n // 2), dtype=np.uint8)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        o = np.empty(n // 2, dtype=np.uint8)
        lib.rqo_pack_row(_ptr(row), n, _ptr(o))
        out[r] = o
    return out.reshape(c.shape[:-1] + (n // 2,))


def unpack(packed, n: int) -> np.ndarray:
    p = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    flat = p.reshape(-1, n // 2)
    out = np.empty((flat.shape[0], n), dtype=np.int8)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        o = np.empty(n, dtype=np.int8)
        lib.rqo_unpack_row(_ptr(row), n, _ptr(o))
        out[r] = o
    return out.reshape(p.shape[:-1] + (n,))


def fwht_quant(x, seed: int, flags: int, want_y: bool = False, want_ratio: bool = False):
    """Rows of x (rows x n): rotate, quantize, pack.

    Returns dict with q (rows x n/2 uint8), scales (rows fp32) and, on request,
    y (rows x n fp64) and ratio (rows x n, y/scale in fp64)."""
    xs = _f64(x)
    rows, n = xs.shape
    q = np.empty((rows, n // 2), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    y = np.empty((rows, n), dtype=np.float64) if want_y else None
    ratio = np.empty((rows, n), dtype=np.float64) if want_ratio else None
    st = _load().rqo_fwht_quant(_ptr(xs), rows, n, n, seed, flags, _ptr(q), _ptr(scales),
                                _ptr(y), _ptr(ratio))
    _check(st, "fwht_quant")
    out = {"q": q, "scales": scales}
    if want_y:
        out["y"] = y
    if want_ratio:
        out["ratio"] = ratio
    return out


def w4a4_gemm(aq, sa, wq, sw, M: int, N: int, K: int):
    """Returns (acc int64 M x N, y fp64 M x N)."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    acc = np.empty((M, N), dtype=np.int64)
    y = np.empty((M, N), dtype=np.float64)
    st = _load().rqo_w4a4_gemm(_ptr(aq), _ptr(sa), _ptr(wq), _ptr(sw), M, N, K, _ptr(acc), _ptr(y))
    _check(st, "w4a4_gemm")
    return acc, y


def w4a4_gemm_entries(aq, sa, wq, sw, K: int, ms, cs):
    """The products at positions (ms[e], cs[e]) only: returns (acc int64, y fp64)."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    cs = np.ascontiguousarray(cs, dtype=np.int64)
    acc = np.empty(ms.shape[0], dtype=np.int64)
    y = np.empty(ms.shape[0], dtype=np.float64)
    st = _load().rqo_w4a4_gemm_entries(_ptr(aq), _ptr(sa), _ptr(wq), _ptr(sw), K, ms.shape[0],
                                       _ptr(ms), _ptr(cs), _ptr(acc), _ptr(y))
    _check(st, "w4a4_gemm_entries")
    return acc, y


def kv_rotate_quant(k, v, seed: int, flags: int):
    """k, v: [tokens][heads][head_dim] (either may be None).

    Returns dict with kq/ks and vq/vs ([T][H][D/2] uint8, [T][H] fp32)."""
    ref = k if k is not None else v
    T, H, D = ref.shape
    kk = _f64(k) if k is not None else None
    vv = _f64(v) if v is not None else None
    kq = np.empty((T, H, D // 2), dtype=np.uint8) if k is not None else None
    ks = np.empty((T, H), dtype=np.float32) if k is not None else None
    vq = np.empty((T, H, D // 2), dtype=np.uint8) if v is not None else None
    vs = np.empty((T, H), dtype=np.float32) if v is not None else None
    st = _load().rqo_kv_rotate_quant(_ptr(kk), _ptr(vv), T, H, D, seed, flags, _ptr(kq), _ptr(ks),
                                     _ptr(vq), _ptr(vs))
    _check(st, "kv_rotate_quant")
    return {"kq": kq, "ks": ks, "vq": vq, "vs": vs}


def attn_decode(q, kq, ks, vq, vs, seed: int, flags: int, softmax_scale: float, rotated_out: bool = False):
    """Attention of query rows q [M][heads][head_dim] over the rotated INT4 cache
    (kq, vq [T][heads][head_dim/2] uint8; ks, vs [T][heads] fp32), in fp64.

    Returns out [M][heads][head_dim] fp64: o~ R^T, or o~ with rotated_out."""
    qq = _f64(q)
    M, H, D = qq.shape
    T = kq.shape[0]
    kq = np.ascontiguousarray(kq, dtype=np.uint8)
    vq = np.ascontiguousarray(vq, dtype=np.uint8)
    ks = np.ascontiguousarray(ks, dtype=np.float32)
    vs = np.ascontiguousarray(vs, dtype=np.float32)
    assert kq.shape == (T, H, D // 2) and vq.shape == (T, H, D // 2) and ks.shape == (T, H) and vs.shape == (T, H)
    out = np.empty((M, H, D), dtype=np.float64)
    st = _load().rqo_attn_decode(_ptr(qq), M, H, D, _ptr(kq), _ptr(ks), _ptr(vq), _ptr(vs), T, seed, flags,
                                 float(softmax_scale), 1 if rotated_out else 0, _ptr(out))
    _check(st, "attn_decode")
    return out


def quant_rows8(y):
    """Per-row symmetric INT8: returns (codes int8, scales fp64, ratios y/scale)."""
    ys = _f64(y)
    n = ys.shape[-1]
    flat = ys.reshape(-1, n)
    codes = np.empty(flat.shape, dtype=np.int8)
    ratio = np.empty(flat.shape, dtype=np.float64)
    scales = np.empty(flat.shape[0], dtype=np.float64)
    sc = ctypes.c_double()
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        c = np.empty(n, dtype=np.int8)
        rt = np.empty(n, dtype=np.float64)
        lib.rqo_quant_row8(_ptr(row), n, _ptr(c), ctypes.byref(sc), _ptr(rt))
        codes[r], ratio[r], scales[r] = c, rt, sc.value
    return codes.reshape(ys.shape), scales.reshape(ys.shape[:-1]), ratio.reshape(ys.shape)


def fwht_quant8(x, seed: int, flags: int, want_ratio: bool = False):
    """Rotation then per-row INT8: dict(q [rows][n] int8, scales fp32[, ratio])."""
    xs = _f64(x)
    rows, n = xs.shape
    q = np.empty((rows, n), dtype=np.int8)
    scales = np.empty(rows, dtype=np.float32)
    ratio = np.empty((rows, n), dtype=np.float64) if want_ratio else None
    _check(_load().rqo_fwht_quant8(_ptr(xs), rows, n, n, seed, flags, _ptr(q), _ptr(scales), _ptr(ratio)),
           "fwht_quant8")
    out = {"q": q, "scales": scales}
    if want_ratio:
        out["ratio"] = ratio
    return out


def fwht_quant_groups(x, seed: int, flags: int, group: int, want_ratio: bool = False):
    """Rotation then INT4 per group of `group` elements: dict(q [rows][n/2], scales
    [rows][n/group] fp32[, ratio])."""
    xs = _f64(x)
    rows, n = xs.shape
    q = np.empty((rows, n // 2), dtype=np.uint8)
    scales = np.empty((rows, n // group), dtype=np.float32)
    ratio = np.empty((rows, n), dtype=np.float64) if want_ratio else None
    _check(_load().rqo_fwht_quant_groups(_ptr(xs), rows, n, n, seed, flags, group, _ptr(q), _ptr(scales),
                                         _ptr(ratio)), "fwht_quant_groups")
    out = {"q": q, "scales": scales}
    if want_ratio:
        out["ratio"] = ratio
    return out


def w4a8_gemm(aq, sa, wq, sw, M: int, N: int, K: int, group: int):
    """INT8 activations x packed INT4 weights with per-group scales sw [N][K/group].
    Returns (acc int64 [M][N] (group == K only, else None), y fp64 [M][N])."""
    aq = np.ascontiguousarray(aq, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    acc = np.empty((M, N), dtype=np.int64) if group == K else None
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().rqo_w4a8_gemm(_ptr(aq), _ptr(sa), _ptr(wq), _ptr(sw), M, N, K, group, _ptr(acc), _ptr(y)),
           "w4a8_gemm")
    return acc, y


def tie_mask(ratio, window: float = 1e-4) -> np.ndarray:
    """Elements whose y/scale lies within `window` of a half-integer: there a
    code may legitimately differ by one between two correct implementations
    that decide the rounding in different precisions."""
    r = np.asarray(ratio, dtype=np.float64)
    return np.abs(r - np.floor(r) - 0.5) < window
