"""Comparison helpers shared by the GPU parity tests (test infrastructure).

Tolerances (stated by the acceptance criteria of the hot path):
* rotated rows y: per-row relative error ||y - y_ref||_inf / ||y_ref||_inf <= 1e-5;
* scales: relative 1e-5 (the scale is max|y|/7, so it inherits the FWHT bound);
* INT4 codes: identical, except where the oracle's y/scale lies within 1e-4 of a
  half-integer; there the two sides may round differently (the GPU decides in
  fp32, the oracle in fp64) and a difference of exactly one is allowed and
  counted;
* GEMM: int32 accumulators bit-exact; fp32 dequantized output within 1e-5
  relative; fp16 output within one fp16 ulp of the exact value.
"""
from __future__ import annotations

import concurrent.futures as cf
import json
import os

import numpy as np
import torch

import oracle

Y_RTOL = 1e-5
SCALE_RTOL = 1e-5
TIE_WINDOW = 1e-4


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def to_dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def unpack_codes(packed: np.ndarray, n: int) -> np.ndarray:
    """Packed INT4 rows -> int16 codes by plain bit arithmetic (byte j: code 2j in
    the low nibble, 2j + 1 in the high one, two's complement).  The GPU's bytes are
    decoded here, not by the oracle, whose inputs never come from the GPU."""
    b = packed.reshape(-1, n // 2).astype(np.int16)
    nib = np.stack([b & 15, b >> 4], axis=-1).reshape(-1, n)
    return np.where(nib >= 8, nib - 16, nib)


def compare_codes(gpu_q: np.ndarray, ref_q: np.ndarray, ref_ratio: np.ndarray, n: int) -> int:
    """Assert code parity; return the number of tie-window differences."""
    g = unpack_codes(gpu_q, n)
    r = unpack_codes(ref_q, n)
    diff = g != r
    if not diff.any():
        return 0
    tie = oracle.tie_mask(ref_ratio.reshape(-1, n), TIE_WINDOW)
    bad = diff & ~(tie & (np.abs(g - r) == 1))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(int(i), int(j), int(g[i, j]), int(r[i, j]), float(ref_ratio.reshape(-1, n)[i, j]))
                  for i, j in idx]
        raise AssertionError(f"{int(bad.sum())} codes differ outside the tie window: {detail}")
    return int(diff.sum())


def compare_scales(gpu_s: np.ndarray, ref_s: np.ndarray):
    np.testing.assert_allclose(gpu_s.reshape(-1), ref_s.reshape(-1), rtol=SCALE_RTOL, atol=0)


def compare_rows(gpu_y: np.ndarray, ref_y: np.ndarray):
    g = gpu_y.astype(np.float64).reshape(ref_y.shape)
    num = np.abs(g - ref_y).max(axis=-1)
    den = np.abs(ref_y).max(axis=-1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    assert rel.max() <= Y_RTOL, f"rotated rows: max per-row relative error {rel.max():.3e}"
    return float(rel.max())


def compare_f16(gpu: np.ndarray, ref: np.ndarray, atol=0.0):
    """Within one fp16 ulp of the exact (fp64) value (plus `atol`, where the fp32
    value before the fp16 rounding carries its own bound, e.g. a sum of scaled
    group partials)."""
    g = gpu.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):   # beyond the fp16 range: handled below
        ref16 = ref.astype(np.float16)
        ulp = np.spacing(np.abs(ref16)).astype(np.float64)
    ok = np.abs(g - ref) <= ulp + atol
    # values beyond the fp16 range must saturate to inf with the right sign
    big = np.abs(ref) > 65504
    ok |= big & np.isinf(g) & (np.sign(g) == np.sign(ref))
    assert ok.all(), f"{int((~ok).sum())} fp16 outputs off by more than one ulp"


def host_threads() -> int:
    """Threads for oracle runs split over row blocks: every core this process may use."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_gemm_row_blocks(aq, sa, wq, sw, M: int, N: int, K: int, threads: int | None = None):
    """The oracle's whole W4A4 product, computed as disjoint row blocks on several
    host threads (the oracle is single-threaded C; ctypes releases the GIL while
    it runs, so the blocks run in parallel).  Yields (row0, acc int64, y fp64) per
    block, in row order; the union is exactly oracle.w4a4_gemm on all M rows."""
    threads = threads or host_threads()
    rows_per = max(1, -(-M // threads))
    bounds = [(r, min(M, r + rows_per)) for r in range(0, M, rows_per)]

    def run(b):
        r0, r1 = b
        acc, y = oracle.w4a4_gemm(aq[r0:r1], sa[r0:r1], wq, sw, r1 - r0, N, K)
        return r0, acc, y

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for out in ex.map(run, bounds):
            yield out


def record(name: str, **fields):
    """Append one JSON line to the file named by RQ_PARITY_RECORD (if set): the
    counts a run of the parity tests is asked to report (tie-window codes, worst
    per-row rotation error, host threads used by the oracle)."""
    path = os.environ.get("RQ_PARITY_RECORD")
    if not path:
        return
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps({"test": name, **fields}) + "\n")


def operand_form(packed: np.ndarray) -> np.ndarray:
    """Packed INT4 rows -> the W4A4 product's operand bytes (rq_fwht_quant with
    RQ_E4M3_CODES): one byte per code, q for q >= 0 and 0x80 | -q for q < 0, and
    within each group of 8 codes the order 0, 2, 4, 6, 1, 3, 5, 7.  Plain bit
    arithmetic on the bytes (test-side re-encoding of the oracle's codes)."""
    rows, half = packed.reshape(-1, packed.shape[-1]).shape
    b = packed.reshape(rows, half // 4, 4).astype(np.int16)
    nib = np.concatenate([b & 15, b >> 4], axis=-1)              # even codes, then odd codes
    byte = np.where(nib >= 8, 0x80 | (16 - nib), nib)
    return byte.astype(np.uint8).reshape(rows, 2 * half)


def operand_scales(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The (rows x 2) fp32 scales that go with operand_form(packed): each row's
    scale and the sum of its codes (rq_fwht_quant with RQ_E4M3_CODES)."""
    n = 2 * packed.shape[-1]
    sums = unpack_codes(packed, n).astype(np.int64).sum(axis=1)
    return np.stack([np.asarray(scales, np.float32).reshape(-1), sums.astype(np.float32)], axis=1)


def from_operand_form(e4: np.ndarray, n: int) -> np.ndarray:
    """Inverse of operand_form: operand bytes -> int16 codes in natural order."""
    b = e4.reshape(-1, n // 8, 8).astype(np.int16)
    q = np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
    out = np.empty_like(q)
    out[..., 0::2] = q[..., :4]
    out[..., 1::2] = q[..., 4:]
    return out.reshape(-1, n)
