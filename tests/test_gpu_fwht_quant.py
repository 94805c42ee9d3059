"""GPU parity of rq_fwht_quant (online rotation + INT4 quant) against the oracle.

Sizes cover every supported n, several row groups with a ragged tail, strided
rows, all input dtypes, both rotation forms, degenerate rows, and the full-size
activation workloads (tiny 64x1024 fp32, decode 16x4096, prefill 2048x4096,
large 4096x8192) plus the offline weight fold on sampled output channels.
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_codes, compare_rows, compare_scales, record, to_np, unpack_codes

pytestmark = pytest.mark.gpu

DEV = "cuda"
DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run_and_compare(x_cpu: torch.Tensor, seed: int, flags: int, x_dev=None, with_err=False):
    """x_cpu: rows x n (the exact values the GPU reads).  Returns the number of
    tie-window code differences (and, with_err, the worst per-row error of y)."""
    rows, n = x_cpu.shape
    xd = x_cpu.to(DEV) if x_dev is None else x_dev
    q, s, y = rq.fwht_quant(xd, seed, flags, want_y=True)
    ref = oracle.fwht_quant(x_cpu.double().numpy(), seed, flags, want_y=True, want_ratio=True)
    err = compare_rows(to_np(y), ref["y"])
    compare_scales(to_np(s), ref["scales"])
    ties = compare_codes(to_np(q), ref["q"], ref["ratio"], n)
    return (ties, err) if with_err else ties


def _rows_for(n):
    # several row groups (a CTA takes 128 >> max(0, log2(n) - 7) rows) plus a ragged tail
    per_group = 128 >> max(0, int(np.log2(n)) - 7)
    return 3 * per_group + 5


@pytest.mark.parametrize("n", [32, 64, 128, 256, 512, 1024, 2048, 4096, 8192])
@pytest.mark.parametrize("dt", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_sizes_dtypes_flags(n, dt, flags):
    rows = _rows_for(n)
    x = synth.activations(rows, n, DTYPES[dt], seed=n + 3, n_outliers=max(1, n // 1000), factor=100.0)
    _run_and_compare(x, seed=0x5EED + n, flags=flags)


@pytest.mark.parametrize("n", [128, 4096, 8192])
def test_strided_rows(n):
    rows, pad = 37, 24
    full = synth.activations(rows, n + pad, torch.bfloat16, seed=5)
    xd = full.to(DEV)[:, :n]
    assert xd.stride(0) == n + pad
    _run_and_compare(full[:, :n].contiguous(), seed=9, flags=rq.RQ_SIGNS_FIRST, x_dev=xd)


@pytest.mark.parametrize("n", [128, 1024, 4096, 8192])
def test_degenerate_rows(n):
    x = torch.zeros(6, n, dtype=torch.float32)
    x[1, 3] = 100.0                   # single spike -> +-100/sqrt(n) everywhere, all codes +-7
    x[2, :] = 1.0                     # constant row -> a single nonzero coordinate
    x[3, n - 1] = -1e-30              # tiny but nonzero
    x[4, :] = torch.linspace(-1, 1, n)
    q, s, y = rq.fwht_quant(x.to(DEV), 3, rq.RQ_SIGNS_FIRST, want_y=True)
    qn, sn = to_np(q), to_np(s)
    assert sn[0] == 0.0 and sn[5] == 0.0 and not qn[0].any() and not qn[5].any()
    codes1 = unpack_codes(qn[1:2], n)[0]
    assert set(np.unique(np.abs(codes1)).tolist()) == {7}
    np.testing.assert_allclose(np.abs(to_np(y)[1]), 100.0 / np.sqrt(n), rtol=1e-6)
    _run_and_compare(x, seed=3, flags=rq.RQ_SIGNS_FIRST)


def test_zero_rows_is_a_no_op():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    q, s = rq.fwht_quant(x, 1, rq.RQ_SIGNS_FIRST)
    assert q.shape == (0, 128) and s.shape == (0,)


@pytest.mark.parametrize("rows", [1212, 1300, 4100, 8192])
def test_n4096_cta_sizes_for_batches(rows):
    """n = 4096 batches around the CTA-size choice on 152 SMs: 1212 rows (8-row
    CTAs, one round), 1300 and 4100 rows (7-row CTAs: fewer rows per SM in all),
    8192 rows (8-row CTAs again)."""
    x = synth.activations(rows, 4096, torch.bfloat16, seed=rows, n_outliers=4, factor=100.0)
    _run_and_compare(x, seed=0x5EED, flags=rq.RQ_SIGNS_FIRST)


@pytest.mark.parametrize("rows,dt", [(7, torch.bfloat16), (301, torch.bfloat16), (311, torch.float16),
                                     (611, torch.bfloat16), (613, torch.float32), (1517, torch.bfloat16)])
def test_n8192_rows_per_cta(rows, dt):
    """n = 8192 batches around the rows-per-CTA choice on 152 SMs (one row per
    CTA below 304 rows, two below 608, then four; fp32 input at most two), each
    with a ragged last group, for both rotation forms."""
    x = synth.activations(rows, 8192, dt, seed=rows, n_outliers=8, factor=100.0)
    for flags in (rq.RQ_SIGNS_FIRST, 0):
        _run_and_compare(x, seed=0x5EED, flags=flags)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_workload_activations_full_size(name):
    w = synth.WORKLOADS[name]
    x = synth.activations(w.rows, w.n, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    ties, err = _run_and_compare(x, synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, with_err=True)
    print(f"{name}: {ties} tie-window code differences out of {x.numel()}")
    record("fwht_workload", workload=name, rows=w.rows, n=w.n, codes=x.numel(), tie_window_differences=ties,
           max_row_rel_err=err, tolerance=1e-5)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_workload_weight_fold_sampled_channels(name):
    # The offline fold W~ = R^T W runs the same kernel over the rows of W^T; the
    # full W^T is rotated on the GPU and 64 sampled output channels (plus the
    # first and last) are checked against the oracle.
    w = synth.WORKLOADS[name]
    wt = synth.weights_t(w.gemm_n, w.n, w.weight_seed, w.w_std)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    rng = np.random.default_rng(w.data_seed)
    idx = np.unique(np.concatenate([[0, w.gemm_n - 1], rng.integers(0, w.gemm_n, 64)]))
    sub = wt[torch.from_numpy(idx)]
    ref = oracle.fwht_quant(sub.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    compare_scales(to_np(s)[idx], ref["scales"])
    compare_codes(to_np(q)[idx], ref["q"], ref["ratio"], w.n)


def test_repeatable_bitwise():
    x = synth.activations(300, 4096, torch.bfloat16, 1, 4, 100.0).to(DEV)
    a = rq.fwht_quant(x, 5, rq.RQ_SIGNS_FIRST, want_y=True)
    b = rq.fwht_quant(x, 5, rq.RQ_SIGNS_FIRST, want_y=True)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_output_guard_bands_untouched():
    # Outputs written into the middle of larger buffers: the margins keep their sentinel.
    rows, n = 77, 2048
    x = synth.activations(rows, n, torch.bfloat16, 2).to(DEV)
    qbuf = torch.full((rows + 4, n // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full((rows + 8,), -3.0, dtype=torch.float32, device=DEV)
    rq.fwht_quant(x, 5, rq.RQ_SIGNS_FIRST, q=qbuf[2:2 + rows], scales=sbuf[4:4 + rows])
    assert bool((qbuf[:2] == 0xA5).all()) and bool((qbuf[2 + rows:] == 0xA5).all())
    assert bool((sbuf[:4] == -3.0).all()) and bool((sbuf[4 + rows:] == -3.0).all())



@pytest.mark.parametrize("n", [128, 256, 1024, 2048, 4096, 8192])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_e4m3_operand_codes(n, dt, flags):
    """RQ_E4M3_CODES: the same codes and scales as the packed INT4 output, one
    operand byte per code (decoded here by bit arithmetic), each row's code sum
    beside its scale (exact), and the oracle's codes within the tie window (the
    oracle's row sums off by at most the row's tie-window differences)."""
    from parity import from_operand_form, unpack_codes
    rows = 77
    x = synth.activations(rows, n, dt, n + rows, 4, 100.0)
    xd = x.to(DEV)
    q_p, s_p = rq.fwht_quant(xd, 5, flags)
    q_e, s_e = rq.fwht_quant(xd, 5, flags | rq.RQ_E4M3_CODES)
    assert q_e.shape == (rows, n) and q_e.dtype == torch.uint8 and s_e.shape == (rows, 2)
    assert torch.equal(s_e[:, 0], s_p)
    codes_e = from_operand_form(to_np(q_e), n)
    assert np.array_equal(codes_e, unpack_codes(to_np(q_p), n))
    assert np.abs(codes_e).max() <= 8
    assert np.array_equal(to_np(s_e)[:, 1], codes_e.astype(np.int64).sum(axis=1).astype(np.float32))
    ref = oracle.fwht_quant(x.double().numpy(), 5, flags, want_ratio=True)
    compare_codes(oracle.pack(codes_e.astype(np.int8)), ref["q"], ref["ratio"], n)
    ref_codes = unpack_codes(ref["q"], n).astype(np.int64)
    per_row = np.abs(codes_e - ref_codes).sum(axis=1)
    assert (np.abs(to_np(s_e)[:, 1] - ref_codes.sum(axis=1)) <= per_row).all()


@pytest.mark.parametrize("n", [128, 4096, 8192])
def test_e4m3_row_sums_ragged_and_zero_rows(n):
    """Code sums at a ragged row count with zero rows and single spikes mixed in
    (sum 0 for a zero row; a spike's row holds +-7 everywhere)."""
    from parity import from_operand_form
    rows = 301
    x = synth.activations(rows, n, torch.bfloat16, n + 11, 4, 100.0)
    x[5] = 0
    x[6] = 0
    x[6, 17] = 3.0
    q, s = rq.fwht_quant(x.to(DEV), 9, rq.RQ_SIGNS_FIRST | rq.RQ_E4M3_CODES)
    codes = from_operand_form(to_np(q), n).astype(np.int64)
    sn = to_np(s)
    assert sn[5, 0] == 0.0 and sn[5, 1] == 0.0
    assert set(np.unique(np.abs(codes[6])).tolist()) == {7}
    assert np.array_equal(sn[:, 1], codes.sum(axis=1).astype(np.float32))
    ref = oracle.fwht_quant(x[6:7].double().numpy(), 9, rq.RQ_SIGNS_FIRST)
    assert sn[6, 1] == unpack_codes(ref["q"], n).sum()
