"""GPU parity of rq_fwht_quant for row lengths n = m 2^k that are not powers of
two (m in {12, 20, 28}, Paley Hadamard blocks), against the oracle.

Same bar as the power-of-two sizes: rotated rows within 1e-5 of each row's
largest magnitude, scales within 1e-5, codes identical outside the tie window.
Cases: every block size with the smallest and largest power-of-two factor, the
FFN widths 14336 = 28 x 512 and 28672 = 28 x 1024, three input dtypes, both
sign sides, strided rows, degenerate rows, a prefill-sized batch of 14336-wide
activations, the fold of 14336-wide weight rows, and the two code modes of the
W4A8 layer (INT8 per row; INT4 per group of 128, groups spanning several
segments or lying inside one).
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_codes, compare_rows, compare_scales, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run_and_compare(x_cpu, seed, flags, x_dev=None):
    xd = x_cpu.to(DEV) if x_dev is None else x_dev
    q, s, y = rq.fwht_quant(xd, seed, flags, want_y=True)
    assert rq.sync_status() == 0
    ref = oracle.fwht_quant(x_cpu.double().numpy(), seed, flags, want_y=True, want_ratio=True)
    compare_rows(to_np(y), ref["y"])
    compare_scales(to_np(s), ref["scales"])
    return compare_codes(to_np(q), ref["q"], ref["ratio"], x_cpu.shape[1])


@pytest.mark.parametrize("m", [12, 20, 28])
@pytest.mark.parametrize("b", [32, 64, 256, 1024])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_block_sizes(m, b, flags):
    n = m * b
    x = synth.activations(7, n, torch.bfloat16, m + b, max(1, n // 1000), 100.0)
    _run_and_compare(x, synth.SIGN_SEED, flags)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("n", [28 * 512, 28 * 1024, 12 * 256])
def test_dtypes_and_ffn_widths(dt, n):
    x = synth.activations(5, n, dt, 31, max(1, n // 1000), 100.0)
    _run_and_compare(x, 0x1234, rq.RQ_SIGNS_FIRST)


def test_strided_rows():
    n = 20 * 128
    x = synth.activations(9, n, torch.bfloat16, 41, 3, 50.0)
    big = torch.zeros(9, n + 64, dtype=torch.bfloat16)
    big[:, :n] = x
    _run_and_compare(x, synth.SIGN_SEED, 0, x_dev=big.to(DEV)[:, :n])


def test_degenerate_rows():
    """A zero row (scale 0, codes 0), a single spike (every rotated value
    +-spike/sqrt(n)), a constant row."""
    n = 12 * 512
    x = torch.zeros(3, n, dtype=torch.float32)
    x[1, 77] = 1000.0
    x[2, :] = 0.25
    _run_and_compare(x, 9, rq.RQ_SIGNS_FIRST)
    _, s, y = rq.fwht_quant(x.to(DEV), 9, rq.RQ_SIGNS_FIRST, want_y=True)
    assert float(s[0]) == 0.0
    np.testing.assert_allclose(np.abs(to_np(y[1])), 1000.0 / np.sqrt(n), rtol=1e-6)


def test_prefill_batch_of_ffn_width():
    """2048 rows of 14336 (the down-projection input of the prefill layer's FFN)."""
    n = 14336
    x = synth.activations(2048, n, torch.bfloat16, 3, synth._n_outliers(n), 100.0)
    ties = _run_and_compare(x, synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    assert ties < 2048 * n * 1e-4


def test_weight_fold_of_width_14336():
    """The offline fold of weight rows of length K = 14336 (W^T of a down
    projection), sampled output channels, fp32 weights."""
    K = 14336
    wt = synth.weights_t(64, K, 105, 0.02)
    _run_and_compare(wt, synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)


def _compare_int8(gpu_q, ref_q, ratio):
    g, r = gpu_q.astype(np.int16), ref_q.astype(np.int16)
    bad = (g != r) & ~(oracle.tie_mask(ratio) & (np.abs(g - r) == 1))
    assert not bad.any(), f"{int(bad.sum())} INT8 codes differ outside the tie window"


@pytest.mark.parametrize("m", [12, 20, 28])
@pytest.mark.parametrize("b", [32, 1024])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_int8_codes(m, b, flags):
    """INT8 codes per row (the W4A8 activations) at n = m 2^k."""
    n = m * b
    x = synth.activations(6, n, torch.bfloat16, 3 * m + b, max(1, n // 1000), 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, flags | rq.RQ_INT8_CODES)
    assert q.dtype == torch.int8 and q.shape == (6, n)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, flags, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])


@pytest.mark.parametrize("m", [12, 20, 28])
@pytest.mark.parametrize("b", [32, 64, 512])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_group_codes(m, b, flags):
    """INT4 with one scale per 128 elements: groups span 4 (b = 32) or 2 (b = 64)
    segments, or lie inside one (b = 512)."""
    n = m * b
    wt = synth.weights_t(5, n, m + b, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, flags | rq.RQ_GROUP_SCALES)
    assert s.shape == (5, n // 128)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, flags, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], n)
    compare_scales(to_np(s), ref["scales"])


def test_w4a8_codes_of_width_14336():
    """The W4A8 down projection's inputs: 600 INT8 activation rows and 300
    per-group weight rows of width 14336 (fp16 activations, fp32 weights)."""
    n = 14336
    x = synth.activations(600, n, torch.float16, 8, synth._n_outliers(n), 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_INT8_CODES)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])
    wt = synth.weights_t(300, n, 12, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_GROUP_SCALES)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], n)
    compare_scales(to_np(s), ref["scales"])
