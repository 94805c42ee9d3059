"""GPU parity of the W4A8 path ([SQ] §The architecture, §End-to-end flow):
INT8 activation codes and per-group INT4 weight codes from rq_fwht_quant
(n = 4096, and the other powers of two from 256 to 8192), and rq_w4a8_gemm
with per-channel or per-group weight scales.

Bars: codes identical to the oracle's except in the tie window (a difference of
one allowed there), scales within 1e-5; the product on the oracle's codes:
int32 sums bit-exact (per-channel), fp32 within 1e-5 relative, fp16 within one
ulp.  The end-to-end decode case compares the GPU's output with the oracle's
computed entirely from the oracle's own codes, within the bound that the tie
window allows: per row, (codes in the tie window) x a_scale x 8 x w_scale.
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_codes, compare_f16, compare_scales, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
K4 = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _compare_int8(gpu_q, ref_q, ratio):
    g, r = gpu_q.astype(np.int16), ref_q.astype(np.int16)
    diff = g != r
    tie = oracle.tie_mask(ratio)
    bad = diff & ~(tie & (np.abs(g - r) == 1))
    assert not bad.any(), f"{int(bad.sum())} INT8 codes differ outside the tie window"


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_int8_activation_codes(dt, flags):
    x = synth.activations(21, K4, dt, 5, 4, 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, flags | rq.RQ_INT8_CODES)
    assert q.dtype == torch.int8 and q.shape == (21, K4)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, flags, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])


@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_group_weight_codes(flags):
    wt = synth.weights_t(37, K4, 7, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, flags | rq.RQ_GROUP_SCALES)
    assert s.shape == (37, K4 // 128)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, flags, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], K4)
    compare_scales(to_np(s), ref["scales"])


# ---- the two code modes at the other power-of-two row lengths ----

SIZES = [128, 256, 512, 1024, 2048, 8192]   # 128: the head-sized kernel


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_int8_codes_other_sizes(n, flags):
    x = synth.activations(13, n, torch.bfloat16, 40 + n % 97, max(1, n // 1000), 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, flags | rq.RQ_INT8_CODES)
    assert q.dtype == torch.int8 and q.shape == (13, n)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, flags, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_group_codes_other_sizes(n, flags):
    """Groups of 128: one per thread for n = 256, 512; from n = 1024 on four
    threads share a group and each thread touches four groups."""
    wt = synth.weights_t(19, n, 7 + n % 13, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, flags | rq.RQ_GROUP_SCALES)
    assert s.shape == (19, n // 128)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, flags, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], n)
    compare_scales(to_np(s), ref["scales"])


@pytest.mark.parametrize("dt", [torch.float32, torch.float16])
@pytest.mark.parametrize("mode", ["int8", "group"])
def test_code_modes_input_dtypes(dt, mode):
    n = 1024
    x = synth.activations(9, n, dt, 77, 2, 100.0)
    if mode == "int8":
        q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_INT8_CODES)
        ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
        _compare_int8(to_np(q), ref["q"], ref["ratio"])
    else:
        q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_GROUP_SCALES)
        ref = oracle.fwht_quant_groups(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, 128, want_ratio=True)
        compare_codes(to_np(q), ref["q"], ref["ratio"], n)
    compare_scales(to_np(s), ref["scales"])


def test_int8_codes_large_batch_8192():
    """1000 rows of 8192 (two warps per row, CTAs looping over row groups)."""
    x = synth.activations(1000, 8192, torch.bfloat16, 5, 8, 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_INT8_CODES)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])


def test_group_codes_large_fold_8192():
    """700 weight rows of 8192 (fp32): the per-group fold of a W4A8 layer with K = 8192."""
    wt = synth.weights_t(700, 8192, 11, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_GROUP_SCALES)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], 8192)
    compare_scales(to_np(s), ref["scales"])


def _random_operands(M, N, K, group, seed):
    g = np.random.default_rng(seed)
    qa = g.integers(-128, 128, size=(M, K)).astype(np.int8)
    qw = g.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    sa = (g.random(M) + 0.05).astype(np.float32)
    sw = (g.random((N, K // group) if group != K else N) + 0.05).astype(np.float32)
    return qa, sa, qw, sw


def _gpu(qa, sa, qw, sw, out_dtype):
    d = [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (qa, sa, qw, sw)]
    y = rq.w4a8_gemm(*d, out_dtype=out_dtype)
    assert rq.sync_status() == 0
    return to_np(y)


@pytest.mark.parametrize("M", [1, 5, 16, 17, 32, 33, 64])
@pytest.mark.parametrize("N,K", [(16, 128), (40, 512), (256, 4096)])
def test_product_per_channel(M, N, K):
    qa, sa, qw, sw = _random_operands(M, N, K, K, 1000 + M + N + K)
    acc, yref = oracle.w4a8_gemm(qa, sa, qw, sw.reshape(N, 1), M, N, K, K)
    np.testing.assert_array_equal(_gpu(qa, sa, qw, sw, torch.int32).astype(np.int64), acc)
    np.testing.assert_allclose(_gpu(qa, sa, qw, sw, torch.float32), yref, rtol=1e-5, atol=0)
    compare_f16(_gpu(qa, sa, qw, sw, torch.float16), yref)


@pytest.mark.parametrize("M", [1, 7, 16, 40, 65, 300])
@pytest.mark.parametrize("N,K", [(16, 128), (48, 1024), (128, 4096)])
def test_product_per_group(M, N, K):
    qa, sa, qw, sw = _random_operands(M, N, K, 128, 2000 + M + N + K)
    _, yref = oracle.w4a8_gemm(qa, sa, qw, sw, M, N, K, 128)
    y = _gpu(qa, sa, qw, sw, torch.float32)
    # fp32 sums of K/128 scaled group partials: relative to the row's magnitude
    err = np.abs(y - yref).max(axis=1)
    assert np.all(err <= 1e-5 * np.abs(yref).max(axis=1))
    compare_f16(_gpu(qa, sa, qw, sw, torch.float16), yref, atol=1e-5 * np.abs(yref).max(axis=1, keepdims=True))


def test_decode_workload_end_to_end():
    """16 tokens x 4096 -> 4096: INT8 activations and the product on the GPU,
    weights folded per group of 128 by the oracle (the offline step), against the
    oracle computed from its own codes."""
    w = synth.WORKLOADS["decode"]
    x = synth.activations(w.rows, w.n, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    wt = synth.weights_t(w.gemm_n, w.n, w.weight_seed, w.w_std)
    fold = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, 128)
    ref_a = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    _, yref = oracle.w4a8_gemm(ref_a["q"], ref_a["scales"], fold["q"], fold["scales"], w.rows, w.gemm_n, w.n, 128)
    qa, sa = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_INT8_CODES)
    y = to_np(rq.w4a8_gemm(qa, sa, torch.from_numpy(fold["q"]).to(DEV), torch.from_numpy(fold["scales"]).to(DEV),
                           out_dtype=torch.float32))
    ties = oracle.tie_mask(ref_a["ratio"]).sum(axis=1)            # per row
    bound = (ties[:, None] * ref_a["scales"].astype(np.float64)[:, None] * 8.0
             * fold["scales"].astype(np.float64).max(axis=1)[None, :])
    bound += 1e-5 * np.abs(yref).max(axis=1, keepdims=True)
    assert np.all(np.abs(y - yref) <= bound)


def test_int8_codes_prefill_batch():
    """2048 rows: the 512-thread CTAs of the n = 4096 kernel."""
    x = synth.activations(2048, K4, torch.bfloat16, 3, 4, 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_INT8_CODES)
    ref = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    _compare_int8(to_np(q), ref["q"], ref["ratio"])
    compare_scales(to_np(s), ref["scales"])


def test_group_codes_large_fold():
    """1300 weight rows (fp32): the 256-thread CTAs of the n = 4096 kernel."""
    wt = synth.weights_t(1300, K4, 9, 0.02)
    q, s = rq.fwht_quant(wt.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST | rq.RQ_GROUP_SCALES)
    ref = oracle.fwht_quant_groups(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, 128, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], K4)
    compare_scales(to_np(s), ref["scales"])


# ---- per-channel products of more than 64 tokens: the tensor-core kernel ----

@pytest.mark.parametrize("M", [65, 130, 257, 600])
@pytest.mark.parametrize("N,K", [(256, 128), (520, 1024), (1024, 4096)])
def test_product_tensor_cores(M, N, K):
    """CTA-pair tiles of 128 rows x 256 channels; ragged M (65 -> one half-empty
    tile, 600 -> 5 tiles) and ragged N (520 = 2 x 256 + 8)."""
    qa, sa, qw, sw = _random_operands(M, N, K, K, 3000 + M + N + K)
    acc, yref = oracle.w4a8_gemm(qa, sa, qw, sw.reshape(N, 1), M, N, K, K)
    np.testing.assert_array_equal(_gpu(qa, sa, qw, sw, torch.int32).astype(np.int64), acc)
    np.testing.assert_allclose(_gpu(qa, sa, qw, sw, torch.float32), yref, rtol=1e-5, atol=0)
    compare_f16(_gpu(qa, sa, qw, sw, torch.float16), yref)


def test_product_row_length_off_the_vector_width():
    """N = 100 fp16 outputs (200-byte rows) with 200 tokens: the mma.sync kernel."""
    M, N, K = 200, 100, 512
    qa, sa, qw, sw = _random_operands(M, N, K, K, 3999)
    acc, yref = oracle.w4a8_gemm(qa, sa, qw, sw.reshape(N, 1), M, N, K, K)
    compare_f16(_gpu(qa, sa, qw, sw, torch.float16), yref)
    np.testing.assert_array_equal(_gpu(qa, sa, qw, sw, torch.int32).astype(np.int64), acc)


def test_extreme_codes_at_max_k():
    """K = 65536 with constant rows and columns: every sum is K a w in closed
    form, up to 2^26 in magnitude; a = 127 against w = 7 drives both 4-bit
    accumulators to their largest value (225 K)."""
    M, N, K = 130, 256, 65536
    a_vals = np.array([-128, 127, -1, 0, 1, -7, 64, -65], dtype=np.int64)
    w_vals = np.array([-8, 7, -1, 0, 3, -5], dtype=np.int64)
    ar = a_vals[np.arange(M) % len(a_vals)]
    wc = w_vals[np.arange(N) % len(w_vals)]
    qa = np.repeat(ar.astype(np.int8)[:, None], K, axis=1)
    nib = (wc & 15).astype(np.uint8)
    qw = np.repeat((nib | (nib << 4))[:, None], K // 2, axis=1)
    sa = np.ones(M, dtype=np.float32)
    sw = np.ones(N, dtype=np.float32)
    y = _gpu(qa, sa, qw, sw, torch.int32).astype(np.int64)
    np.testing.assert_array_equal(y, K * ar[:, None] * wc[None, :])


def test_prefill_shape_sampled_rows():
    """2048 x 4096 -> 14336: INT8 codes of the prefill activations (from the
    oracle) against random INT4 weights; int32 sums and fp16 outputs of 27 rows,
    spread over every tile row and both CTAs of a pair, against the oracle."""
    w = synth.WORKLOADS["prefill"]
    M, K, N = w.rows, w.n, w.gemm_n
    x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    ref_a = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    qw, sw = synth.random_codes(N, K, 4001)
    qw, sw = qw.numpy(), sw.numpy()
    y32 = _gpu(ref_a["q"], ref_a["scales"], qw, sw, torch.int32)
    y16 = _gpu(ref_a["q"], ref_a["scales"], qw, sw, torch.float16)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [63, 64, 127, 128, M - 1]]))
    acc, yref = oracle.w4a8_gemm(ref_a["q"][rows], ref_a["scales"][rows], qw, sw.reshape(N, 1), len(rows), N, K, K)
    np.testing.assert_array_equal(y32[rows].astype(np.int64), acc)
    compare_f16(y16[rows], yref)


def test_product_operands_beyond_l2_sampled_rows():
    """4160 x 8192 -> 8192: 66 MB of operands, past the size up to which the
    tensor-core kernel runs four converter teams, so this case takes the
    three-team configuration.  int32 sums of 30 rows (every tile row and both
    CTAs of a pair) against the oracle."""
    M, N, K = 4160, 8192, 8192
    qa, sa, qw, sw = _random_operands(M, N, K, K, 4242)
    y32 = _gpu(qa, sa, qw, sw, torch.int32)
    rows = np.unique(np.concatenate([np.arange(0, M, 173), [127, 128, 255, 256, M - 1]]))
    acc, _ = oracle.w4a8_gemm(qa[rows], sa[rows], qw, sw.reshape(N, 1), len(rows), N, K, K)
    np.testing.assert_array_equal(y32[rows].astype(np.int64), acc)


# ---- per-group scales with more than 64 tokens: the tensor-core kernel ----

def _check_per_group(y, yref):
    err = np.abs(y.astype(np.float64) - yref).max(axis=1)
    assert np.all(err <= 1e-5 * np.abs(yref).max(axis=1)), float((err / np.abs(yref).max(axis=1)).max())


@pytest.mark.parametrize("M", [65, 130, 600])
@pytest.mark.parametrize("N,K", [(128, 128), (2560, 384), (384, 2048), (256, 8192)])
def test_product_per_group_tensor_cores(M, N, K):
    """N a multiple of 128 and K <= 8192: CTA pairs with 128 x 128 tiles, one
    TMEM partial per group; one group (K = 128) up to the 64 groups staged per
    column (K = 8192); ragged M.  The MMA issuer waits once per pair of K
    blocks: K = 128 and K = 384 leave a pair's last block without a partner,
    and at 600 x 2560 (100 tiles) pairs of blocks straddle two tiles."""
    qa, sa, qw, sw = _random_operands(M, N, K, 128, 5000 + M + N + K)
    _, yref = oracle.w4a8_gemm(qa, sa, qw, sw, M, N, K, 128)
    _check_per_group(_gpu(qa, sa, qw, sw, torch.float32), yref)
    compare_f16(_gpu(qa, sa, qw, sw, torch.float16), yref, atol=1e-5 * np.abs(yref).max(axis=1, keepdims=True))


def test_per_group_more_groups_than_staged():
    """K = 8320 (65 groups) is past the tensor-core kernel's staging: the mma.sync
    kernel takes it."""
    M, N, K = 100, 128, 8320
    qa, sa, qw, sw = _random_operands(M, N, K, 128, 5999)
    _, yref = oracle.w4a8_gemm(qa, sa, qw, sw, M, N, K, 128)
    _check_per_group(_gpu(qa, sa, qw, sw, torch.float32), yref)


def test_per_group_prefill_shape_sampled_rows():
    """2048 x 4096 -> 14336 with per-group weight scales: INT8 codes of the
    prefill activations (oracle) against random per-group INT4 weights; 27 rows
    over every tile row and both CTAs of a pair, fp32 and fp16, against the oracle."""
    w = synth.WORKLOADS["prefill"]
    M, K, N = w.rows, w.n, w.gemm_n
    x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    ref_a = oracle.fwht_quant8(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    g = np.random.default_rng(6001)
    qw = g.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    sw = (g.random((N, K // 128)) + 0.05).astype(np.float32)
    y32 = _gpu(ref_a["q"], ref_a["scales"], qw, sw, torch.float32)
    y16 = _gpu(ref_a["q"], ref_a["scales"], qw, sw, torch.float16)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [63, 64, 127, 128, M - 1]]))
    _, yref = oracle.w4a8_gemm(ref_a["q"][rows], ref_a["scales"][rows], qw, sw, len(rows), N, K, 128)
    _check_per_group(y32[rows], yref)
    compare_f16(y16[rows], yref, atol=1e-5 * np.abs(yref).max(axis=1, keepdims=True))


# ---------------------------------------------------------------------------
# W4A4 with per-group weight scales: INT4 activation codes one per byte
# (RQ_INT4_BYTES) into the W4A8 product.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [128, 256, 1024, 4096, 8192, 3072])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_int4_byte_codes(n, flags):
    """RQ_INT4_BYTES: the oracle's INT4 codes (tie window aside) and scales, one
    int8 byte per code, and exactly the GPU's own packed codes and scales."""
    x = synth.activations(37, n, torch.bfloat16, n + 9, 4, 100.0)
    xd = x.to(DEV)
    qb, sb = rq.fwht_quant(xd, 5, flags | rq.RQ_INT4_BYTES)
    qp, sp = rq.fwht_quant(xd, 5, flags)
    ref = oracle.fwht_quant(x.double().numpy(), 5, flags, want_ratio=True)
    g = to_np(qb).astype(np.int16)
    assert g.min() >= -8 and g.max() <= 7
    # the same codes as the packed form (decoded by bit arithmetic), the same scales
    b = to_np(qp).astype(np.int16)
    nib = np.stack([b & 15, b >> 4], axis=-1).reshape(37, n)
    np.testing.assert_array_equal(g, np.where(nib >= 8, nib - 16, nib))
    np.testing.assert_array_equal(to_np(sb), to_np(sp))
    _compare_int8(g, oracle.unpack(ref["q"], n), ref["ratio"].reshape(37, n))
    compare_scales(to_np(sb), ref["scales"])


@pytest.mark.parametrize("M,N,K", [(16, 256, 4096), (130, 384, 2048), (600, 256, 8192)])
def test_w4a4_per_group_product(M, N, K):
    """The W4A4 product with per-group weight scales on the oracle's codes: INT4
    activation codes as bytes, per-group INT4 weight codes, against the oracle's
    per-group product (fp32 sums of group partials: 1e-5 of each row's largest)."""
    x = synth.activations(M, K, torch.bfloat16, M + K, 4, 100.0)
    wt = synth.weights_t(N, K, 7 + N)
    ra = oracle.fwht_quant(x.double().numpy(), 5, rq.RQ_SIGNS_FIRST)
    rw = oracle.fwht_quant_groups(wt.double().numpy(), 5, rq.RQ_SIGNS_FIRST, 128)
    qa = oracle.unpack(ra["q"], K).astype(np.int8)
    _, yref = oracle.w4a8_gemm(qa, ra["scales"], rw["q"], rw["scales"], M, N, K, 128)
    _check_per_group(_gpu(qa, ra["scales"], rw["q"], rw["scales"], torch.float32), yref)
    # and the GPU's own INT4 bytes are those codes within the tie window
    qb, _ = rq.fwht_quant(x.to(DEV), 5, rq.RQ_SIGNS_FIRST | rq.RQ_INT4_BYTES)
    ra2 = oracle.fwht_quant(x.double().numpy(), 5, rq.RQ_SIGNS_FIRST, want_ratio=True)
    _compare_int8(to_np(qb).astype(np.int16), qa.astype(np.int16), ra2["ratio"].reshape(M, K))


# ---------------------------------------------------------------------------
# W4A4 with per-group weight scales on the tensor cores: operand-form INT4
# activations (RQ_E4M3_CODES) into rq_w4a4_gemm with [N][K/128] weight scales.
# ---------------------------------------------------------------------------

def _w4a4_group(qa_packed, sa, qw, sw, out_dtype):
    """The operand form of the packed activation codes (bit arithmetic on the
    host) and its (scale, code sum) pairs, through rq_w4a4_gemm's per-group path."""
    from parity import operand_form, operand_scales
    ae = torch.from_numpy(operand_form(qa_packed)).to(DEV)
    sa2 = torch.from_numpy(operand_scales(qa_packed, sa)).to(DEV)
    y = rq.w4a4_gemm(ae, sa2, torch.from_numpy(qw).to(DEV), torch.from_numpy(sw).to(DEV), out_dtype=out_dtype)
    assert rq.sync_status() == 0
    return to_np(y)


@pytest.mark.parametrize("M", [65, 300, 600])
@pytest.mark.parametrize("N,K", [(128, 128), (2560, 384), (384, 2048), (256, 8192)])
def test_w4a4_per_group_tensor_cores(M, N, K):
    """256-row tiles on CTA pairs: one group (K = 128) up to 64 groups, ragged M
    (65: one CTA of the pair without rows; 300, 600: partial tiles), odd group
    counts and, at 600 x 2560, pairs running several tiles; fp32 within 1e-5 of
    each row's largest output, fp16 within one ulp of that."""
    g = np.random.default_rng(7000 + M + N + K)
    qa = g.integers(0, 256, size=(M, K // 2)).astype(np.uint8)
    sa = (g.random(M) + 0.05).astype(np.float32)
    qw = g.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    sw = (g.random((N, K // 128)) + 0.05).astype(np.float32)
    codes = oracle.unpack(qa, K).astype(np.int8)
    _, yref = oracle.w4a8_gemm(codes, sa, qw, sw, M, N, K, 128)
    _check_per_group(_w4a4_group(qa, sa, qw, sw, torch.float32), yref)
    compare_f16(_w4a4_group(qa, sa, qw, sw, torch.float16), yref, atol=1e-5 * np.abs(yref).max(axis=1, keepdims=True))


@pytest.mark.parametrize("ba,bw", [(0x77, 0x77), (0x88, 0x88), (0x88, 0x77)])
def test_w4a4_per_group_extreme_codes(ba, bw):
    """All codes at +7 or -8 over 64 groups with unit scales: every output is
    64 x 128 x qa x qw exactly (fp32 sums of exact integers below 2^24)."""
    M, N, K = 256, 256, 8192
    qa = np.full((M, K // 2), ba, dtype=np.uint8)
    qw = np.full((N, K // 2), bw, dtype=np.uint8)
    y = _w4a4_group(qa, np.ones(M, np.float32), qw, np.ones((N, K // 128), np.float32), torch.float32)
    qa1, qw1 = (ba & 15) - 16 * ((ba >> 3) & 1), (bw & 15) - 16 * ((bw >> 3) & 1)
    assert (y == float(K * qa1 * qw1)).all()


def test_w4a4_per_group_end_to_end():
    """Rotation in operand form, then the per-group product, against the W4A8
    route on the GPU's own INT4 codes (RQ_INT4_BYTES): the same codes and scales,
    the same group partials; the two sum the scaled partials in different
    orders, so they agree within 1e-5 of each row's largest output."""
    M, N, K = 384, 1024, 4096
    x = synth.activations(M, K, torch.bfloat16, 11, 4, 100.0).to(DEV)
    wt = synth.weights_t(N, K, 13).to(DEV)
    qw, sw = rq.fwht_quant(wt, 7, rq.RQ_SIGNS_FIRST | rq.RQ_GROUP_SCALES)
    qe, se = rq.fwht_quant(x, 7, rq.RQ_SIGNS_FIRST | rq.RQ_E4M3_CODES)
    qb, sb = rq.fwht_quant(x, 7, rq.RQ_SIGNS_FIRST | rq.RQ_INT4_BYTES)
    y4 = to_np(rq.w4a4_gemm(qe, se, qw, sw, out_dtype=torch.float32))
    y8 = to_np(rq.w4a8_gemm(qb, sb, qw, sw, out_dtype=torch.float32))
    _check_per_group(y4, y8.astype(np.float64))


def test_w4a4_per_group_prefill_shape_sampled_rows():
    """2048 x 4096 -> 14336 with per-group weight scales on the prefill workload's
    activations: the oracle's INT4 codes in the operand form, random per-group
    weights; rows sampled over every 256-row tile and both CTAs of a pair,
    against the oracle's per-group product (fp32 and fp16)."""
    from parity import operand_form, operand_scales
    w = synth.WORKLOADS["prefill"]
    M, K, N = w.rows, w.n, w.gemm_n
    x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    ra = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    g = np.random.default_rng(6101)
    qw = g.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    sw = (g.random((N, K // 128)) + 0.05).astype(np.float32)
    ae = torch.from_numpy(operand_form(ra["q"])).to(DEV)
    sa2 = torch.from_numpy(operand_scales(ra["q"], ra["scales"])).to(DEV)
    wd, sd = torch.from_numpy(qw).to(DEV), torch.from_numpy(sw).to(DEV)
    y32 = to_np(rq.w4a4_gemm(ae, sa2, wd, sd, out_dtype=torch.float32))
    y16 = to_np(rq.w4a4_gemm(ae, sa2, wd, sd, out_dtype=torch.float16))
    assert rq.sync_status() == 0
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [127, 128, 255, 256, M - 1]]))
    codes = oracle.unpack(ra["q"][rows], K).astype(np.int8)
    _, yref = oracle.w4a8_gemm(codes, ra["scales"][rows], qw, sw, len(rows), N, K, 128)
    _check_per_group(y32[rows], yref)
    compare_f16(y16[rows], yref, atol=1e-5 * np.abs(yref).max(axis=1, keepdims=True))
