"""GPU parity of rq_fwht_quant_gemm, the decode-sized fusion of the rotation,
INT4 quantization and W4A4 product, against the oracle and against the unfused
entry points.

The fused kernel forms the activation codes on chip and multiplies them in the
same launch.  It must produce what rq_fwht_quant followed by rq_w4a4_gemm
produce, bit for bit (the same arithmetic in the same order), and that must
match the oracle, which computes everything from its own codes: codes within
the tie window, scales within 1e-5, and the product within what the tie window
allows.  A code there may differ by one and |q_w| <= 8, so a row's int32 sums
may differ by 8 x (its codes in the tie window); they are exact when it has
none.  The fp32 and fp16 outputs get the same bound, scaled, plus 1e-5 relative
(one fp16 ulp for fp16).  Shapes cover M = 1..16 (rows missing from some cluster
ranks), several N (cluster counts), both input dtypes, both sign forms and every
output mode, for every row length the fused kernel takes (K = 1024, 2048, 4096,
8192: clusters of 1 to 8 CTAs, one or several rotated rows per CTA).
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
KS = [1024, 2048, 4096, 8192]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _tie_bound(ref, wq_np, sw_np):
    """Per-output bounds from the oracle's tie-window codes: integer sums and the
    dequantized value."""
    ties = oracle.tie_mask(ref["ratio"]).sum(axis=1).astype(np.int64)          # per row
    ibound = 8 * ties[:, None]
    fbound = ibound * ref["scales"].astype(np.float64)[:, None] * sw_np.astype(np.float64)[None, :]
    return ibound, fbound


def _inputs(M, N, dt, seed, K=4096):
    x = synth.activations(M, K, dt, seed, 4, 100.0)
    wq, sw = synth.random_codes(N, K, seed + 50)
    return x, wq, sw


def _fused(x, flags, wq, sw, out_dtype):
    M, K = x.shape
    aq = torch.empty(M, K // 2, dtype=torch.uint8, device=DEV)
    asc = torch.empty(M, dtype=torch.float32, device=DEV)
    y = rq.fwht_quant_gemm(x.to(DEV), synth.SIGN_SEED, flags, wq.to(DEV), sw.to(DEV),
                           out_dtype=out_dtype, a_q=aq, a_scales=asc)
    return y, aq, asc


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M", [1, 5, 9, 16])
@pytest.mark.parametrize("N", [128, 640, 4096])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_matches_unfused_and_oracle(K, M, N, flags):
    x, wq, sw = _inputs(M, N, torch.bfloat16, 3 * M + N + K, K)
    xd, wd, sd = x.to(DEV), wq.to(DEV), sw.to(DEV)
    # unfused reference on the GPU
    q_u, s_u = rq.fwht_quant(xd, synth.SIGN_SEED, flags)
    for out_dtype in (torch.int32, torch.float32, torch.float16):
        y, aq, asc = _fused(x, flags, wq, sw, out_dtype)
        y_u = rq.w4a4_gemm(q_u, s_u, wd, sd, out_dtype=out_dtype)
        assert torch.equal(aq, q_u), "codes differ from rq_fwht_quant"
        assert torch.equal(asc, s_u), "scales differ from rq_fwht_quant"
        assert torch.equal(y, y_u), f"{out_dtype} output differs from rq_w4a4_gemm"
    # oracle, from its own codes: rotation codes and scales, then the product
    ref = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, flags, want_ratio=True)
    compare_scales(to_np(asc), ref["scales"])
    compare_codes(to_np(aq), ref["q"], ref["ratio"], K)
    acc, yref = oracle.w4a4_gemm(ref["q"], ref["scales"], wq.numpy(), sw.numpy(), M, N, K)
    ibound, fbound = _tie_bound(ref, wq.numpy(), sw.numpy())
    y32 = to_np(_fused(x, flags, wq, sw, torch.int32)[0]).astype(np.int64)
    assert np.all(np.abs(y32 - acc) <= ibound)
    yf = to_np(_fused(x, flags, wq, sw, torch.float32)[0]).astype(np.float64)
    assert np.all(np.abs(yf - yref) <= fbound + 1e-5 * np.abs(yref))
    compare_f16(to_np(_fused(x, flags, wq, sw, torch.float16)[0]), yref, atol=fbound)


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_dtypes_and_strided_rows(K, dt):
    M, N = 12, 1024
    x, wq, sw = _inputs(M, N, dt, 77, K)
    big = torch.zeros(M, K + 64, dtype=dt)
    big[:, :K] = x
    xd = big.to(DEV)[:, :K]                       # row stride K + 64 elements
    y = rq.fwht_quant_gemm(xd, synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, wq.to(DEV), sw.to(DEV), out_dtype=torch.int32)
    q_u, s_u = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    y_u = rq.w4a4_gemm(q_u, s_u, wq.to(DEV), sw.to(DEV), out_dtype=torch.int32)
    assert torch.equal(y, y_u)


@pytest.mark.parametrize("K", KS)
def test_zero_row_and_no_code_outputs(K):
    M, N = 3, 256
    x, wq, sw = _inputs(M, N, torch.bfloat16, 5, K)
    x[1] = 0
    y = rq.fwht_quant_gemm(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, wq.to(DEV), sw.to(DEV),
                           out_dtype=torch.float32)
    assert torch.all(y[1] == 0)
    q_u, s_u = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    assert torch.equal(y, rq.w4a4_gemm(q_u, s_u, wq.to(DEV), sw.to(DEV), out_dtype=torch.float32))


def test_decode_workload_full_size():
    """16 tokens x 4096 -> 4096 with the folded weights of the oracle's fold."""
    w = synth.WORKLOADS["decode"]
    x = synth.activations(w.rows, w.n, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    wt = synth.weights_t(w.gemm_n, w.n, w.weight_seed, w.w_std)             # W^T, N x K fp32
    fold = oracle.fwht_quant(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    wq, sw = torch.from_numpy(fold["q"]), torch.from_numpy(fold["scales"])
    y, aq, asc = _fused(x, rq.RQ_SIGNS_FIRST, wq, sw, torch.float32)
    K = w.n
    ref = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    compare_codes(to_np(aq), ref["q"], ref["ratio"], K)
    _, yref = oracle.w4a4_gemm(ref["q"], ref["scales"], fold["q"], fold["scales"], w.rows, w.gemm_n, K)
    _, fbound = _tie_bound(ref, fold["q"], fold["scales"])
    assert np.all(np.abs(to_np(y).astype(np.float64) - yref) <= fbound + 1e-5 * np.abs(yref))


def test_large_model_width_decode():
    """16 tokens of the large workload's activations (8192 wide, 0.1% outlier
    channels x100) through 28672 output channels (224 channel tiles in clusters
    of 8: several waves), against the oracle from its own codes."""
    w = synth.WORKLOADS["large"]
    M, K, N = 16, w.n, w.gemm_n
    x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    wq, sw = synth.random_codes(N, K, 515)
    y, aq, asc = _fused(x, rq.RQ_SIGNS_FIRST, wq, sw, torch.float32)
    q_u, s_u = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    assert torch.equal(aq, q_u) and torch.equal(asc, s_u)
    ref = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    compare_codes(to_np(aq), ref["q"], ref["ratio"], K)
    _, yref = oracle.w4a4_gemm(ref["q"], ref["scales"], wq.numpy(), sw.numpy(), M, N, K)
    _, fbound = _tie_bound(ref, wq.numpy(), sw.numpy())
    assert np.all(np.abs(to_np(y).astype(np.float64) - yref) <= fbound + 1e-5 * np.abs(yref))
