"""GPU parity of rq_w4a4_gemm against the oracle.

The GEMM is fed the oracle's (or seeded random) codes, so the comparison is of
the product alone: int32 accumulators bit-exact, fp32 dequant within 1e-5
relative, fp16 within one ulp.  Shapes cover decode-sized and prefill-sized M,
ragged M / N, every output mode, extreme codes, and the full-size workloads
(every output against the oracle, run over row blocks on all host cores, plus
row and column sums that hold at any size).
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_f16, host_threads, operand_form, operand_scales, oracle_gemm_row_blocks, record, to_dev, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _codes(M, N, K, seed):
    aq, sa = synth.random_codes(M, K, seed)
    wq, sw = synth.random_codes(N, K, seed + 1)
    return aq, sa, wq, sw


def _all_modes(aq, sa, wq, sw):
    d = [t.to(DEV) for t in (aq, sa, wq, sw)]
    return {dt: to_np(rq.w4a4_gemm(*d, out_dtype=dt)) for dt in (torch.int32, torch.float32, torch.float16)}


@pytest.mark.parametrize("M,N,K", [
    (1, 64, 128), (16, 64, 256), (17, 72, 384), (64, 1024, 1024), (100, 136, 512),
    (128, 256, 256), (130, 264, 512), (256, 512, 1024), (300, 392, 640), (512, 1024, 2048),
])
def test_shapes_all_modes(M, N, K):
    aq, sa, wq, sw = _codes(M, N, K, M * 7 + N)
    out = _all_modes(aq, sa, wq, sw)
    acc, y = oracle.w4a4_gemm(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K)
    np.testing.assert_array_equal(out[torch.int32].astype(np.int64), acc)
    np.testing.assert_allclose(out[torch.float32], y, rtol=1e-5, atol=0)
    compare_f16(out[torch.float16], y)


@pytest.mark.parametrize("M,N,K", [(16, 64, 65536), (256, 256, 65536)])
@pytest.mark.parametrize("ba,bw", [(0x77, 0x77), (0x88, 0x88), (0x88, 0x77), (0x78, 0x87)])
def test_extreme_codes_at_max_k(M, N, K, ba, bw):
    aq = synth.extreme_codes(M, K, ba)
    wq = synth.extreme_codes(N, K, bw)
    one_m, one_n = torch.ones(M), torch.ones(N)
    acc = to_np(rq.w4a4_gemm(aq.to(DEV), one_m.to(DEV), wq.to(DEV), one_n.to(DEV), out_dtype=torch.int32))
    ref, _ = oracle.w4a4_gemm(aq[:1].numpy(), one_m[:1].numpy(), wq[:1].numpy(), one_n[:1].numpy(), 1, 1, K)
    assert (acc.astype(np.int64) == ref[0, 0]).all()


@pytest.mark.parametrize("M,N,K", [
    (128, 81920, 128),    # one CTA per tile row: 320 tiles, 1 K block each
    (96, 51200, 640),     # single CTAs, 200 tiles, 5 K blocks (not a multiple of 3)
    (256, 40960, 384),    # CTA pairs: 160 tiles on 76 pairs, 3 K blocks
    (384, 20480, 640),    # CTA pairs, 160 tiles, 5 K blocks, ragged last M tile
])
def test_many_tiles_per_cta(M, N, K):
    """Persistent CTAs walk several tiles; the converter teams take K blocks
    round-robin across tile boundaries and the per-tile sums and accumulators
    alternate between two buffers."""
    aq, sa, wq, sw = _codes(M, N, K, 11 + M + K)
    d = [t.to(DEV) for t in (aq, sa, wq, sw)]
    acc_gpu = to_np(rq.w4a4_gemm(*d, out_dtype=torch.int32)).astype(np.int64)
    y_gpu = to_np(rq.w4a4_gemm(*d, out_dtype=torch.float32))
    acc, y = oracle.w4a4_gemm(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K)
    np.testing.assert_array_equal(acc_gpu, acc)
    np.testing.assert_allclose(y_gpu, y, rtol=1e-5, atol=0)


def test_large_then_small_partial_sums():
    # Accumulation order hazard: a huge partial sum followed by +-1 products.
    M, N, K = 128, 128, 16384
    a = np.zeros((M, K), np.int8)
    w = np.zeros((N, K), np.int8)
    a[:, : K // 2] = 7
    w[:, : K // 2] = 7
    rng = np.random.default_rng(0)
    a[:, K // 2:] = rng.choice([-1, 1], size=(M, K // 2))
    w[:, K // 2:] = rng.choice([-1, 1], size=(N, K // 2))
    aq, wq = oracle.pack(a), oracle.pack(w)
    ones_m, ones_n = np.ones(M, np.float32), np.ones(N, np.float32)
    acc = to_np(rq.w4a4_gemm(to_dev(aq), to_dev(ones_m), to_dev(wq), to_dev(ones_n), out_dtype=torch.int32))
    ref, _ = oracle.w4a4_gemm(aq, ones_m, wq, ones_n, M, N, K)
    np.testing.assert_array_equal(acc.astype(np.int64), ref)


def test_pipeline_codes_from_oracle_fold():
    # X rotated+quantized and W^T folded+quantized by the oracle, product on the GPU.
    w = synth.TINY
    x = synth.activations(w.rows, w.n, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    wt = synth.weights_t(w.gemm_n, w.n, w.weight_seed, w.w_std)
    xa = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    wf = oracle.fwht_quant(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    out = _all_modes(torch.from_numpy(xa["q"]), torch.from_numpy(xa["scales"]),
                     torch.from_numpy(wf["q"]), torch.from_numpy(wf["scales"]))
    acc, y = oracle.w4a4_gemm(xa["q"], xa["scales"], wf["q"], wf["scales"], w.rows, w.gemm_n, w.n)
    np.testing.assert_array_equal(out[torch.int32].astype(np.int64), acc)
    np.testing.assert_allclose(out[torch.float32], y, rtol=1e-5, atol=0)
    compare_f16(out[torch.float16], y)


@pytest.mark.parametrize("name", ["decode", "prefill", "large"])
def test_workload_full_output(name):
    """Every output of the full-size decode, prefill and large products against
    the oracle: int32 accumulators bit-exact, fp32 within 1e-5 relative, fp16
    within one ulp.  The oracle runs over disjoint row blocks on all host cores."""
    import time
    w = synth.WORKLOADS[name]
    M, N, K = w.rows, w.gemm_n, w.n
    aq, sa, wq, sw = _codes(M, N, K, 1000 + w.data_seed)
    d = [t.to(DEV) for t in (aq, sa, wq, sw)]
    acc_np = to_np(rq.w4a4_gemm(*d, out_dtype=torch.int32)).astype(np.int64)
    yf = to_np(rq.w4a4_gemm(*d, out_dtype=torch.float32))
    yh = to_np(rq.w4a4_gemm(*d, out_dtype=torch.float16))
    assert rq.sync_status() == 0
    a_np, sa_np, w_np, sw_np = aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy()
    threads = host_threads()
    t0 = time.perf_counter()
    for r0, r_acc, r_y in oracle_gemm_row_blocks(a_np, sa_np, w_np, sw_np, M, N, K, threads):
        r1 = r0 + r_acc.shape[0]
        np.testing.assert_array_equal(acc_np[r0:r1], r_acc)
        np.testing.assert_allclose(yf[r0:r1], r_y, rtol=1e-5, atol=0)
        compare_f16(yh[r0:r1], r_y)
    record("gemm_full_output", workload=name, M=M, N=N, K=K, outputs=M * N, host_threads=threads,
           oracle_seconds=round(time.perf_counter() - t0, 2))
    # Whole-output properties as well: sum_c acc[m,c] = a_m . (sum_c w_c) and
    # sum_m acc[m,c] = (sum_m a_m) . w_c, from the oracle's code decoding.
    a = oracle.unpack(a_np, K)
    wc = oracle.unpack(w_np, K)
    a_sum = a.sum(axis=0, dtype=np.int64)
    w_sum = wc.sum(axis=0, dtype=np.int64)
    row_ref = np.concatenate([a[i:i + 512].astype(np.int64) @ w_sum for i in range(0, M, 512)])
    col_ref = np.concatenate([wc[i:i + 512].astype(np.int64) @ a_sum for i in range(0, N, 512)])
    np.testing.assert_array_equal(acc_np.sum(axis=1), row_ref)
    np.testing.assert_array_equal(acc_np.sum(axis=0), col_ref)


def test_full_output_on_oracle_codes_prefill():
    """The prefill product on the oracle's own codes of the workload (rotated and
    quantized activations, folded and quantized weights), every output compared."""
    w = synth.PREFILL
    M, N, K = w.rows, w.gemm_n, w.n
    x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor)
    wt = synth.weights_t(N, K, w.weight_seed, w.w_std)
    xa = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    wf = oracle.fwht_quant(wt.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    d = [torch.from_numpy(a).to(DEV) for a in (xa["q"], xa["scales"], wf["q"], wf["scales"])]
    acc_np = to_np(rq.w4a4_gemm(*d, out_dtype=torch.int32)).astype(np.int64)
    yf = to_np(rq.w4a4_gemm(*d, out_dtype=torch.float32))
    for r0, r_acc, r_y in oracle_gemm_row_blocks(xa["q"], xa["scales"], wf["q"], wf["scales"], M, N, K):
        r1 = r0 + r_acc.shape[0]
        np.testing.assert_array_equal(acc_np[r0:r1], r_acc)
        np.testing.assert_allclose(yf[r0:r1], r_y, rtol=1e-5, atol=0)


def test_repeatable_bitwise():
    aq, sa, wq, sw = _codes(512, 1024, 4096, 3)
    d = [t.to(DEV) for t in (aq, sa, wq, sw)]
    r1 = rq.w4a4_gemm(*d, out_dtype=torch.float16)
    r2 = rq.w4a4_gemm(*d, out_dtype=torch.float16)
    assert torch.equal(r1, r2)


# Decode-sized products (M <= 64, N a multiple of 128, K <= 8192) run on the
# tensor-core decode kernel: weights in tensor memory, K split over a cluster of
# 1, 2, 4 or 8 CTAs (chosen from K and the number of 128-channel tiles) whose
# exact partials meet in distributed shared memory.  The shapes below reach
# every split, uneven K slices (K blocks not a multiple of the split), every
# token-tile count (16, 32, 48, 64 padded rows) and the largest slice.
@pytest.mark.parametrize("M,N,K", [
    (1, 128, 128),       # one CTA, one K block
    (5, 256, 384),       # split 2, slices of 1 and 2 blocks
    (16, 128, 1152),     # split 8, slices of 1 and 2 blocks
    (17, 512, 4096),     # split 8, 4 blocks each, two token tiles
    (33, 1024, 2048),    # three token tiles
    (48, 4096, 8192),    # split 8, 8 blocks each (the largest slice)
    (64, 2048, 1024),    # four token tiles, split 8 of one block
    (7, 19200, 512),     # 150 channel tiles, split 1
])
def test_decode_tensor_core_shapes(M, N, K):
    aq, sa, wq, sw = _codes(M, N, K, 77 + M + K)
    out = _all_modes(aq, sa, wq, sw)
    assert rq.sync_status() == 0
    acc, y = oracle.w4a4_gemm(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K)
    np.testing.assert_array_equal(out[torch.int32].astype(np.int64), acc)
    np.testing.assert_allclose(out[torch.float32], y, rtol=1e-5, atol=0)
    compare_f16(out[torch.float16], y)


@pytest.mark.parametrize("ba,bw", [(0x77, 0x77), (0x88, 0x88), (0x88, 0x77), (0x78, 0x87)])
def test_decode_tensor_core_extreme_codes(ba, bw):
    """All-extreme codes at the decode kernel's largest K (8192): every partial
    and the cluster's integer sum stay exact."""
    M, N, K = 16, 256, 8192
    aq = synth.extreme_codes(M, K, ba)
    wq = synth.extreme_codes(N, K, bw)
    one_m, one_n = torch.ones(M), torch.ones(N)
    acc = to_np(rq.w4a4_gemm(aq.to(DEV), one_m.to(DEV), wq.to(DEV), one_n.to(DEV), out_dtype=torch.int32))
    ref, _ = oracle.w4a4_gemm(aq[:1].numpy(), one_m[:1].numpy(), wq[:1].numpy(), one_n[:1].numpy(), 1, 1, K)
    assert (acc.astype(np.int64) == ref[0, 0]).all()


def test_decode_tensor_core_large_model_width():
    """16 tokens through the large workload's 8192 -> 28672 weights (224 channel
    tiles, split 8: several waves of clusters), every output against the oracle."""
    M, N, K = 16, 28672, 8192
    aq, sa, wq, sw = _codes(M, N, K, 4242)
    d = [t.to(DEV) for t in (aq, sa, wq, sw)]
    acc_np = to_np(rq.w4a4_gemm(*d, out_dtype=torch.int32)).astype(np.int64)
    yf = to_np(rq.w4a4_gemm(*d, out_dtype=torch.float32))
    for r0, r_acc, r_y in oracle_gemm_row_blocks(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K):
        r1 = r0 + r_acc.shape[0]
        np.testing.assert_array_equal(acc_np[r0:r1], r_acc)
        np.testing.assert_allclose(yf[r0:r1], r_y, rtol=1e-5, atol=0)



# Activations in the operand form (RQ_A_E4M3, M > 64): the product reads the
# codes as signed E4M3 bytes straight into its operand ring, widens only W (to
# q + 8) and removes 8 x each row's code sum, which comes beside its scale.
def _e4m3_all_modes(aq, sa, wq, sw):
    ae = torch.from_numpy(operand_form(aq.numpy())).to(DEV)
    sa2 = torch.from_numpy(operand_scales(aq.numpy(), sa.numpy())).to(DEV)
    d = [t.to(DEV) for t in (wq, sw)]
    return {dt: to_np(rq.w4a4_gemm(ae, sa2, d[0], d[1], out_dtype=dt)) for dt in (torch.int32, torch.float32, torch.float16)}


@pytest.mark.parametrize("M,N,K", [
    (65, 256, 128), (100, 136, 512), (128, 256, 256), (130, 264, 512), (256, 512, 1024), (300, 392, 640),
    (384, 20480, 640), (256, 40960, 384), (512, 1024, 4096),
])
def test_e4m3_activations_shapes(M, N, K):
    aq, sa, wq, sw = _codes(M, N, K, 5 * M + N)
    out = _e4m3_all_modes(aq, sa, wq, sw)
    assert rq.sync_status() == 0
    acc, y = oracle.w4a4_gemm(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K)
    np.testing.assert_array_equal(out[torch.int32].astype(np.int64), acc)
    np.testing.assert_allclose(out[torch.float32], y, rtol=1e-5, atol=0)
    compare_f16(out[torch.float16], y)


@pytest.mark.parametrize("ba,bw", [(0x77, 0x77), (0x88, 0x88), (0x88, 0x77), (0x78, 0x87)])
def test_e4m3_activations_extreme_codes_at_max_k(ba, bw):
    M, N, K = 256, 256, 65536
    aq = synth.extreme_codes(M, K, ba)
    wq = synth.extreme_codes(N, K, bw)
    one_m, one_n = torch.ones(M), torch.ones(N)
    ae = torch.from_numpy(operand_form(aq.numpy())).to(DEV)
    sa2 = torch.from_numpy(operand_scales(aq.numpy(), one_m.numpy())).to(DEV)
    acc = to_np(rq.w4a4_gemm(ae, sa2, wq.to(DEV), one_n.to(DEV), out_dtype=torch.int32))
    ref, _ = oracle.w4a4_gemm(aq[:1].numpy(), one_m[:1].numpy(), wq[:1].numpy(), one_n[:1].numpy(), 1, 1, K)
    assert (acc.astype(np.int64) == ref[0, 0]).all()


@pytest.mark.parametrize("name", ["prefill", "large"])
def test_e4m3_activations_workload_full_output(name):
    """Every output of the prefill and large products with operand-form activations."""
    w = synth.WORKLOADS[name]
    M, N, K = w.rows, w.gemm_n, w.n
    aq, sa, wq, sw = _codes(M, N, K, 2000 + w.data_seed)
    out = _e4m3_all_modes(aq, sa, wq, sw)
    acc_np = out[torch.int32].astype(np.int64)
    for r0, r_acc, r_y in oracle_gemm_row_blocks(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), M, N, K):
        r1 = r0 + r_acc.shape[0]
        np.testing.assert_array_equal(acc_np[r0:r1], r_acc)
        np.testing.assert_allclose(out[torch.float32][r0:r1], r_y, rtol=1e-5, atol=0)
        compare_f16(out[torch.float16][r0:r1], r_y)


def test_e4m3_path_end_to_end_matches_packed_path():
    """Rotation in operand form, then the product, equals the packed-code path bit for bit."""
    M, N, K = 384, 1024, 4096
    x = synth.activations(M, K, torch.bfloat16, 9, 4, 100.0).to(DEV)
    wq, sw = synth.random_codes(N, K, 10)
    wd, sd = wq.to(DEV), sw.to(DEV)
    qp, sp = rq.fwht_quant(x, 7, rq.RQ_SIGNS_FIRST)
    qe, se = rq.fwht_quant(x, 7, rq.RQ_SIGNS_FIRST | rq.RQ_E4M3_CODES)
    for dt in (torch.int32, torch.float32, torch.float16):
        assert torch.equal(rq.w4a4_gemm(qe, se, wd, sd, out_dtype=dt), rq.w4a4_gemm(qp, sp, wd, sd, out_dtype=dt))
