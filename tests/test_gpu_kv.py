"""GPU parity of rq_kv_rotate_quant (head-wise rotation + INT4 of K and V)."""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_codes, compare_scales, record, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check(k, v, seed, flags):
    out = rq.kv_rotate_quant(None if k is None else k.to(DEV), None if v is None else v.to(DEV), seed, flags)
    ref = oracle.kv_rotate_quant(None if k is None else k.double().numpy(),
                                 None if v is None else v.double().numpy(), seed, flags)
    D = (k if k is not None else v).shape[-1]
    ties = 0
    for src, qk, sk in ((k, "kq", "ks"), (v, "vq", "vs")):
        if src is None:
            continue
        compare_scales(to_np(out[sk]), ref[sk])
        # tie-window ratios from the oracle's own rotation of the same rows
        rot = oracle.rotate(src.double().numpy().reshape(-1, D), seed, flags)
        _, sc, ratio = oracle.quant_rows(rot)
        ties += compare_codes(to_np(out[qk]), ref[qk], ratio, D)
    return ties


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("flags", [rq.RQ_SIGNS_FIRST, 0])
def test_head_dims(D, flags):
    k, v = synth.kv_pair(37, 5, D, seed=D, outliers_per_head=2, factor=30.0)
    _check(k, v, 77, flags)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_dtypes(dtype):
    k, v = synth.kv_pair(50, 3, 128, seed=4, outliers_per_head=2, factor=30.0, dtype=dtype)
    _check(k, v, 5, rq.RQ_SIGNS_FIRST)


def test_k_only_and_v_only():
    k, v = synth.kv_pair(9, 2, 128, seed=6)
    _check(k, None, 3, rq.RQ_SIGNS_FIRST)
    _check(None, v, 3, rq.RQ_SIGNS_FIRST)


def test_kv_workload_full_size():
    w = synth.KV
    k, v = synth.kv_pair(w.kv_tokens, w.kv_heads, w.kv_head_dim, w.data_seed,
                         w.kv_outliers_per_head, w.kv_outlier_factor)
    ties = _check(k, v, synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    print(f"kv: {ties} tie-window code differences")
    record("kv_workload", tokens=w.kv_tokens, heads=w.kv_heads, head_dim=w.kv_head_dim,
           codes=2 * k.numel(), tie_window_differences=ties)


def test_kv_equals_fwht_quant_on_flattened_rows():
    # the KV path is the row path with n = head_dim over [T*H] rows
    k, v = synth.kv_pair(64, 8, 128, seed=8)
    out = rq.kv_rotate_quant(k.to(DEV), v.to(DEV), 11, rq.RQ_SIGNS_FIRST)
    q, s = rq.fwht_quant(k.reshape(-1, 128).to(DEV), 11, rq.RQ_SIGNS_FIRST)
    assert torch.equal(out["kq"].reshape(-1, 64), q) and torch.equal(out["ks"].reshape(-1), s)
