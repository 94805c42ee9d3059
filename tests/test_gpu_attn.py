"""GPU parity of rq_attn_decode (attention of decode queries over the rotated INT4
KV cache) against the oracle.

The cache is written by the oracle's own KV rotation + quantization, so the GPU
kernel and the oracle read the same codes and scales.  The kernel works in fp32
(rotation of the query, scores, exp2, sums); the tolerance is 1e-4 of each output
row's largest magnitude: fp32 dot products of head_dim terms and sums over the
tokens of one CTA slice carry relative errors of order 1e-6 for these inputs, and
exp2 of the scores adds ~2e-7.  Shapes cover every head_dim, both sign sides,
both output bases, three query dtypes, several query rows, token counts below the
8 CTAs of a cluster, ragged slices, a near one-hot softmax and the full
8192-token x 32-head x 128 workload.
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = synth.SIGN_SEED
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(T, H, D, M, flags, data_seed, q_dtype=torch.bfloat16, factor=30.0):
    k, v = synth.kv_pair(T, H, D, data_seed, 2, factor)
    q = synth.kv_pair(M, H, D, data_seed + 500, 2, factor)[0].to(q_dtype)
    cache = oracle.kv_rotate_quant(k.double().numpy(), v.double().numpy(), SEED, flags & 1)
    return q, cache


def _gpu(q, cache, flags, scale):
    dc = {name: torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for name, a in cache.items()}
    out = rq.attn_decode(q.to(DEV), dc, SEED, flags, scale)
    assert rq.sync_status() == 0
    return to_np(out)


def _compare(got, ref):
    err = np.abs(got - ref).max(axis=-1)
    bound = TOL * np.abs(ref).max(axis=-1)
    assert np.all(err <= bound), f"max rel error {float((err / np.abs(ref).max(axis=-1)).max()):.3e}"


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_matches_oracle_every_head_dim(D, flags):
    T, H, M = 777, 3, 2
    q, cache = _case(T, H, D, M, flags, 10 + D)
    scale = D ** -0.5
    ref = oracle.attn_decode(q.double().numpy(), cache["kq"], cache["ks"], cache["vq"], cache["vs"], SEED,
                             flags & 1, scale, rotated_out=bool(flags & 2))
    _compare(_gpu(q, cache, flags, scale), ref)


@pytest.mark.parametrize("T", [1, 3, 8, 9, 64, 511, 513, 4096 + 37])
def test_token_counts(T):
    """Fewer tokens than CTAs in a cluster (empty slices), one token, ragged slices."""
    H, D, M, flags = 2, 128, 1, 1
    q, cache = _case(T, H, D, M, flags, 70 + T)
    ref = oracle.attn_decode(q.double().numpy(), cache["kq"], cache["ks"], cache["vq"], cache["vs"], SEED, 1,
                             D ** -0.5)
    _compare(_gpu(q, cache, flags, D ** -0.5), ref)


@pytest.mark.parametrize("q_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_query_dtypes(q_dtype):
    T, H, D, M, flags = 300, 4, 64, 3, 1
    q, cache = _case(T, H, D, M, flags, 91, q_dtype=q_dtype)
    ref = oracle.attn_decode(q.double().numpy(), cache["kq"], cache["ks"], cache["vq"], cache["vs"], SEED, 1,
                             D ** -0.5)
    _compare(_gpu(q, cache, flags, D ** -0.5), ref)


def test_sharp_and_flat_softmax():
    """A large softmax scale (weights close to one-hot) and a zero scale (the mean
    of the values)."""
    T, H, D, M, flags = 1000, 2, 128, 1, 1
    q, cache = _case(T, H, D, M, flags, 93)
    for scale in (2.0, 0.0):
        ref = oracle.attn_decode(q.double().numpy(), cache["kq"], cache["ks"], cache["vq"], cache["vs"], SEED, 1,
                                 scale)
        _compare(_gpu(q, cache, flags, scale), ref)


def test_kv_workload_full_size():
    """The 8192-token x 32-head x 128 cache of the KV workload, one decode query."""
    w = synth.KV
    T, H, D = w.kv_tokens, w.kv_heads, w.kv_head_dim
    k, v = synth.kv_pair(T, H, D, w.data_seed, w.kv_outliers_per_head, w.kv_outlier_factor)
    q = synth.kv_pair(1, H, D, w.data_seed + 500, w.kv_outliers_per_head, w.kv_outlier_factor)[0]
    cache = oracle.kv_rotate_quant(k.double().numpy(), v.double().numpy(), SEED, 1)
    ref = oracle.attn_decode(q.double().numpy(), cache["kq"], cache["ks"], cache["vq"], cache["vs"], SEED, 1,
                             D ** -0.5)
    _compare(_gpu(q, cache, 1, D ** -0.5), ref)


def test_cache_from_gpu_writer_runs_and_repeats():
    """The cache written by rq_kv_rotate_quant on the GPU feeds the read directly;
    two launches give identical bits."""
    T, H, D = 2048, 8, 128
    k, v = synth.kv_pair(T, H, D, 95, 2, 30.0)
    q = synth.kv_pair(2, H, D, 96, 2, 30.0)[0]
    cache = rq.kv_rotate_quant(k.to(DEV), v.to(DEV), SEED, 1)
    a = rq.attn_decode(q.to(DEV), cache, SEED, 1)
    b = rq.attn_decode(q.to(DEV), cache, SEED, 1)
    assert rq.sync_status() == 0
    assert torch.equal(a, b)
    assert torch.isfinite(a).all()
