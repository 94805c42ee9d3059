"""Failure detection on the GPU without a fault: a bounded device-side wait that
runs out.

The self-test launches one thread that waits, through the same bounded mbarrier
wait the rotation kernels use for their bulk copies, on a barrier that nothing
arrives on.  The wait gives up after its cycle limit, raises the library's
device error word and returns; the host reads RQ_ERR_TIMEOUT from
rq_sync_status, the word is cleared, and the context stays usable for the next
real call.
"""
import numpy as np
import pytest
import torch

import oracle
import rotational_w4a4_quantization_gb300 as rq
from rotational_w4a4_quantization_gb300 import synth

from parity import compare_codes, compare_scales, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
RQ_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_wait_runs_out_and_is_reported():
    assert rq.sync_status() == 0
    rq.selftest_wait_timeout(20_000_000)          # ~10 ms at 2 GHz
    assert rq.sync_status() == RQ_ERR_TIMEOUT
    assert rq.sync_status() == 0                  # read and cleared


def test_context_usable_after_timeout():
    rq.selftest_wait_timeout(5_000_000)
    assert rq.sync_status() == RQ_ERR_TIMEOUT
    x = synth.activations(8, 1024, torch.bfloat16, 3, 2, 100.0)
    q, s = rq.fwht_quant(x.to(DEV), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST)
    assert rq.sync_status() == 0
    ref = oracle.fwht_quant(x.double().numpy(), synth.SIGN_SEED, rq.RQ_SIGNS_FIRST, want_ratio=True)
    compare_codes(to_np(q), ref["q"], ref["ratio"], 1024)
    compare_scales(to_np(s), ref["scales"])


def test_timeout_on_a_side_stream():
    st = torch.cuda.Stream()
    rq.selftest_wait_timeout(5_000_000, stream=st)
    assert rq.sync_status(stream=st) == RQ_ERR_TIMEOUT
    assert rq.sync_status() == 0
