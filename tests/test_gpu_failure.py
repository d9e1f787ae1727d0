"""Failure detection on the GPU without a fault: the LM-head kernel's bounded waits.

tim_selftest_wait_timeout runs the kernel with its TMA producer stalled, so nothing
ever arrives on the pipeline barriers; every wait gives up after the limit, the
kernel records TIM_ERR_TIMEOUT and winds down.  The test checks the status, that
the call returned within a bounded time, and that the context still scores
correctly afterwards."""
import time

import numpy as np
import pytest

import oracle
import synth
from parity import assert_logprob_parity, bf16_cuda, cuda_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tim():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


def test_bounded_wait_reports_timeout_and_context_survives(tim):
    t0 = time.monotonic()
    assert tim.selftest_wait_timeout(50) == "TIM_ERR_TIMEOUT"
    assert time.monotonic() - t0 < 10.0
    b = synth.make_tiny()
    got = [x.cpu().numpy() for x in tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma),
                                                bf16_cuda(b.head.W), cuda_tensor(b.token_ids),
                                                1.0, b.eps)]
    orc = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    assert_logprob_parity(got, orc, what="after the self-test")
    assert tim.selftest_wait_timeout(1) == "TIM_ERR_TIMEOUT"   # shortest limit, again


def test_selftest_limits(tim):
    for bad in (0, -5, 2001):
        with pytest.raises(tim.TimError) as ei:
            tim.selftest_wait_timeout(bad)
        assert ei.value.name == "TIM_ERR_INVALID_ARG"
