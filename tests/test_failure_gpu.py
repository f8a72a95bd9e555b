"""Failure detection on the GPU without a GPU fault.

Every wait in the kernels is bounded: a wait that does not complete within
about a second makes the kernel give up, let its in-flight copies land,
free what it holds and return, and the host reads SS_ERR_TIMEOUT from the
library's device status word.  The test makes one wait run out on purpose
(a copy that is never issued, via the test-only fault_inject option) and
checks the status, then checks that the same context still computes
correctly.
"""
import math
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import block_sparse_attention_sm_gb300 as ss
    import oracle

    ss.build()
    oracle.build()
    assert torch.cuda.is_available()


def test_expired_wait_reports_timeout_and_context_survives():
    from _parity import check_decode, hot_decode
    from block_sparse_attention_sm_gb300 import capi

    # One CTA: one sequence, one KV head, one split of 8 tiles.
    inp = hot_decode(1, 4, 1, 1024, 128, frac=0.2, seed=12)
    o = torch.empty_like(inp.q)
    counts = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert capi.ss_stream_status() == capi.SS_OK
    st = capi.ss_attn_decode_ex(inp.q, inp.k, inp.v, o, 1, 4, 1, 1024, 128, 1 / math.sqrt(128),
                                0.002, 1, counts, None, 0, fault_inject=1)
    assert st == capi.SS_OK  # launched; the failure is found on the device
    t0 = time.time()
    status = capi.ss_stream_status()
    elapsed = time.time() - t0
    assert status == capi.SS_ERR_TIMEOUT
    assert elapsed < 30.0
    # the status word was cleared and the context is still usable
    assert capi.ss_stream_status() == capi.SS_OK
    check_decode(inp.q, inp.k, inp.v, scale=1 / math.sqrt(128), lam=0.002, num_splits=1)
    assert capi.ss_stream_status() == capi.SS_OK


def test_calibration_reports_an_expired_wait():
    """ss_calibrate reads the device status word after each count-only
    launch: when a bounded wait expired (test-only fault_inject), the
    counters are not used and it returns SS_ERR_TIMEOUT instead of an a."""
    from _parity import hot_decode
    from block_sparse_attention_sm_gb300 import capi

    inp = hot_decode(1, 4, 1, 1024, 128, frac=0.2, seed=12)
    counts = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert capi.ss_stream_status() == capi.SS_OK
    prob = capi.ss_problem(capi.SS_DECODE, inp.q.data_ptr(), inp.k.data_ptr(), inp.v.data_ptr(),
                           1, 4, 1, 1, 1024, 128, 1 / math.sqrt(128), 0, 1, counts.data_ptr(),
                           capi._stream(None), 1)
    st, _, _ = capi.ss_calibrate(prob, 0.5)
    assert st == capi.SS_ERR_TIMEOUT
    assert capi.ss_stream_status() == capi.SS_OK  # read and cleared by the calibration
    prob.fault_inject = 0
    st, a, achieved = capi.ss_calibrate(prob, 0.5)
    assert st == capi.SS_OK and a > 0 and achieved > 0
