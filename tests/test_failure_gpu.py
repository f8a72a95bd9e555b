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
