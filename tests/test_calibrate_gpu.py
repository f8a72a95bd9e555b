"""Calibration (lambda = a / L) from the kernels' skipped-tile counters (GPU)."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import block_sparse_attention_sm_gb300 as ss
    import oracle

    ss.build()
    oracle.build()


def _near(margin, mask, a, L):
    ln_lam = math.log(a / L) if a > 0 else -math.inf
    ev = mask != 2
    return int((np.abs(margin[ev] - ln_lam) < 1e-2).sum())


@pytest.mark.parametrize("target", [0.3, 0.5, 0.7])
def test_prefill_calibration_hits_target_count(target):
    """ss_calibrate returns an a whose oracle sparsity is round(s N)/N, up to
    near-margin tiles; it agrees with the oracle's order-statistic a."""
    import oracle
    from _parity import hot_prefill
    import block_sparse_attention_sm_gb300 as ss

    inp = hot_prefill(1, 4, 2, 1024, 2048, 128, frac=0.3, seed=2)
    scale = 128 ** -0.5
    a, achieved = ss.calibrate("prefill", inp.q, inp.k, inp.v, scale=scale,
                               target_sparsity=target, causal=True)
    ref0 = oracle.prefill(inp.q, inp.k, inp.v, scale=scale, causal=True, lam=0.0)
    a_orc, k_orc, N = oracle.calibrate(ref0.margin, ref0.mask, target, 2048)
    k_want = k_orc
    res = oracle.prefill(inp.q, inp.k, inp.v, scale=scale, causal=True, lam=a / 2048)
    tol = _near(ref0.margin, ref0.mask, a, 2048)
    assert abs(int(res.counts.sum()) - k_want) <= tol
    assert abs(round(achieved * N) - k_want) <= tol
    # Both a's are the log-midpoint of the plateau of ln(lambda) that skips
    # k_want tiles: the oracle's from its fp64 statistics, ss_calibrate's from
    # the GPU's fp32 ones, whose ends differ by at most the statistic's error
    # (the margin tolerance of the parity tests).  So the two midpoints agree
    # to that error, and the oracle's own a skips exactly k_want tiles.
    assert a > 0 and a_orc > 0
    assert abs(math.log(a) - math.log(a_orc)) <= 2e-2 + 2e-4 * abs(math.log(a_orc / 2048))
    res_orc = oracle.prefill(inp.q, inp.k, inp.v, scale=scale, causal=True, lam=a_orc / 2048)
    assert int(res_orc.counts.sum()) == k_want


def test_decode_calibration_and_fit():
    import oracle
    from _parity import hot_decode
    import block_sparse_attention_sm_gb300 as ss

    inp = hot_decode(4, 8, 2, 8192, 128, frac=0.1, seed=1)
    scale = 128 ** -0.5
    ss_pts, a_pts = [], []
    ref0 = oracle.decode(inp.q, inp.k, inp.v, scale=scale, lam=0.0, num_splits=4)
    for target in (0.5, 0.7, 0.85):
        a, achieved = ss.calibrate("decode", inp.q, inp.k, inp.v, scale=scale,
                                   target_sparsity=target, num_kv_splits=4)
        a_orc, k_orc, N = oracle.calibrate(ref0.margin, ref0.mask, target, 8192)
        tol = _near(ref0.margin, ref0.mask, a, 8192)
        assert abs(round(achieved * N) - k_orc) <= tol
        ss_pts.append(target)
        a_pts.append(a)
    A, B = ss.fit_factor(ss_pts, a_pts)
    assert A > 0 and math.isfinite(B)
    assert ss.lambda_of(A, B, 0.7, 8192) > 0
