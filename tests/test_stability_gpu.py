"""Calibration stability: count-only launches against the oracle (GPU).

BLASST summary, §Calibratie and §Resultaten ("Stabiliteit"): with lambda =
a/L and a calibrated once, the fraction of skipped tiles is meant to stay
near its target across context lengths, while a fixed lambda drifts.  The
study (bench.py --suite, part "stability") calibrates a at L = 32768 on
decode-shaped inputs and then counts skipped tiles at L = 4K ... 128K under
both rules with count-only launches.  This test checks those counting
launches themselves: at every length and under both rules, the skip mask and
the per-unit counts of sampled (sequence, KV head) units must equal the
oracle's, except on near-margin tiles (counted and reported).
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LENGTHS = [4096, 8192, 16384, 32768, 65536, 131072]
REF_L = 32768
B, HQ, HKV, D = 8, 32, 8, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import block_sparse_attention_sm_gb300 as ss
    import oracle

    ss.build()
    oracle.build()
    assert torch.cuda.is_available()


def _inputs(L):
    from block_sparse_attention_sm_gb300 import synth

    return synth.decode_inputs(B=B, Hq=HQ, Hkv=HKV, Lk=L, d=D, hot_frac=0.10, seed=3,
                               device="cuda")


def test_stability_sweep_counts_match_oracle():
    import oracle
    import block_sparse_attention_sm_gb300 as ss
    from _parity import Parity, _finish, compare_decisions, guarded
    from block_sparse_attention_sm_gb300 import capi

    scale = D ** -0.5
    ref = _inputs(REF_L)
    a, achieved = ss.calibrate("decode", ref.q, ref.k, ref.v, scale=scale, target_sparsity=0.7,
                               num_kv_splits=1)
    assert abs(achieved - 0.7) < 0.01
    del ref
    rng = np.random.default_rng(17)
    n = B * HKV
    units = sorted({0, n - 1, *rng.choice(n, size=3, replace=False).tolist()})
    fractions = {}
    for L in LENGTHS:
        inp = _inputs(L)
        nT = -(-L // 128)
        for rule, lam in (("a_over_L", min(1.0, a / L)), ("fixed", a / REF_L)):
            cg = guarded((n,), torch.int32, "cuda", -1)
            mg = guarded((n, nT), torch.uint8, "cuda", 7)
            gg = guarded((n, nT), torch.float32, "cuda", 12345.0)
            st = capi.ss_attn_decode_ex(inp.q, inp.k, inp.v, None, B, HQ, HKV, L, D, scale, lam,
                                        1, cg.t, None, 0, mg.t, gg.t, count_only=True)
            assert st == capi.SS_OK, capi.ss_status_string(st)
            assert capi.ss_stream_status() == capi.SS_OK
            torch.cuda.synchronize()
            for g, what in ((cg, "skip_counts"), (mg, "skip_mask"), (gg, "vote_margin")):
                g.check(what)
            counts, mask, margin = (g.t.cpu().numpy() for g in (cg, mg, gg))
            np.testing.assert_array_equal(counts, (mask == 1).sum(axis=1))
            fractions[(L, rule)] = counts.sum() / (n * nT)
            rec = Parity(f"stability_{rule}", lam)
            for u in units:
                b, kvh = divmod(u, HKV)
                G = HQ // HKV
                res = oracle.decode(inp.q[b:b + 1, kvh * G:(kvh + 1) * G],
                                    inp.k[b:b + 1, kvh:kvh + 1], inp.v[b:b + 1, kvh:kvh + 1],
                                    scale=scale, lam=lam, num_splits=1)
                nd, row_dis = compare_decisions(mask[u:u + 1], margin[u:u + 1], res.mask,
                                                res.margin, lam)
                rec.units += 1
                rec.disagree += nd
                rec.add_decisions(mask[u:u + 1], res.mask, res.margin, lam)
                if not row_dis[0]:
                    assert counts[u] == res.counts[0, 0], (L, rule, u)
            _finish(rec)
        del inp
        torch.cuda.empty_cache()
    # the calibration length reproduces the target under both rules (same lambda)
    assert abs(fractions[(REF_L, "a_over_L")] - 0.7) < 0.01
    assert fractions[(REF_L, "fixed")] == fractions[(REF_L, "a_over_L")]
