"""Latent-attention (MLA) prefill vs the fp64 oracle (GPU).

BLASST summary, §Belangrijkste Bijdragen item 4: the prefill kernels support
MLA.  Read in its unabsorbed prefill form: per head the query and key rows
are 128 non-rotary + 64 rotary entries (d_qk = 192) and the value rows 128
wide (d_v = 128).  The oracle computes the same tile pass with separate key
and value widths; decisions, counts and outputs follow the acceptance of the
other parity tests, the near-margin tiles are reported in the session summary.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DQK, DV = 192, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import block_sparse_attention_sm_gb300 as ss
    import oracle

    ss.build()
    oracle.build()
    assert torch.cuda.is_available()


def _inputs(B, Hq, Hkv, Lq, Lk, seed, frac=0.25):
    from block_sparse_attention_sm_gb300 import synth

    return synth.prefill_inputs(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=DQK, dv=DV, hot_frac=frac,
                                seed=seed, per_head_u=True, device="cuda")


SHAPES = [
    # B, Hq, Hkv, Lq, Lk, causal
    (1, 2, 2, 1000, 1000, True),      # ragged tail, causal
    (1, 4, 2, 300, 1500, True),       # GQA, Lq < Lk (bottom-right)
    (2, 2, 1, 640, 640, False),       # MQA, batch of two
    (1, 2, 2, 129, 129, False),       # one row past a block (odd block count)
    (1, 2, 2, 400, 250, True),        # Lq > Lk: first rows see no key
    (2, 2, 1, 1, 200, True),          # a single query row (causal: it sees every key)
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("lam_kind", ["dense", "mid", "high"])
def test_mla_prefill_shapes(shape, lam_kind):
    from _parity import check_prefill

    B, Hq, Hkv, Lq, Lk, causal = shape
    inp = _inputs(B, Hq, Hkv, Lq, Lk, seed=4)
    assert inp.v.shape[-1] == DV and inp.k.shape[-1] == DQK
    lam = {"dense": 0.0, "mid": 1.0 / Lk, "high": min(1.0, 64.0 / Lk)}[lam_kind]
    rec = check_prefill(inp.q, inp.k, inp.v, scale=DQK ** -0.5, causal=causal, lam=lam)
    assert rec.kind == "mla_prefill"


def test_mla_prefill_rejects_other_widths():
    from block_sparse_attention_sm_gb300 import capi

    x = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    st = capi.ss_attn_mla_prefill(x, x, x, x, 1, 1, 1, 8, 8, 128, 128, 0.1, 0, 0.0, None)
    assert st == capi.SS_ERR_UNSUPPORTED
    st = capi.ss_attn_mla_prefill(x, x, x, x, 1, 1, 1, 8, 8, 192, 64, 0.1, 0, 0.0, None)
    assert st == capi.SS_ERR_UNSUPPORTED


@pytest.mark.slow
@pytest.mark.parametrize("target", [0.5, 0.7])
def test_mla_prefill_full_size_at_calibrated_lambda(target):
    """mla_prefill_16k (16 heads, 16K causal) at the a ss_calibrate fits."""
    import block_sparse_attention_sm_gb300 as ss
    from _parity import check_prefill
    from block_sparse_attention_sm_gb300 import synth

    inp, cfg = synth.make("mla_prefill_16k", seed=0, device="cuda")
    a, achieved = ss.calibrate("mla_prefill", inp.q, inp.k, inp.v, scale=cfg["scale"],
                               target_sparsity=target, causal=True)
    assert abs(achieved - target) < 0.01, achieved
    rng = np.random.default_rng(5)
    nqb = cfg["Lq"] // 128
    units = []
    for h in sorted(rng.choice(cfg["Hq"], size=3, replace=False).tolist()):
        for qb in sorted({0, nqb - 1, *rng.choice(nqb, size=4, replace=False).tolist()}):
            units.append((0, int(h), int(qb)))
    rec = check_prefill(inp.q, inp.k, inp.v, scale=cfg["scale"], causal=True, lam=a / cfg["Lk"],
                        units=units)
    assert rec.skipped > 0
