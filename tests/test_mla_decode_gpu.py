"""Latent-attention (MLA) decode vs the fp64 oracle (GPU).

The keys are the 576-entry latent cache rows (512 latent + 64 rotary
entries), the values their latent part, and all query heads of a sequence
vote together on each tile ("Skip-Softmax" design doc: MLA listed among the
supported attention kinds; the absorbed-form reading is the oracle's).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SCALE = 192 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import block_sparse_attention_sm_gb300 as ss
    import oracle

    ss.build()
    oracle.build()
    assert torch.cuda.is_available()


def _inputs(B, Hq, Lk, frac=0.2, seed=0):
    from block_sparse_attention_sm_gb300 import synth

    return synth.mla_decode_inputs(B=B, Hq=Hq, Lk=Lk, hot_frac=frac, seed=seed, device="cuda")


CASES = [
    # B, Hq, Lk, splits
    (2, 16, 1000, 1),     # ragged last tile, one split (no merge)
    (3, 16, 5000, 3),     # several splits, several tiles each
    (2, 8, 129, 2),       # one key past a tile
    (1, 1, 1, 1),         # a single key, a single head
    (2, 12, 4096, 8),     # heads padded to the MMA's 16 rows
    (1, 16, 300, 5),      # more splits than tiles: empty splits
    (1, 16, 20000, 2),    # long splits: the copy ring wraps many times
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("a", [0.0, 1.0, 8.0])
def test_mla_decode(case, a):
    from _parity import check_mla

    B, Hq, Lk, S = case
    inp = _inputs(B, Hq, Lk, seed=4)
    check_mla(inp.q, inp.kv, scale=SCALE, lam=min(1.0, a / Lk), num_splits=S)


def test_mla_random_scores_many_decisions():
    """Plain N(0,1) inputs: margins spread out around the threshold."""
    from _parity import check_mla

    g = torch.Generator(device="cuda").manual_seed(8)
    q = torch.randn(2, 16, 576, device="cuda", generator=g).to(torch.bfloat16)
    kv = torch.randn(2, 3000, 576, device="cuda", generator=g).to(torch.bfloat16)
    for lam in (0.3, 0.8):
        check_mla(q, kv, scale=576 ** -0.5, lam=lam, num_splits=3)


def test_mla_count_only_matches_the_full_launch():
    from block_sparse_attention_sm_gb300 import capi

    B, Hq, Lk, S = 4, 16, 8192, 4
    inp = _inputs(B, Hq, Lk, frac=0.1, seed=2)
    lam = 3.0 / Lk
    ws_n = capi.ss_attn_mla_decode_workspace_size(B, Hq, 512, S)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    o = torch.empty(B, Hq, 512, dtype=torch.bfloat16, device="cuda")
    c1 = torch.full((B * S,), -1, dtype=torch.int32, device="cuda")
    c2 = torch.full_like(c1, -1)
    assert capi.ss_attn_mla_decode(inp.q, inp.kv, o, B, Hq, Lk, 512, 64, SCALE, lam, S, c1, ws,
                                   ws_n) == capi.SS_OK
    assert capi.ss_attn_mla_decode_ex(inp.q, inp.kv, None, B, Hq, Lk, 512, 64, SCALE, lam, S, c2,
                                      None, 0, count_only=True) == capi.SS_OK
    assert capi.ss_stream_status() == capi.SS_OK
    assert torch.equal(c1, c2) and int(c1.sum()) > 0


def test_mla_calibration_hits_the_target():
    import block_sparse_attention_sm_gb300 as ss

    B, Hq, Lk, S = 4, 16, 16384, 4
    inp = _inputs(B, Hq, Lk, frac=0.1, seed=5)
    nT = Lk // 128
    for target in (0.5, 0.7):
        a, achieved = ss.calibrate("mla_decode", inp.q, inp.kv, None, scale=SCALE,
                                   target_sparsity=target, num_kv_splits=S)
        assert a > 0
        assert abs(achieved - round(target * B * nT) / (B * nT)) <= 2.0 / (B * nT)


@pytest.mark.slow
def test_mla_full_size_sampled():
    """The bench's workload (64 sequences x 32K keys, 16 splits) at lambda for
    70% skipped tiles; the oracle checks the first, last and two random
    sequences."""
    import block_sparse_attention_sm_gb300 as ss
    from _parity import check_mla
    from block_sparse_attention_sm_gb300 import synth

    inp, cfg = synth.make("mla_decode_32k", seed=0, device="cuda")
    a, _ = ss.calibrate("mla_decode", inp.q, inp.kv, None, scale=cfg["scale"], target_sparsity=0.7,
                        num_kv_splits=cfg["num_splits"])
    rng = np.random.default_rng(3)
    units = sorted({0, cfg["B"] - 1, *rng.choice(cfg["B"], size=2, replace=False).tolist()})
    check_mla(inp.q, inp.kv, scale=cfg["scale"], lam=min(1.0, a / cfg["Lk"]),
              num_splits=cfg["num_splits"], units=units)
