"""Key lengths at the top of the supported range (GPU).

Prefill decides and computes the key tiles in runs of 2048; 300K keys take
two runs at the default run length.  Decode and latent-attention decode
stream very long splits (one split of 8192 and 2048 tiles).
"""
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
    assert torch.cuda.is_available()


@pytest.mark.slow
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_two_vote_runs_at_default_length(causal):
    from _parity import check_prefill, hot_prefill

    Lk = 300_000                      # 2344 key tiles: runs of 2048 and 296
    Lq = 256 if not causal else 300   # causal: the last rows see every key
    inp = hot_prefill(1, 2, 1, Lq, Lk, 128, frac=0.02, seed=13)
    check_prefill(inp.q, inp.k, inp.v, scale=128 ** -0.5, causal=causal, lam=4.0 / Lk)


def test_decode_one_split_over_a_million_keys():
    from _parity import check_decode, hot_decode

    Lk = 1 << 20
    inp = hot_decode(1, 8, 2, Lk, 128, frac=0.01, seed=14)
    check_decode(inp.q, inp.k, inp.v, scale=128 ** -0.5, lam=8.0 / Lk, num_splits=1)


def test_mla_one_split_over_256k_keys():
    from _parity import check_mla
    from block_sparse_attention_sm_gb300 import synth

    Lk = 1 << 18
    inp = synth.mla_decode_inputs(B=1, Hq=16, Lk=Lk, hot_frac=0.01, seed=15, device="cuda")
    check_mla(inp.q, inp.kv, scale=192 ** -0.5, lam=8.0 / Lk, num_splits=1)
