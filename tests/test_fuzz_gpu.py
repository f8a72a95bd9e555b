"""Seeded random shapes against the fp64 oracle (GPU).

Each case draws its batch, heads, vote-group size, lengths (ragged tails
included), head dimension, causal flag, split count and threshold from a
fixed seed, builds planted hot-tile inputs of that shape and runs the full
parity check: decisions, counters and outputs.
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


def _lam(rng, L):
    kind = rng.integers(0, 4)
    if kind == 0:
        return 0.0
    if kind == 1:
        return 1.0
    return min(1.0, float(rng.choice([0.5, 1.0, 2.0, 8.0, 32.0])) / L)


@pytest.mark.parametrize("seed", range(12))
def test_prefill_random_shapes(seed):
    from _parity import check_prefill, hot_prefill

    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    Lk = int(rng.integers(1, 1700))
    Lq = int(rng.integers(1, 700)) if rng.integers(0, 2) else Lk
    inp = hot_prefill(B, Hkv * G, Hkv, Lq, Lk, d, frac=float(rng.uniform(0.05, 0.4)),
                      seed=seed)
    check_prefill(inp.q, inp.k, inp.v, scale=1.0 / math.sqrt(d), causal=causal,
                  lam=_lam(rng, Lk))


@pytest.mark.parametrize("seed", range(12))
def test_decode_random_shapes(seed):
    from _parity import check_decode, hot_decode

    rng = np.random.default_rng(2000 + seed)
    Hkv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 3, 4, 8, 16, 20, 32]))
    B = int(rng.integers(1, 4))
    d = int(rng.choice([64, 128]))
    Lk = int(rng.integers(1, 6000))
    S = int(rng.integers(1, 9))
    inp = hot_decode(B, Hkv * G, Hkv, Lk, d, frac=float(rng.uniform(0.05, 0.4)), seed=seed)
    check_decode(inp.q, inp.k, inp.v, scale=1.0 / math.sqrt(d), lam=_lam(rng, Lk), num_splits=S)


@pytest.mark.parametrize("seed", range(8))
def test_mla_random_shapes(seed):
    from _parity import check_mla
    from block_sparse_attention_sm_gb300 import synth

    rng = np.random.default_rng(3000 + seed)
    B = int(rng.integers(1, 4))
    Hq = int(rng.integers(1, 33))
    Lk = int(rng.integers(1, 6000))
    S = int(rng.integers(1, 7))
    inp = synth.mla_decode_inputs(B=B, Hq=Hq, Lk=Lk, hot_frac=float(rng.uniform(0.05, 0.4)),
                                  seed=seed, device="cuda")
    check_mla(inp.q, inp.kv, scale=192 ** -0.5, lam=_lam(rng, Lk), num_splits=S)


@pytest.mark.parametrize("seed", range(6))
def test_decode_random_large_groups(seed):
    """Vote groups of 17..128 heads at d = 128 (the heads as MMA rows),
    including groups that leave a warp partly empty."""
    from _parity import check_decode, hot_decode

    rng = np.random.default_rng(2500 + seed)
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([17, 24, 33, 40, 64, 100, 128]))
    B = int(rng.integers(1, 3))
    Lk = int(rng.integers(1, 5000))
    S = int(rng.integers(1, 7))
    inp = hot_decode(B, Hkv * G, Hkv, Lk, 128, frac=float(rng.uniform(0.05, 0.4)), seed=seed)
    check_decode(inp.q, inp.k, inp.v, scale=1.0 / math.sqrt(128), lam=_lam(rng, Lk),
                 num_splits=S)


@pytest.mark.parametrize("seed", range(4))
def test_mla_random_shapes_many_heads(seed):
    """Latent-attention decode with 33..64 heads (heads as MMA rows, the
    latent entries of O over two CTAs)."""
    from _parity import check_mla
    from block_sparse_attention_sm_gb300 import synth

    rng = np.random.default_rng(3500 + seed)
    B = int(rng.integers(1, 3))
    Hq = int(rng.integers(33, 65))
    Lk = int(rng.integers(1, 5000))
    S = int(rng.integers(1, 6))
    inp = synth.mla_decode_inputs(B=B, Hq=Hq, Lk=Lk, hot_frac=float(rng.uniform(0.05, 0.4)),
                                  seed=seed, device="cuda")
    check_mla(inp.q, inp.kv, scale=192 ** -0.5, lam=_lam(rng, Lk), num_splits=S)
