"""Split-KV decode kernel vs the fp64 oracle (GPU)."""
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


SHAPES = [
    # B, Hq, Hkv, Lk, d, splits
    (3, 8, 2, 1000, 128, 1),
    (3, 8, 2, 1000, 128, 3),    # splits that do not divide the 8 tiles
    (2, 32, 8, 4096, 128, 8),
    (2, 4, 4, 777, 64, 2),      # MHA (G = 1), d = 64
    (1, 8, 1, 2000, 128, 16),   # G = 8 (MQA with 8 query heads); one split per tile
    (2, 6, 2, 1500, 64, 4),     # G = 3 (padded vote group)
    (1, 4, 1, 100, 128, 1),     # one partial tile
    (1, 4, 1, 300, 128, 8),     # more splits than tiles: empty splits
    (2, 8, 1, 900, 64, 3),      # d = 64 with an 8-row vote group
    (1, 16, 1, 1000, 128, 2),   # G = 16 (largest group of the 16-row MMA)
    (2, 24, 2, 700, 64, 1),     # G = 12 (padded to 16 rows)
    (2, 32, 1, 3000, 128, 3),   # G = 32: MQA with 32 query heads (the largest vote group)
    (2, 48, 2, 1300, 64, 2),    # G = 24 (padded to 32 rows), d = 64
    (1, 17, 1, 640, 128, 1),    # G = 17: the smallest group of the 32-row MMA
    # d = 128 groups above 16 heads: the heads as MMA rows
    (1, 33, 1, 700, 128, 1),    # G = 33: a warp with one head
    (2, 96, 2, 900, 128, 4),    # G = 48, two KV heads
    (2, 64, 1, 3000, 128, 3),   # G = 64 (MQA with 64 query heads)
    (1, 128, 1, 1500, 128, 2),  # G = 128: every row of the MMA
    (1, 40, 1, 300, 128, 8),    # more splits than tiles: empty splits
    (2, 8, 2, 1, 128, 2),       # a single key (the second split is empty)
    (1, 40, 1, 1, 128, 1),      # a single key, heads as MMA rows
    (1, 4, 4, 1, 64, 1),        # a single key, d = 64
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("a", [0.0, 1.0, 8.0])
def test_decode_shapes(shape, a):
    from _parity import check_decode, hot_decode

    B, Hq, Hkv, Lk, d, S = shape
    inp = hot_decode(B, Hq, Hkv, Lk, d, frac=0.2, seed=4)
    check_decode(inp.q, inp.k, inp.v, scale=1.0 / math.sqrt(d), lam=min(1.0, a / Lk),
                 num_splits=S)


def test_decode_random_scores():
    """N(0,1) inputs; two thresholds on critical values of the oracle's vote
    statistic (near-margin tiles certain, counted), two elsewhere."""
    import oracle
    from _parity import check_decode
    from test_prefill_gpu import _lambdas_on_critical_values

    g = torch.Generator(device="cuda").manual_seed(9)
    q = torch.randn(4, 8, 128, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(4, 2, 3000, 128, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(4, 2, 3000, 128, device="cuda", generator=g).to(torch.bfloat16)
    ref0 = oracle.decode(q, k, v, scale=128 ** -0.5, lam=0.0, num_splits=5)
    near = 0
    for lam in _lambdas_on_critical_values(ref0.margin, 2) + [0.2, 0.6, 1.0]:
        near += check_decode(q, k, v, scale=128 ** -0.5, lam=lam, num_splits=5).near
    assert near >= 2
