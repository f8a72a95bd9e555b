"""The oracle over a grid of tiny shapes (CPU).

Lengths Lq, Lk in {1, 5, 128, 130, 300, 1024} pairwise, head dims {4, 64,
128}, causal on and off, vote groups G in {1, 4} for prefill; decode over the
same key lengths with S in {1, 2, 3} splits and G in {1, 4}.  Each case is
checked against a direct two-pass softmax: the whole attention at lambda = 0,
and the attention restricted to the keys of the kept tiles at a threshold
that skips some of them.  The tile size is the kernels' 128.
"""
import itertools
import math

import numpy as np
import pytest

from test_oracle_pins import f64, rand_bits, two_pass, visible

LENS = [1, 5, 128, 130, 300, 1024]
DIMS = [4, 64, 128]


def _prefill_inputs(rng, B, Hq, Hkv, Lq, Lk, d):
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, Lq, d), shift=3.0 * u)
    kx = rng.standard_normal((B, Hkv, Lk, d))
    kx[rng.random((B, Hkv, Lk)) < 0.2] += 3.0 * u
    from test_oracle_pins import bf16_bits

    return q, bf16_bits(kx), rand_bits(rng, (B, Hkv, Lk, d))


PREFILL_GRID = [(Lq, Lk, DIMS[i % 3], bool(i % 2), 1 if (i // 2) % 2 == 0 else 4)
                for i, (Lq, Lk) in enumerate(itertools.product(LENS, LENS))]


@pytest.mark.parametrize("Lq,Lk,d,causal,G", PREFILL_GRID)
def test_prefill_grid(oracle_lib, Lq, Lk, d, causal, G):
    rng = np.random.default_rng(Lq * 7919 + Lk * 31 + d)
    Hkv = 1
    Hq = G
    q, k, v = _prefill_inputs(rng, 1, Hq, Hkv, Lq, Lk, d)
    scale = 1.0 / math.sqrt(d)
    vis = visible(Lq, Lk, causal)
    dense = oracle_lib.prefill(q, k, v, scale=scale, causal=causal, lam=0.0)
    nqb = -(-Lq // 128)
    for h in range(Hq):
        ref = two_pass(f64(q[0, h]), f64(k[0, 0]), f64(v[0, 0]), scale, vis)
        got = dense.o[h * nqb:(h + 1) * nqb].reshape(-1, d)[:Lq]
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)
    sparse = oracle_lib.prefill(q, k, v, scale=scale, causal=causal, lam=0.05)
    nT = -(-Lk // 128)
    for h in range(Hq):
        got = sparse.o[h * nqb:(h + 1) * nqb].reshape(-1, d)[:Lq]
        for qb in range(nqb):
            r0, r1 = qb * 128, min(Lq, qb * 128 + 128)
            keep = np.repeat(sparse.mask[h * nqb + qb] == 0, 128)[:Lk]
            ref = two_pass(f64(q[0, h, r0:r1]), f64(k[0, 0]), f64(v[0, 0]), scale,
                           vis[r0:r1] & keep[None, :])
            np.testing.assert_allclose(got[r0:r1], ref, rtol=0, atol=1e-10)
    # the not-evaluated tiles are exactly those no row of the block sees
    for qb in range(nqb):
        r0, r1 = qb * 128, min(Lq, qb * 128 + 128)
        for j in range(nT):
            seen = vis[r0:r1, j * 128:min(Lk, j * 128 + 128)].any()
            assert (sparse.mask[qb, j] == 2) == (not seen)


DECODE_GRID = [(Lk, S, G, DIMS[(i + j) % 3]) for i, Lk in enumerate(LENS)
               for j, (S, G) in enumerate(itertools.product([1, 2, 3], [1, 4]))]


@pytest.mark.parametrize("Lk,S,G,d", DECODE_GRID)
def test_decode_grid(oracle_lib, Lk, S, G, d):
    rng = np.random.default_rng(Lk * 131 + S * 17 + G + d)
    B, Hkv = 2, 2
    Hq = G * Hkv
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, d), shift=3.0 * u)
    _, k, v = _prefill_inputs(rng, B, Hkv, Hkv, 1, Lk, d)
    scale = 1.0 / math.sqrt(d)
    for lam in (0.0, 0.05):
        res = oracle_lib.decode(q, k, v, scale=scale, lam=lam, num_splits=S)
        for i, unit in enumerate(res.units):
            b, kvh = divmod(int(unit), Hkv)
            keep = np.repeat(res.mask[i] == 0, 128)[:Lk]
            ref = two_pass(f64(q[b, kvh * G:(kvh + 1) * G]), f64(k[b, kvh]), f64(v[b, kvh]),
                           scale, np.broadcast_to(keep, (G, Lk)))
            np.testing.assert_allclose(res.o[i], ref, rtol=0, atol=1e-10)
            if lam == 0.0:
                assert (res.mask[i] == 0).all()
