"""Pins for the fp64 oracle, each from something other than the oracle itself.

* lambda = 0 equals a direct two-pass softmax(Q K^T scale) V (numpy, fp64);
* the skip decisions equal a brute-force prefix-maximum form of the test
  (no online recurrence): skipped tiles never raise the running maximum when
  lambda <= 1, so the running maximum before tile j is the maximum over all
  earlier tiles, whatever was skipped;
* the sparse output equals the two-pass softmax restricted to the keys of the
  kept tiles;
* the exact error identity o' - o = rho (o' - N_s / D_s) and its bound;
* split-KV decode at lambda = 0 is independent of the number of splits;
* hand-worked examples (tests/golden/worked_examples.json);
* the order-statistic calibration skips exactly round(s N) tiles.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ----------------------------------------------------------------- helpers
def bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bits(rng, shape, scale=1.0, shift=None):
    x = rng.standard_normal(shape) * scale
    if shift is not None:
        x = x + shift
    return bf16_bits(x)


def visible(Lq, Lk, causal):
    if not causal:
        return np.ones((Lq, Lk), bool)
    r = np.arange(Lq)[:, None]
    c = np.arange(Lk)[None, :]
    return c <= r + (Lk - Lq)


def two_pass(q, k, v, scale, vis):
    """Direct softmax(scale q k^T) v over the visible keys; rows with none -> 0."""
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    M = s.max(axis=1)
    out = np.zeros((q.shape[0], v.shape[1]))
    ok = np.isfinite(M)
    p = np.exp(s[ok] - M[ok, None])
    out[ok] = (p @ v) / p.sum(axis=1, keepdims=True)
    return out


def prefix_decisions(s, Bk, tiles, ln_lam):
    """Decisions from the prefix maximum of the row scores (property P).

    s: [rows, Lk] masked scores (-inf where not visible).  Returns
    (mask, margin) for the listed tiles in order, running the maximum over
    every evaluated tile regardless of its decision."""
    rows, Lk = s.shape
    prev = np.full(rows, -np.inf)
    mask, margin = [], []
    for j in tiles:
        t = s[:, j * Bk:min(Lk, (j + 1) * Bk)].max(axis=1)
        fin = np.isfinite(t)
        if not fin.any():
            mask.append(2)
            margin.append(np.nan)
            continue
        diff = np.where(np.isfinite(prev[fin]), t[fin] - prev[fin], np.inf)
        c = diff.max()
        mask.append(1 if c < ln_lam else 0)
        margin.append(c)
        prev = np.maximum(prev, t)
    return np.array(mask, np.uint8), np.array(margin)


def unit_rows(u, Hq, nqb, Bq, Lq):
    qb = u % nqb
    bh = u // nqb
    return bh // Hq, bh % Hq, qb * Bq, min(Lq, qb * Bq + Bq)


PREFILL_SHAPES = [
    # B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk
    (1, 1, 1, 16, 16, 8, False, 4, 4),
    (1, 2, 1, 13, 13, 5, True, 4, 4),     # MQA, ragged tails, causal
    (2, 4, 2, 10, 23, 6, True, 4, 4),     # GQA, Lq < Lk (chunked-prefill alignment)
    (1, 2, 2, 23, 9, 4, True, 8, 4),      # Lq > Lk: early rows see no key at all
    (1, 3, 3, 7, 30, 16, False, 3, 7),
    (1, 2, 1, 130, 300, 64, True, 128, 128),
    (1, 1, 1, 5, 1, 4, False, 128, 128),  # a single key
]


def run_prefill_case(oracle_lib, shape, lam, seed, hot=False, shift=3.0):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, Lq, d), shift=(shift * u if hot else None))
    kx = rng.standard_normal((B, Hkv, Lk, d))
    if hot:  # a few hot keys so that decisions vary
        sel = rng.random((B, Hkv, Lk)) < 0.15
        kx[sel] += shift * u
    k = bf16_bits(kx)
    v = rand_bits(rng, (B, Hkv, Lk, d))
    scale = 1.0 / math.sqrt(d)
    res = oracle_lib.prefill(q, k, v, scale=scale, causal=causal, lam=lam, Bq=Bq, Bk=Bk)
    return (q, k, v, scale), res


# ------------------------------------------------------------ dense pins
@pytest.mark.parametrize("shape", PREFILL_SHAPES)
def test_dense_equals_two_pass_softmax(oracle_lib, shape):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    (q, k, v, scale), res = run_prefill_case(oracle_lib, shape, 0.0, 1)
    G = Hq // Hkv
    nqb = -(-Lq // Bq)
    vis = visible(Lq, Lk, causal)
    for i, u in enumerate(res.units):
        b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
        ref = two_pass(f64(q[b, h]), f64(k[b, h // G]), f64(v[b, h // G]), scale, vis)
        np.testing.assert_allclose(res.o[i, : r1 - r0], ref[r0:r1], rtol=0, atol=1e-10)
        assert not res.o[i, r1 - r0:].any()
    assert (res.counts == 0).all() and not (res.mask == 1).any()


# ------------------------------------------------------- decision pins
def unit_scores(q, k, scale, shape, u):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    G = Hq // Hkv
    nqb = -(-Lq // Bq)
    b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
    s = scale * (f64(q[b, h, r0:r1]) @ f64(k[b, h // G]).T)
    return np.where(visible(Lq, Lk, causal)[r0:r1], s, -np.inf), (b, h, r0, r1)


@pytest.mark.parametrize("shape", PREFILL_SHAPES[:6])
def test_decisions_equal_prefix_max_form(oracle_lib, shape):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    nT = -(-Lk // Bk)
    (q, k, v, scale), res0 = run_prefill_case(oracle_lib, shape, 0.0, 2, hot=True)
    # Critical values from the brute force; thresholds between them.
    cs = []
    for u in res0.units:
        s, _ = unit_scores(q, k, scale, shape, u)
        _, c = prefix_decisions(s, Bk, range(nT), -np.inf)
        cs.extend(x for x in c if np.isfinite(x))
    cs = np.unique(np.array(cs))
    cs = cs[cs < 0]
    mids = (cs[:-1] + cs[1:]) / 2 if len(cs) > 1 else np.array([])
    lams = sorted({0.0, 1.0} | {float(np.exp(x)) for x in mids[:: max(1, len(mids) // 6)]})
    prev_mask = None
    for lam in lams:
        _, res = run_prefill_case(oracle_lib, shape, lam, 2, hot=True)
        ln_lam = math.log(lam) if lam > 0 else -np.inf
        for i, u in enumerate(res.units):
            s, _ = unit_scores(q, k, scale, shape, u)
            m_ref, c_ref = prefix_decisions(s, Bk, range(nT), ln_lam)
            np.testing.assert_array_equal(res.mask[i], m_ref)
            fin = np.isfinite(c_ref)
            np.testing.assert_allclose(res.margin[i][fin], c_ref[fin], rtol=0, atol=1e-12)
            assert np.array_equal(np.isposinf(res.margin[i]), np.isposinf(c_ref))
            assert res.counts[i] == (m_ref == 1).sum()
        # Invariant I4: the skipped set only grows with lambda.
        if prev_mask is not None:
            assert ((prev_mask == 1) <= (res.mask == 1)).all()
        prev_mask = res.mask.copy()


@pytest.mark.parametrize("shape", [(1, 2, 1, 16, 24, 8, False, 4, 4),
                                   (1, 1, 1, 13, 13, 5, True, 4, 4)])
def test_every_critical_value_sweep(oracle_lib, shape):
    """lambda at every midpoint between consecutive critical values (and
    below / above all of them): by property P a tile is skipped exactly when
    its statistic c_j < ln(lambda), so the launch skips exactly the number of
    critical values below ln(lambda), and the skipped sets are nested."""
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    nT = -(-Lk // Bk)
    (q, k, v, scale), res0 = run_prefill_case(oracle_lib, shape, 0.0, 5, hot=True)
    cs = []
    for u in res0.units:
        s, _ = unit_scores(q, k, scale, shape, u)
        _, c = prefix_decisions(s, Bk, range(nT), -np.inf)
        cs.extend(x for x in c if np.isfinite(x))
    cs = np.sort(np.array(cs))
    below_zero = np.unique(cs[cs < 0])
    assert len(below_zero) >= 3, "the case must have several critical values below ln 1"
    pts = np.concatenate([[below_zero[0] - 1.0], (below_zero[:-1] + below_zero[1:]) / 2, [0.0]])
    prev = None
    for x in pts:
        lam = float(np.exp(x))
        _, res = run_prefill_case(oracle_lib, shape, lam, 5, hot=True)
        skipped = int(res.counts.sum())
        assert skipped == int((cs < math.log(lam)).sum())
        if prev is not None:
            assert ((prev == 1) <= (res.mask == 1)).all()
        prev = res.mask.copy()


@pytest.mark.parametrize("shape", PREFILL_SHAPES[:6])
@pytest.mark.parametrize("lam", [0.02, 0.2, 0.6])
def test_sparse_output_is_softmax_over_kept_tiles(oracle_lib, shape, lam):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    G = Hq // Hkv
    nqb = -(-Lq // Bq)
    (q, k, v, scale), res = run_prefill_case(oracle_lib, shape, lam, 3, hot=True)
    vis = visible(Lq, Lk, causal)
    for i, u in enumerate(res.units):
        b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
        keep = np.repeat(res.mask[i] == 0, Bk)[:Lk]
        ref = two_pass(f64(q[b, h]), f64(k[b, h // G]), f64(v[b, h // G]), scale,
                       vis & keep[None, :])
        np.testing.assert_allclose(res.o[i, : r1 - r0], ref[r0:r1], rtol=0, atol=1e-10)


@pytest.mark.parametrize("shape", PREFILL_SHAPES[:6])
def test_invariants_first_tile_and_no_new_max(oracle_lib, shape):
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    nT = -(-Lk // Bk)
    (q, k, v, scale), res = run_prefill_case(oracle_lib, shape, 0.9, 4, hot=True)
    for i, u in enumerate(res.units):
        ev = np.nonzero(res.mask[i] != 2)[0]
        if len(ev) == 0:
            assert res.counts[i] == 0
            continue
        assert res.mask[i, ev[0]] == 0                        # I1
        assert res.counts[i] <= len(ev) - 1                   # I3
        s, _ = unit_scores(q, k, scale, shape, u)
        run = np.full(s.shape[0], -np.inf)
        for j in range(nT):                                   # I2
            t = s[:, j * Bk:(j + 1) * Bk].max(axis=1)
            if res.mask[i, j] == 1:
                assert (t <= run).all()
            if res.mask[i, j] == 0:
                run = np.maximum(run, t)


@pytest.mark.parametrize("lam", [0.05, 0.3, 0.9])
def test_error_identity_and_bound(oracle_lib, lam):
    shape = (1, 2, 1, 24, 40, 8, True, 8, 4)
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    G = Hq // Hkv
    nqb = -(-Lq // Bq)
    (q, k, v, scale), dense = run_prefill_case(oracle_lib, shape, 0.0, 5, hot=True, shift=5.0)
    _, sparse = run_prefill_case(oracle_lib, shape, lam, 5, hot=True, shift=5.0)
    assert sparse.counts.sum() > 0
    vis = visible(Lq, Lk, causal)
    for i, u in enumerate(sparse.units):
        b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
        vv = f64(v[b, h // G])
        s = scale * (f64(q[b, h, r0:r1]) @ f64(k[b, h // G]).T)
        s = np.where(vis[r0:r1], s, -np.inf)
        skipped_key = np.repeat(sparse.mask[i] == 1, Bk)[:Lk]
        for r in range(r1 - r0):
            if not np.isfinite(s[r]).any():
                continue
            M = s[r].max()
            w = np.exp(s[r] - M)
            Ds = w[skipped_key].sum()
            if Ds == 0:
                np.testing.assert_allclose(sparse.o[i, r], dense.o[i, r], atol=1e-12)
                continue
            Ns = w[skipped_key] @ vv[skipped_key]
            Dk = w[~skipped_key].sum()
            rho = Ds / (Dk + Ds)
            o_s, o_d = sparse.o[i, r], dense.o[i, r]
            np.testing.assert_allclose(o_s - o_d, rho * (o_s - Ns / Ds), rtol=0, atol=1e-12)
            bound = rho * (np.abs(o_s).max() + np.abs(vv[skipped_key]).max())
            assert np.abs(o_s - o_d).max() <= bound + 1e-15
            # every skipped key's weight relative to the row maximum is below lambda
            assert (w[skipped_key & np.isfinite(s[r])] < lam).all()


# ---------------------------------------------------------- decode pins
DECODE_SHAPES = [
    # B, Hq, Hkv, Lk, d, S, Bk
    (2, 4, 1, 37, 8, 1, 4),
    (2, 8, 2, 37, 8, 3, 4),
    (1, 4, 4, 50, 6, 4, 5),
    (3, 4, 1, 9, 4, 8, 4),     # more splits than tiles: empty splits
    (1, 2, 1, 300, 64, 2, 128),
    (2, 4, 2, 64, 8, 4, 4),     # splits that divide the 16 tiles: 4 tiles each
    (1, 8, 1, 48, 8, 2, 4),     # 12 tiles in 2 splits of 6
]


def decode_case(oracle_lib, shape, lam, seed, hot=True):
    B, Hq, Hkv, Lk, d, S, Bk = shape
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, d), shift=3.0 * u)
    kx = rng.standard_normal((B, Hkv, Lk, d))
    if hot:
        kx[rng.random((B, Hkv, Lk)) < 0.15] += 3.0 * u
    k = bf16_bits(kx)
    v = rand_bits(rng, (B, Hkv, Lk, d))
    scale = 1.0 / math.sqrt(d)
    return (q, k, v, scale), oracle_lib.decode(q, k, v, scale=scale, lam=lam, num_splits=S, Bk=Bk)


@pytest.mark.parametrize("shape", DECODE_SHAPES)
def test_decode_dense_equals_two_pass_and_is_split_invariant(oracle_lib, shape):
    B, Hq, Hkv, Lk, d, S, Bk = shape
    G = Hq // Hkv
    (q, k, v, scale), res = decode_case(oracle_lib, shape, 0.0, 6)
    for i, u in enumerate(res.units):
        b, kvh = divmod(int(u), Hkv)
        ref = two_pass(f64(q[b, kvh * G:(kvh + 1) * G]), f64(k[b, kvh]), f64(v[b, kvh]), scale,
                       np.ones((G, Lk), bool))
        np.testing.assert_allclose(res.o[i], ref, rtol=0, atol=1e-10)
    for S2 in (1, 2, 5, 16):
        _, r2 = decode_case(oracle_lib, (B, Hq, Hkv, Lk, d, S2, Bk), 0.0, 6)
        np.testing.assert_allclose(r2.o, res.o, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", DECODE_SHAPES)
@pytest.mark.parametrize("lam", [0.01, 0.3, 1.0])
def test_decode_sparse_decisions_and_output(oracle_lib, shape, lam):
    B, Hq, Hkv, Lk, d, S, Bk = shape
    G = Hq // Hkv
    nT = -(-Lk // Bk)
    T = -(-nT // S)
    (q, k, v, scale), res = decode_case(oracle_lib, shape, lam, 7)
    for i, u in enumerate(res.units):
        b, kvh = divmod(int(u), Hkv)
        qq, kk, vv = f64(q[b, kvh * G:(kvh + 1) * G]), f64(k[b, kvh]), f64(v[b, kvh])
        s = scale * (qq @ kk.T)
        for sp in range(S):
            tiles = range(sp * T, min(nT, (sp + 1) * T))
            m_ref, c_ref = prefix_decisions(s, Bk, tiles, math.log(lam))
            np.testing.assert_array_equal(res.mask[i, list(tiles)], m_ref)
            assert res.counts[i, sp] == (m_ref == 1).sum()
            if len(m_ref):
                assert m_ref[0] == 0  # the first tile of a split is never skipped
            fin = np.isfinite(c_ref)
            np.testing.assert_allclose(res.margin[i, list(tiles)][fin], c_ref[fin], atol=1e-12)
        keep = np.repeat(res.mask[i] == 0, Bk)[:Lk]
        ref = two_pass(qq, kk, vv, scale, np.broadcast_to(keep, (G, Lk)))
        np.testing.assert_allclose(res.o[i], ref, rtol=0, atol=1e-10)


# ----------------------------------------------- latent-attention decode pins
MLA_SHAPES = [
    # B, Hq, Lk, dk (latent + rotary), d_latent, S, Bk
    (2, 4, 37, 12, 8, 1, 4),
    (1, 3, 50, 9, 6, 4, 5),
    (3, 5, 9, 7, 4, 8, 4),          # more splits than tiles
    (2, 16, 260, 576, 512, 2, 128),  # the kernel's widths, a ragged last tile
]


def mla_case(oracle_lib, shape, lam, seed):
    B, Hq, Lk, dk, dl, S, Bk = shape
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(dk)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, dk), shift=3.0 * u)
    kx = rng.standard_normal((B, Lk, dk))
    kx[rng.random((B, Lk)) < 0.15] += 3.0 * u
    kv = bf16_bits(kx)
    scale = 1.0 / math.sqrt(dk)
    res = oracle_lib.mla_decode(q, kv, d_latent=dl, scale=scale, lam=lam, num_splits=S, Bk=Bk)
    return (q, kv, scale), res


@pytest.mark.parametrize("shape", MLA_SHAPES)
def test_mla_dense_equals_two_pass_over_latent_values(oracle_lib, shape):
    """lambda = 0: every head's output is softmax(scale q kv^T) kv[:, :d_latent]
    (values are the leading latent entries of the same rows), for any split."""
    B, Hq, Lk, dk, dl, S, Bk = shape
    (q, kv, scale), res = mla_case(oracle_lib, shape, 0.0, 11)
    assert res.o.shape == (B, Hq, dl)
    for b in range(B):
        kk = f64(kv[b])
        ref = two_pass(f64(q[b]), kk, kk[:, :dl], scale, np.ones((Hq, Lk), bool))
        np.testing.assert_allclose(res.o[b], ref, rtol=0, atol=1e-10)
    for S2 in (1, 3, 7):
        _, r2 = mla_case(oracle_lib, (B, Hq, Lk, dk, dl, S2, Bk), 0.0, 11)
        np.testing.assert_allclose(r2.o, res.o, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", MLA_SHAPES)
@pytest.mark.parametrize("lam", [0.05, 1.0])
def test_mla_sparse_decisions_and_output(oracle_lib, shape, lam):
    """All Hq heads vote together; decisions follow the prefix-maximum form
    over the full key width and the output is the softmax over the kept
    tiles' keys with latent values."""
    B, Hq, Lk, dk, dl, S, Bk = shape
    nT = -(-Lk // Bk)
    T = -(-nT // S)
    (q, kv, scale), res = mla_case(oracle_lib, shape, lam, 12)
    for b in range(B):
        qq, kk = f64(q[b]), f64(kv[b])
        s = scale * (qq @ kk.T)
        for sp in range(S):
            tiles = list(range(sp * T, min(nT, (sp + 1) * T)))
            m_ref, c_ref = prefix_decisions(s, Bk, tiles, math.log(lam))
            np.testing.assert_array_equal(res.mask[b, tiles], m_ref)
            assert res.counts[b, sp] == (m_ref == 1).sum()
        keep = np.repeat(res.mask[b] == 0, Bk)[:Lk]
        ref = two_pass(qq, kk, kk[:, :dl], scale, np.broadcast_to(keep, (Hq, Lk)))
        np.testing.assert_allclose(res.o[b], ref, rtol=0, atol=1e-10)


# ------------------------------------------- prefill with wider keys than values
# Multi-head latent attention (BLASST summary, §Belangrijkste Bijdragen item 4)
# in its unabsorbed prefill form is attention whose query/key rows (latent
# non-rotary + rotary parts) are wider than the value rows: d_qk != d_v.
ASYM_SHAPES = [
    # B, Hq, Hkv, Lq, Lk, dk, dv, causal, Bq, Bk
    (1, 2, 2, 13, 29, 12, 8, True, 4, 4),
    (1, 2, 1, 9, 17, 6, 10, False, 4, 5),    # values wider than keys, MQA
    (1, 2, 2, 130, 260, 192, 128, True, 128, 128),  # the kernel's widths
]


def asym_case(oracle_lib, shape, lam, seed):
    B, Hq, Hkv, Lq, Lk, dk, dv, causal, Bq, Bk = shape
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(dk)
    u /= np.linalg.norm(u)
    q = rand_bits(rng, (B, Hq, Lq, dk), shift=3.0 * u)
    kx = rng.standard_normal((B, Hkv, Lk, dk))
    kx[rng.random((B, Hkv, Lk)) < 0.15] += 3.0 * u
    k = bf16_bits(kx)
    v = rand_bits(rng, (B, Hkv, Lk, dv))
    scale = 1.0 / math.sqrt(dk)
    res = oracle_lib.prefill(q, k, v, scale=scale, causal=causal, lam=lam, Bq=Bq, Bk=Bk)
    return (q, k, v, scale), res


@pytest.mark.parametrize("shape", ASYM_SHAPES)
def test_prefill_value_width_dense_equals_two_pass(oracle_lib, shape):
    """lambda = 0 with d_v != d_qk: o = softmax(scale q k^T) v over the
    visible keys, computed directly (numpy, fp64)."""
    B, Hq, Hkv, Lq, Lk, dk, dv, causal, Bq, Bk = shape
    (q, k, v, scale), res = asym_case(oracle_lib, shape, 0.0, 31)
    nqb = -(-Lq // Bq)
    assert res.o.shape == (B * Hq * nqb, Bq, dv)
    G = Hq // Hkv
    vis = visible(Lq, Lk, causal)
    for u in range(B * Hq * nqb):
        b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
        ref = two_pass(f64(q[b, h]), f64(k[b, h // G]), f64(v[b, h // G]), scale, vis)
        np.testing.assert_allclose(res.o[u, : r1 - r0], ref[r0:r1], rtol=0, atol=1e-10)


@pytest.mark.parametrize("shape", ASYM_SHAPES)
@pytest.mark.parametrize("lam", [0.05, 1.0])
def test_prefill_value_width_sparse(oracle_lib, shape, lam):
    """Decisions follow the prefix-maximum form over the key width alone (the
    values play no part in them), and the output is the softmax restricted to
    the kept tiles' keys with the dv-wide values."""
    B, Hq, Hkv, Lq, Lk, dk, dv, causal, Bq, Bk = shape
    (q, k, v, scale), res = asym_case(oracle_lib, shape, lam, 32)
    nqb, nT = -(-Lq // Bq), -(-Lk // Bk)
    G = Hq // Hkv
    vis = visible(Lq, Lk, causal)
    for u in range(B * Hq * nqb):
        b, h, r0, r1 = unit_rows(u, Hq, nqb, Bq, Lq)
        s = scale * (f64(q[b, h])[r0:r1] @ f64(k[b, h // G]).T)
        s = np.where(vis[r0:r1], s, -np.inf)
        m_ref, _ = prefix_decisions(s, Bk, range(nT), math.log(lam))
        np.testing.assert_array_equal(res.mask[u], m_ref)
        keep = np.repeat(res.mask[u] == 0, Bk)[:Lk]
        ref = two_pass(f64(q[b, h])[r0:r1], f64(k[b, h // G]), f64(v[b, h // G]), scale,
                       vis[r0:r1] & keep[None, :])
        np.testing.assert_allclose(res.o[u, : r1 - r0], ref, rtol=0, atol=1e-10)


# ------------------------------------------------------ worked examples
def _decode_scalar(vals):
    return np.array([math.inf if x == "inf" else x for x in vals], dtype=np.float64)


def _softmax_closed_form(keys, values, kept):
    num = sum(math.exp(keys[j]) * values[j] for j in kept)
    den = sum(math.exp(keys[j]) for j in kept)
    return num / den


def test_worked_example_prefill(oracle_lib):
    ex = json.load(open(GOLDEN))["prefill_three_tiles"]
    keys = np.array(ex["keys"], np.float32)
    q = bf16_bits(np.ones((1, 1, 1, 1)))
    k = bf16_bits(keys.reshape(1, 1, -1, 1))
    v = bf16_bits(np.array(ex["values"], np.float32).reshape(1, 1, -1, 1))
    for case in ex["cases"]:
        res = oracle_lib.prefill(q, k, v, scale=1.0, causal=False, lam=case["lambda"], Bq=1,
                                 Bk=ex["tile"])
        assert res.mask[0].tolist() == case["mask"]
        assert int(res.counts[0]) == case["skipped"]
        np.testing.assert_array_equal(res.margin[0], _decode_scalar(ex["margins"]))
        expect = _softmax_closed_form(ex["keys"], ex["values"], case["kept_keys"])
        assert abs(res.o[0, 0, 0] - expect) < 1e-13


def test_worked_example_decode_split_restart(oracle_lib):
    ex = json.load(open(GOLDEN))["decode_split_restart"]
    q = bf16_bits(np.ones((1, 1, 1)))
    k = bf16_bits(np.array(ex["keys"], np.float32).reshape(1, 1, -1, 1))
    v = bf16_bits(np.array(ex["values"], np.float32).reshape(1, 1, -1, 1))
    for key, S, margins in (("one_split", 1, ex["margins_one_split"]),
                            ("two_splits", ex["num_splits"], ex["margins_two_splits"])):
        res = oracle_lib.decode(q, k, v, scale=1.0, lam=ex["lambda"], num_splits=S, Bk=ex["tile"])
        assert res.mask[0].tolist() == ex[key]["mask"]
        assert res.counts[0].tolist() == ex[key]["skipped"]
        np.testing.assert_array_equal(res.margin[0], _decode_scalar(margins))
        expect = _softmax_closed_form(ex["keys"], ex["values"], ex[key]["kept_keys"])
        assert abs(res.o[0, 0, 0] - expect) < 1e-13


# ---------------------------------------------------------- calibration
@pytest.mark.parametrize("target", [0.0, 0.3, 0.5, 0.7, 0.9])
def test_calibration_skips_exactly_round_sN(oracle_lib, target):
    shape = (1, 4, 2, 64, 64, 8, True, 8, 4)
    B, Hq, Hkv, Lq, Lk, d, causal, Bq, Bk = shape
    (q, k, v, scale), res0 = run_prefill_case(oracle_lib, shape, 0.0, 8, hot=True)
    a, skipped, N = oracle_lib.calibrate(res0.margin, res0.mask, target, Lk)
    assert N == int((res0.mask != 2).sum())
    c = np.sort(res0.margin[res0.mask != 2])
    reach = int((c < 0).sum())  # tiles that lambda <= 1 can skip at all
    want = min(int(np.floor(target * N + 0.5)), reach)
    assert skipped == want
    lam = a / Lk if a > 0 else 0.0
    assert 0.0 <= lam <= 1.0
    _, res = run_prefill_case(oracle_lib, shape, lam, 8, hot=True)
    assert int(res.counts.sum()) == want
    if 0 < want < reach:  # strictly inside the plateau (c_(k), c_(k+1))
        assert c[want - 1] < math.log(lam) < c[want]


def test_calibration_rounds_half_up(oracle_lib):
    """k = round(s N), not floor(s N): a target whose s N has a fractional
    part of 3/4 (inside the reachable range) skips one tile more than the
    floor would."""
    shape = (1, 4, 2, 64, 64, 8, True, 8, 4)
    Lk = shape[4]
    _, res0 = run_prefill_case(oracle_lib, shape, 0.0, 8, hot=True)
    c = np.sort(res0.margin[res0.mask != 2])
    N, reach = c.size, int((c < 0).sum())
    k0 = reach // 2
    assert 1 <= k0 < reach - 1
    a, skipped, n_eval = oracle_lib.calibrate(res0.margin, res0.mask, (k0 + 0.75) / N, Lk)
    assert n_eval == N and skipped == k0 + 1
    assert c[k0] < math.log(a / Lk) < c[k0 + 1]


def test_synthetic_hot_tiles_are_the_kept_set(oracle_lib):
    """Tiny prefill workload: only the hot tiles survive at a in {1, 4}.

    Hot scores sit near 18 (scale 1/8 of 144), cold ones near 0, so the
    decision margins are about 12 nats on either side of ln(a/1024)."""
    from block_sparse_attention_sm_gb300 import synth

    inp, cfg = synth.make("tiny_prefill", seed=0)
    nT = 1024 // 128
    for a in (0.0, 1.0, 4.0):
        res = oracle_lib.prefill(inp.q, inp.k, inp.v, scale=cfg["scale"], causal=False,
                                 lam=a / 1024)
        if a == 0.0:
            assert res.counts.sum() == 0
            continue
        kept = res.mask == 0
        assert (kept == inp.hot[0, 0][None, :]).all()
        assert res.counts.sum() == 8 * (nT - 2)
        fin = np.isfinite(res.margin)
        assert (np.abs(res.margin[fin] - math.log(a / 1024)) > 2.0).all()


# ------------------------------------------------- readings at the boundary
def test_tie_keeps_the_tile(oracle_lib):
    """The comparison is strict: a tile whose maximum equals the running
    maximum has c_j = 0 exactly, and lambda = 1 (ln lambda = 0) keeps it.

    Tile 1 is a bit-for-bit copy of tile 0, so every row's tile maximum
    repeats its running maximum."""
    rng = np.random.default_rng(5)
    d, Bq, Bk = 4, 4, 4
    q = rand_bits(rng, (1, 1, 4, d))
    k0 = rand_bits(rng, (1, 1, 4, d))
    v = rand_bits(rng, (1, 1, 8, d))
    k = np.concatenate([k0, k0], axis=2)
    res = oracle_lib.prefill(q, k, v, scale=0.5, causal=False, lam=1.0, Bq=Bq, Bk=Bk)
    assert res.margin[0, 1] == 0.0
    assert res.mask[0].tolist() == [0, 0] and int(res.counts[0]) == 0
    ref = two_pass(f64(q[0, 0]), f64(k[0, 0]), f64(v[0, 0]), 0.5, visible(4, 8, False))
    np.testing.assert_allclose(res.o[0, :4], ref, rtol=0, atol=1e-12)
    # just below lambda = 1 the same tile is still kept (c_j = 0 > ln lambda is false)
    res2 = oracle_lib.prefill(q, k, v, scale=0.5, causal=False, lam=np.nextafter(1.0, 0.0),
                              Bq=Bq, Bk=Bk)
    assert res2.mask[0].tolist() == [0, 0]


def test_row_without_any_key_does_not_veto(oracle_lib):
    """Causal with Lq > Lk (bottom-right): rows 0-2 of the first block see no
    key at all; the other rows' votes alone decide each tile.

    Lq = 11, Lk = 8, Bq = 8, Bk = 2, offset Lk - Lq = -3: row r sees keys
    <= r - 3.  Every query is e1; keys 0-1 are 8 e1 (score 4 at scale 1/2),
    keys 2-7 are -8 e1 (score -4), so every later tile has c_j = -8 for the
    rows that see it.  At lambda = 0.01 (ln = -4.6) those tiles are skipped;
    tile 3 (keys 6, 7) is seen by no row of block 0: not evaluated."""
    d = 4
    q = np.zeros((1, 1, 11, d), np.float32)
    q[..., 0] = 1.0
    kx = np.zeros((1, 1, 8, d), np.float32)
    kx[..., :2, 0] = 8.0
    kx[..., 2:, 0] = -8.0
    rng = np.random.default_rng(6)
    v = rand_bits(rng, (1, 1, 8, d))
    res = oracle_lib.prefill(bf16_bits(q), bf16_bits(kx), v, scale=0.5, causal=True, lam=0.01,
                             Bq=8, Bk=2)
    assert res.mask[0].tolist() == [0, 1, 1, 2] and int(res.counts[0]) == 2
    assert res.mask[1].tolist() == [0, 1, 1, 1] and int(res.counts[1]) == 3
    np.testing.assert_allclose(res.margin[0, 1:3], [-8.0, -8.0], rtol=0, atol=1e-12)
    assert not res.o[0, :3].any()  # rows with no visible key return zeros
    # rows that kept only tile 0 average its two values (equal scores)
    vk = f64(v[0, 0])
    np.testing.assert_allclose(res.o[0, 4], 0.5 * (vk[0] + vk[1]), rtol=0, atol=1e-12)
