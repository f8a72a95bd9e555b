"""Shared comparison logic for the GPU-vs-oracle parity tests.

Acceptance (per unit):
* skip decisions agree bit-exactly except on "near-margin" tiles, where the
  oracle's vote statistic c_j lies within 1e-2 (natural log) of ln(lambda);
  those disagreements are counted and returned, not failed;
* skipped-tile counts agree exactly on units whose decisions all agree, and
  always equal the number of skipped tiles in the GPU's own mask;
* outputs agree within max-abs 2e-2 and mean-abs 2e-3 (bf16 output), both
  against the oracle with its own decisions (units without disagreement) and
  against the oracle re-run under the GPU's decisions (arithmetic only).

Every check returns a `Parity` record (units, evaluated tiles, near-margin
tiles, disagreements, errors) and appends it to `LOG`; conftest.py prints the
session's records and totals at the end of the run, so the near-margin
disagreements are reported, not only tolerated.

Every output the kernels write (o, counters, skip mask, vote margins) sits in
a buffer with a guard band of GUARD_BYTES on each side, filled with the byte
GUARD_BYTE; after each call the bands must be intact.  This is the bounds
check of the outputs (a store one element past the end, or before the start,
of any output fails the test).
"""
from __future__ import annotations

import dataclasses
import math
import os

import numpy as np
import torch

import oracle
from block_sparse_attention_sm_gb300 import capi, synth

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
NEAR_MARGIN = 1e-2
TILE = 128
GUARD_BYTES = 256  # keeps the guarded view 256-byte aligned
GUARD_BYTE = 0xA5


@dataclasses.dataclass
class Parity:
    """Outcome of one parity check (one launch, the sampled units of it)."""
    kind: str
    lam: float
    units: int = 0
    tiles: int = 0          # evaluated (unit, tile) pairs compared
    skipped: int = 0        # tiles the GPU skipped among them
    near: int = 0           # of which the oracle's |c_j - ln lambda| < NEAR_MARGIN
    disagree: int = 0       # decisions that differ (all of them near-margin)
    max_abs: float = 0.0    # output error against the oracle's own decisions
    mean_abs: float = 0.0
    max_abs_gpu_mask: float = 0.0  # against the oracle run under the GPU's decisions
    test: str = ""

    def add_decisions(self, gmask, omask, omargin, lam):
        ev = omask != 2
        self.tiles += int(ev.sum())
        self.skipped += int((gmask == 1).sum())
        self.near += int((ev & (np.abs(omargin - _ln(lam)) < NEAR_MARGIN)).sum())

    def add_error(self, err, own_mask: bool):
        if own_mask:
            self.max_abs = max(self.max_abs, err[0])
            # mean over units, weighted equally (each unit's mean is bounded)
            self.mean_abs = max(self.mean_abs, err[1])
        else:
            self.max_abs_gpu_mask = max(self.max_abs_gpu_mask, err[0])


LOG: list[Parity] = []


def _finish(rec: Parity) -> Parity:
    rec.test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    LOG.append(rec)
    return rec


class Guarded:
    """A device tensor of `shape` inside a buffer with guard bands."""

    def __init__(self, shape, dtype, device, fill):
        self.n = int(np.prod(shape)) if len(shape) else 1
        item = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // item
        self.buf = torch.empty(self.n + 2 * self.g, dtype=dtype, device=device)
        self.buf.view(torch.uint8).fill_(GUARD_BYTE)
        self.t = self.buf[self.g:self.g + self.n].view(shape)
        self.t.fill_(fill)

    def check(self, what):
        raw = self.buf.view(torch.uint8)
        nb = self.g * self.buf.element_size()
        head, tail = raw[:nb], raw[raw.numel() - nb:]
        assert bool((head == GUARD_BYTE).all()), f"{what}: write before the start of the output"
        assert bool((tail == GUARD_BYTE).all()), f"{what}: write past the end of the output"


def guarded(shape, dtype, device, fill):
    return Guarded(tuple(shape), dtype, device, fill)


def _ln(lam):
    return math.log(lam) if lam > 0 else -math.inf


def compare_decisions(gpu_mask, gpu_margin, orc_mask, orc_margin, lam):
    """Returns (n_disagree, per-row disagreement flags); asserts the rest."""
    ln_lam = _ln(lam)
    gm = gpu_mask.astype(np.int64)
    om = orc_mask.astype(np.int64)
    # "not evaluated" must agree exactly (pure index arithmetic).
    assert np.array_equal(gm == 2, om == 2), "evaluated-tile sets differ"
    dis = gm != om
    near = np.abs(orc_margin - ln_lam) < NEAR_MARGIN
    bad = dis & ~near
    assert not bad.any(), (
        f"{int(bad.sum())} decision(s) disagree outside the {NEAR_MARGIN} log margin; "
        f"first at {np.argwhere(bad)[0].tolist()} margin {orc_margin[bad][0]} ln(lam) {ln_lam}")
    # vote statistic itself: +inf where the oracle has +inf, close elsewhere
    ev = om != 2
    inf_o = np.isposinf(orc_margin) & ev
    assert np.array_equal(np.isposinf(gpu_margin) & ev, inf_o), "first-tile (+inf) margins differ"
    fin = ev & ~inf_o
    if fin.any():
        err = np.abs(gpu_margin[fin].astype(np.float64) - orc_margin[fin])
        assert err.max() <= 2e-2 + 2e-4 * np.abs(orc_margin[fin]).max(), f"margin error {err.max()}"
    return int(dis.sum()), dis.any(axis=-1)


def check_output(o_gpu, o_ref, what=""):
    o_gpu = o_gpu.astype(np.float64)
    err = np.abs(o_gpu - o_ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean


def gpu_prefill_all(q, k, v, scale, causal, lam, chunk=0, kernel=0):
    """Bench-configuration call (plain entry point) plus the debug call.

    chunk > 0: both calls use the debug entry point with that vote-run length
    (test-only option), so that short inputs take the multi-run path.
    kernel > 0: both calls use the debug entry point with that prefill kernel
    (test-only option: 1 the one-CTA kernel, 2 the CTA-pair kernel)."""
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    dv = v.shape[-1]  # != d: latent-attention prefill (its own entry point)
    nqb, nT = -(-Lq // TILE), -(-Lk // TILE)
    n_units = B * Hq * nqb
    dev = q.device
    oshape = (B, Hq, Lq, dv)
    og = guarded(oshape, q.dtype, dev, float("nan"))
    cg = guarded((n_units,), torch.int32, dev, -1)
    o, counts = og.t, cg.t
    if dv != d:
        assert chunk == 0
        st = capi.ss_attn_mla_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, dv, scale, causal, lam,
                                      counts)
    elif chunk == 0 and kernel == 0:
        st = capi.ss_attn_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam, counts)
    else:
        st = capi.ss_attn_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam,
                                     counts, vote_chunk_tiles=chunk, prefill_kernel=kernel)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    o2g = guarded(oshape, q.dtype, dev, float("nan"))
    c2g = guarded((n_units,), torch.int32, dev, -1)
    mg = guarded((n_units, nT), torch.uint8, dev, 7)
    gg = guarded((n_units, nT), torch.float32, dev, 12345.0)
    o2, counts2, mask, margin = o2g.t, c2g.t, mg.t, gg.t
    if dv != d:
        st = capi.ss_attn_mla_prefill_ex(q, k, v, o2, B, Hq, Hkv, Lq, Lk, d, dv, scale, causal,
                                         lam, counts2, mask, margin)
    else:
        st = capi.ss_attn_prefill_ex(q, k, v, o2, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam,
                                     counts2, mask, margin, vote_chunk_tiles=chunk,
                                     prefill_kernel=kernel)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    assert capi.ss_stream_status() == capi.SS_OK
    torch.cuda.synchronize()
    for gb, what in ((og, "o"), (cg, "skip_counts"), (o2g, "o (debug call)"),
                     (c2g, "skip_counts (debug call)"), (mg, "skip_mask"), (gg, "vote_margin")):
        gb.check(what)
    # The debug outputs do not change the result.  (lambda = 0 with debug
    # outputs runs the voting kernel with nothing skipped instead of the
    # dense kernel: the same values up to rounding.)
    assert torch.equal(counts, counts2)
    if lam > 0 or chunk > 0:
        assert torch.equal(o, o2)
    else:
        diff = (o.float() - o2.float()).abs()
        assert float(diff.max()) <= MAX_ABS and float(diff.mean()) <= MEAN_ABS
    return o, counts, mask, margin


def check_prefill(q, k, v, *, scale, causal, lam, units=None, chunk=0, kernel=0) -> Parity:
    """Parity of one prefill launch; `units` = list of (b, h, qb) or None (all)."""
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    G = Hq // Hkv
    nqb = -(-Lq // TILE)
    o, counts, mask, margin = gpu_prefill_all(q, k, v, scale, causal, lam, chunk, kernel)
    if units is None:
        units = [(b, h, qb) for b in range(B) for h in range(Hq) for qb in range(nqb)]
    by_head = {}
    for (b, h, qb) in units:
        by_head.setdefault((b, h), []).append(qb)
    rec = Parity("prefill" if v.shape[-1] == d else "mla_prefill", lam)
    counts_h = counts.cpu().numpy()
    mask_h = mask.cpu().numpy()
    margin_h = margin.cpu().numpy()
    for (b, h), qbs in sorted(by_head.items()):
        kvh = h // G
        qs, ks, vs = q[b:b + 1, h:h + 1], k[b:b + 1, kvh:kvh + 1], v[b:b + 1, kvh:kvh + 1]
        ref = oracle.prefill(qs, ks, vs, scale=scale, causal=causal, lam=lam, units=qbs)
        gids = [(b * Hq + h) * nqb + qb for qb in qbs]
        gmask, gmargin = mask_h[gids], margin_h[gids]
        nd, row_dis = compare_decisions(gmask, gmargin, ref.mask, ref.margin, lam)
        rec.units += len(qbs)
        rec.disagree += nd
        rec.add_decisions(gmask, ref.mask, ref.margin, lam)
        np.testing.assert_array_equal(counts_h[gids], (gmask == 1).sum(axis=1))
        for i, qb in enumerate(qbs):
            if not row_dis[i]:
                assert counts_h[gids[i]] == ref.counts[i]
        over = oracle.prefill(qs, ks, vs, scale=scale, causal=causal, lam=lam, units=qbs,
                              mask_override=(gmask == 1).astype(np.uint8))
        og = o[b, h].float().cpu().numpy()
        for i, qb in enumerate(qbs):
            r0, r1 = qb * TILE, min(Lq, qb * TILE + TILE)
            rec.add_error(check_output(og[r0:r1], over.o[i, : r1 - r0],
                                       f"unit {(b, h, qb)} under GPU mask"), False)
            if not row_dis[i]:
                rec.add_error(check_output(og[r0:r1], ref.o[i, : r1 - r0], f"unit {(b, h, qb)}"),
                              True)
    return _finish(rec)


def check_decode(q, k, v, *, scale, lam, num_splits, units=None) -> Parity:
    """Parity of one decode launch; `units` = list of b*Hkv + kvh (None: all)."""
    B, Hq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    G = Hq // Hkv
    nT = -(-Lk // TILE)
    S = num_splits
    dev = q.device
    ws_n = capi.ss_attn_decode_workspace_size(B, Hq, d, S)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    og = guarded(q.shape, q.dtype, dev, float("nan"))
    cg = guarded((B * Hkv * S,), torch.int32, dev, -1)
    o, counts = og.t, cg.t
    st = capi.ss_attn_decode(q, k, v, o, B, Hq, Hkv, Lk, d, scale, lam, S, counts, ws, ws_n)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    o2g = guarded(q.shape, q.dtype, dev, float("nan"))
    c2g = guarded((B * Hkv * S,), torch.int32, dev, -1)
    mg = guarded((B * Hkv, nT), torch.uint8, dev, 7)
    gg = guarded((B * Hkv, nT), torch.float32, dev, 12345.0)
    o2, counts2, mask, margin = o2g.t, c2g.t, mg.t, gg.t
    st = capi.ss_attn_decode_ex(q, k, v, o2, B, Hq, Hkv, Lk, d, scale, lam, S, counts2, ws, ws_n,
                                mask, margin)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    assert capi.ss_stream_status() == capi.SS_OK
    torch.cuda.synchronize()
    for gb, what in ((og, "o"), (cg, "skip_counts"), (o2g, "o (debug call)"),
                     (c2g, "skip_counts (debug call)"), (mg, "skip_mask"), (gg, "vote_margin")):
        gb.check(what)
    assert torch.equal(o, o2) and torch.equal(counts, counts2)
    if units is None:
        units = list(range(B * Hkv))
    units = sorted(units)
    ch = counts.cpu().numpy().reshape(B * Hkv, S)
    mh = mask.cpu().numpy()
    gh = margin.cpu().numpy()
    og_h = o.float().cpu().numpy()
    T = -(-nT // S)
    rec = Parity("decode", lam)
    for u in units:
        b, kvh = divmod(u, Hkv)
        qs = q[b:b + 1, kvh * G:(kvh + 1) * G]
        ks, vs = k[b:b + 1, kvh:kvh + 1], v[b:b + 1, kvh:kvh + 1]
        ref = oracle.decode(qs, ks, vs, scale=scale, lam=lam, num_splits=S)
        nd, row_dis = compare_decisions(mh[u:u + 1], gh[u:u + 1], ref.mask, ref.margin, lam)
        rec.units += 1
        rec.disagree += nd
        rec.add_decisions(mh[u:u + 1], ref.mask, ref.margin, lam)
        for sp in range(S):
            tiles = range(sp * T, min(nT, sp * T + T))
            gsk = int((mh[u, list(tiles)] == 1).sum()) if len(tiles) else 0
            assert ch[u, sp] == gsk
            if not row_dis[0]:
                assert ch[u, sp] == ref.counts[0, sp]
        over = oracle.decode(qs, ks, vs, scale=scale, lam=lam, num_splits=S,
                             mask_override=(mh[u:u + 1] == 1).astype(np.uint8))
        rec.add_error(check_output(og_h[b, kvh * G:(kvh + 1) * G], over.o[0],
                                   f"decode unit {u} under GPU mask"), False)
        if not row_dis[0]:
            rec.add_error(check_output(og_h[b, kvh * G:(kvh + 1) * G], ref.o[0],
                                       f"decode unit {u}"), True)
    return _finish(rec)


def check_mla(q, kv, *, scale, lam, num_splits, units=None, d_latent=512) -> Parity:
    """Parity of one latent-attention decode launch; `units` = sequences."""
    B, Hq, dk = q.shape
    Lk = kv.shape[1]
    nT = -(-Lk // TILE)
    S = num_splits
    dev = q.device
    ws_n = capi.ss_attn_mla_decode_workspace_size(B, Hq, d_latent, S)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    og = guarded((B, Hq, d_latent), q.dtype, dev, float("nan"))
    cg = guarded((B * S,), torch.int32, dev, -1)
    o, counts = og.t, cg.t
    st = capi.ss_attn_mla_decode(q, kv, o, B, Hq, Lk, d_latent, dk - d_latent, scale, lam, S,
                                 counts, ws, ws_n)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    o2g = guarded((B, Hq, d_latent), q.dtype, dev, float("nan"))
    c2g = guarded((B * S,), torch.int32, dev, -1)
    mg = guarded((B, nT), torch.uint8, dev, 7)
    gg = guarded((B, nT), torch.float32, dev, 12345.0)
    o2, counts2, mask, margin = o2g.t, c2g.t, mg.t, gg.t
    st = capi.ss_attn_mla_decode_ex(q, kv, o2, B, Hq, Lk, d_latent, dk - d_latent, scale, lam, S,
                                    counts2, ws, ws_n, mask, margin)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    assert capi.ss_stream_status() == capi.SS_OK
    torch.cuda.synchronize()
    for gb, what in ((og, "o"), (cg, "skip_counts"), (o2g, "o (debug call)"),
                     (c2g, "skip_counts (debug call)"), (mg, "skip_mask"), (gg, "vote_margin")):
        gb.check(what)
    if lam > 0:
        assert torch.equal(o, o2) and torch.equal(counts, counts2)
    else:  # the plain call runs the dense kernel, the debug call the voting one
        assert torch.equal(counts, counts2)
        check_output(o.float().cpu().numpy(), o2.double().cpu().numpy(), "dense vs voting kernel")
    units = sorted(range(B) if units is None else units)
    ch = counts.cpu().numpy().reshape(B, S)
    mh, gh = mask.cpu().numpy(), margin.cpu().numpy()
    og_h = o.float().cpu().numpy()
    T = -(-nT // S)
    rec = Parity("mla_decode", lam)
    for b in units:
        qs, kvs = q[b:b + 1], kv[b:b + 1]
        ref = oracle.mla_decode(qs, kvs, d_latent=d_latent, scale=scale, lam=lam, num_splits=S)
        nd, row_dis = compare_decisions(mh[b:b + 1], gh[b:b + 1], ref.mask, ref.margin, lam)
        rec.units += 1
        rec.disagree += nd
        rec.add_decisions(mh[b:b + 1], ref.mask, ref.margin, lam)
        for sp in range(S):
            tiles = list(range(sp * T, min(nT, sp * T + T)))
            assert ch[b, sp] == (int((mh[b, tiles] == 1).sum()) if tiles else 0)
            if not row_dis[0]:
                assert ch[b, sp] == ref.counts[0, sp]
        over = oracle.mla_decode(qs, kvs, d_latent=d_latent, scale=scale, lam=lam, num_splits=S,
                                 mask_override=(mh[b:b + 1] == 1).astype(np.uint8))
        rec.add_error(check_output(og_h[b], over.o[0], f"mla sequence {b} under GPU mask"), False)
        if not row_dis[0]:
            rec.add_error(check_output(og_h[b], ref.o[0], f"mla sequence {b}"), True)
    return _finish(rec)


def hot_prefill(B, Hq, Hkv, Lq, Lk, d, frac=0.2, seed=0, per_head_u=True):
    inp = synth.prefill_inputs(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=d, hot_frac=frac, seed=seed,
                               per_head_u=per_head_u, device="cuda")
    return inp


def hot_decode(B, Hq, Hkv, Lk, d, frac=0.2, seed=0):
    return synth.decode_inputs(B=B, Hq=Hq, Hkv=Hkv, Lk=Lk, d=d, hot_frac=frac, seed=seed,
                               device="cuda")
