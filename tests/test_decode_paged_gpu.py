"""Paged, variable-length decode vs the fp64 oracle (GPU).

The cache is pages of 128 keys ([num_pages][Hkv][128][d]) reached through a
page table; each sequence has its own length, its own threshold
lambda_b = min(1, a / L_b) ("Skip-Softmax" §The threshold) and its own split
of its tiles.  The oracle sees each sequence's keys gathered back into a
contiguous [1][Hkv][L_b][d] slice (a copy, no arithmetic).  Unused pages and
the rows of a last page past the sequence end are filled with NaN: a kernel
that read them into a result would fail the comparison.
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


def make_paged(k, v, lens, spare_pages, seed):
    """Scatter each sequence's keys into shuffled pages; NaN elsewhere."""
    B, Hkv, _, d = k.shape
    n_used = sum(-(-L // 128) for L in lens)
    num_pages = n_used + spare_pages
    max_pages = max(1, max(-(-L // 128) for L in lens))
    rng = np.random.default_rng(seed)
    phys = rng.permutation(num_pages)
    nan = float("nan")
    kp = torch.full((num_pages, Hkv, 128, d), nan, dtype=k.dtype, device=k.device)
    vp = torch.full_like(kp, nan)
    # entries past a sequence's pages point at a page of another sequence:
    # they must not be read
    table = np.full((B, max_pages), int(phys[0]), dtype=np.int32)
    nxt = 0
    for b, L in enumerate(lens):
        for j in range(-(-L // 128)):
            pg = int(phys[nxt])
            nxt += 1
            rows = min(128, L - 128 * j)
            kp[pg, :, :rows] = k[b, :, 128 * j:128 * j + rows]
            vp[pg, :, :rows] = v[b, :, 128 * j:128 * j + rows]
            table[b, j] = pg
    return kp, vp, torch.from_numpy(table).to(k.device), num_pages, max_pages


def check_paged(q, k, v, lens, *, scale, a, num_splits, spare_pages=3, seed=0):
    import oracle
    from _parity import Parity, _finish, check_output, compare_decisions, guarded
    from block_sparse_attention_sm_gb300 import capi

    B, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    S = num_splits
    kp, vp, table, num_pages, max_pages = make_paged(k, v, lens, spare_pages, seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=q.device)
    ws_n = capi.ss_attn_decode_workspace_size(B, Hq, d, S)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=q.device)
    gbs = [guarded(q.shape, q.dtype, q.device, float("nan")),
           guarded((B * Hkv * S,), torch.int32, q.device, -1),
           guarded((B * Hkv, max_pages), torch.uint8, q.device, 7),
           guarded((B * Hkv, max_pages), torch.float32, q.device, 12345.0)]
    o, counts, mask, margin = (g.t for g in gbs)
    st = capi.ss_attn_decode_paged(q, kp, vp, table, seq_lens, o, B, Hq, Hkv, num_pages, max_pages,
                                   d, scale, a, S, counts, ws, ws_n, mask, margin)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    assert capi.ss_stream_status() == capi.SS_OK
    torch.cuda.synchronize()
    for g, what in zip(gbs, ("o", "skip_counts", "skip_mask", "vote_margin")):
        g.check(what)
    og = o.float().cpu().numpy()
    mh, gh = mask.cpu().numpy(), margin.cpu().numpy()
    ch = counts.cpu().numpy().reshape(B * Hkv, S)
    rec = Parity("decode_paged", a)
    for b, L in enumerate(lens):
        nT = -(-L // 128)
        T = -(-nT // S) if nT else 0
        lam = min(1.0, a / L) if (a > 0 and L > 0) else 0.0
        for kvh in range(Hkv):
            u = b * Hkv + kvh
            assert (mh[u, nT:] == 2).all(), "tiles past the sequence end must be 'not evaluated'"
            rows = og[b, kvh * G:(kvh + 1) * G]
            if L == 0:
                assert (ch[u] == 0).all()
                np.testing.assert_array_equal(rows, 0.0)
                continue
            qs = q[b:b + 1, kvh * G:(kvh + 1) * G]
            ks, vs = k[b:b + 1, kvh:kvh + 1, :L], v[b:b + 1, kvh:kvh + 1, :L]
            ref = oracle.decode(qs, ks, vs, scale=scale, lam=lam, num_splits=S)
            nd, row_dis = compare_decisions(mh[u:u + 1, :nT], gh[u:u + 1, :nT], ref.mask,
                                            ref.margin, lam)
            rec.units += 1
            rec.disagree += nd
            rec.add_decisions(mh[u:u + 1, :nT], ref.mask, ref.margin, lam)
            for sp in range(S):
                tiles = list(range(sp * T, min(nT, sp * T + T)))
                assert ch[u, sp] == (int((mh[u, tiles] == 1).sum()) if tiles else 0)
                if not row_dis[0]:
                    assert ch[u, sp] == ref.counts[0, sp]
            over = oracle.decode(qs, ks, vs, scale=scale, lam=lam, num_splits=S,
                                 mask_override=(mh[u:u + 1, :nT] == 1).astype(np.uint8))
            rec.add_error(check_output(rows, over.o[0], f"paged unit {u} under GPU mask"), False)
            if not row_dis[0]:
                rec.add_error(check_output(rows, ref.o[0], f"paged unit {u}"), True)
    return _finish(rec)


CASES = [
    # B, Hq, Hkv, d, lens, splits
    (5, 8, 2, 128, [1000, 0, 128, 129, 3000], 3),
    (3, 8, 2, 64, [700, 1, 5000], 1),
    (2, 16, 1, 128, [2500, 4096], 4),          # G = 16
    (4, 32, 8, 128, [333, 8191, 8192, 1], 8),  # Llama-shaped heads, ragged lengths
    (3, 32, 1, 128, [4000, 129, 2048], 2),     # G = 32 (MQA)
    (3, 64, 1, 128, [4000, 129, 2048], 2),     # G = 64 (MQA, heads as MMA rows)
    (2, 96, 2, 128, [1000, 2500], 3),          # G = 48
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("a", [0.0, 1.0, 8.0])
def test_paged_varlen(case, a):
    from _parity import hot_decode

    B, Hq, Hkv, d, lens, S = case
    Lmax = max(128, -(-max(lens) // 128) * 128)
    inp = hot_decode(B, Hq, Hkv, Lmax, d, frac=0.2, seed=21)
    check_paged(inp.q, inp.k, inp.v, lens, scale=1.0 / math.sqrt(d), a=a, num_splits=S, seed=5)


def test_paged_matches_contiguous_layout():
    """Equal lengths and pages in order: the paged kernel sees the same keys as
    the contiguous one, so with the same lambda both give the same decisions."""
    from _parity import hot_decode
    from block_sparse_attention_sm_gb300 import capi

    B, Hq, Hkv, d, L, S = 3, 8, 2, 128, 2048, 4
    inp = hot_decode(B, Hq, Hkv, L, d, frac=0.2, seed=3)
    nP = L // 128
    kp = inp.k.reshape(B, Hkv, nP, 128, d).permute(0, 2, 1, 3, 4).reshape(B * nP, Hkv, 128, d).contiguous()
    vp = inp.v.reshape(B, Hkv, nP, 128, d).permute(0, 2, 1, 3, 4).reshape(B * nP, Hkv, 128, d).contiguous()
    table = torch.arange(B * nP, dtype=torch.int32, device="cuda").reshape(B, nP)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    ws_n = capi.ss_attn_decode_workspace_size(B, Hq, d, S)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    a = 4.0
    o1, o2 = torch.empty_like(inp.q), torch.empty_like(inp.q)
    c1 = torch.zeros(B * Hkv * S, dtype=torch.int32, device="cuda")
    c2 = torch.zeros_like(c1)
    assert capi.ss_attn_decode_paged(inp.q, kp, vp, table, lens, o1, B, Hq, Hkv, B * nP, nP, d,
                                     d ** -0.5, a, S, c1, ws, ws_n) == capi.SS_OK
    assert capi.ss_attn_decode(inp.q, inp.k, inp.v, o2, B, Hq, Hkv, L, d, d ** -0.5, a / L, S, c2,
                               ws, ws_n) == capi.SS_OK
    assert capi.ss_stream_status() == capi.SS_OK
    # The per-sequence threshold is formed on the device in fp32, the
    # contiguous one on the host in fp64: the decisions may differ only on
    # tiles at the threshold, which these inputs do not have.
    assert torch.equal(c1, c2)
    diff = (o1.float() - o2.float()).abs().max().item()
    assert diff <= 1e-6, diff


@pytest.mark.slow
def test_paged_full_size_sampled():
    """The bench's paged workload (64 sequences of 8K..32K keys in shuffled
    pages, 8 splits) at the a calibrated for 70% on the contiguous cache, in
    one launch; the oracle checks every sequence."""
    import block_sparse_attention_sm_gb300 as ss
    from block_sparse_attention_sm_gb300 import synth

    B, Hq, Hkv, d, S, Lmax = 64, 32, 8, 128, 8, 32768
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(8192, Lmax + 1, size=B)]
    inp = synth.decode_inputs(B=B, Hq=Hq, Hkv=Hkv, Lk=Lmax, d=d, hot_frac=0.10, seed=0,
                              device="cuda")
    a, _ = ss.calibrate("decode", inp.q, inp.k, inp.v, scale=d ** -0.5, target_sparsity=0.7,
                        num_kv_splits=S)
    check_paged(inp.q, inp.k, inp.v, lens, scale=d ** -0.5, a=a, num_splits=S, seed=11)
