"""Latent-attention (MLA) decode vs the fp64 oracle (GPU).

The keys are the 576-entry latent cache rows (512 latent + 64 rotary
entries), the values their latent part, and all query heads of a sequence
vote together on each tile (BLASST summary, §Belangrijkste Bijdragen item 4:
MLA listed beside MHA, GQA and MQA among the attention kinds the kernels
support; the absorbed-form reading is the oracle's).
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
    # 17..32 heads: two softmax warpgroups of 16 heads each
    (2, 17, 1000, 1),     # one head in the second warpgroup
    (3, 24, 5000, 3),     # heads padded to the MMA's 32 rows
    (2, 32, 4096, 8),     # both warpgroups full
    (1, 32, 20000, 2),    # long splits
    # 33..64 heads: heads as the MMA rows, O's latent entries over two CTAs
    (2, 33, 1000, 1),     # ragged last tile, one split (no merge)
    (3, 48, 5000, 3),     # several splits
    (2, 64, 4096, 8),     # every row of the staged query block
    (1, 64, 300, 5),      # more splits than tiles: empty splits
    (1, 40, 20000, 2),    # long splits: the copy ring wraps many times
    (1, 48, 1, 2),        # a single key (the second split is empty)
    (2, 24, 1, 1),        # a single key, two softmax warpgroups
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("a", [0.0, 1.0, 8.0])
def test_mla_decode(case, a):
    from _parity import check_mla

    B, Hq, Lk, S = case
    inp = _inputs(B, Hq, Lk, seed=4)
    check_mla(inp.q, inp.kv, scale=SCALE, lam=min(1.0, a / Lk), num_splits=S)


@pytest.mark.parametrize("Hq", [16, 32, 64])
def test_mla_random_scores_many_decisions(Hq):
    """Plain N(0,1) inputs: margins spread out around the threshold."""
    from _parity import check_mla

    g = torch.Generator(device="cuda").manual_seed(8)
    q = torch.randn(2, Hq, 576, device="cuda", generator=g).to(torch.bfloat16)
    kv = torch.randn(2, 3000, 576, device="cuda", generator=g).to(torch.bfloat16)
    for lam in (0.3, 0.8):
        check_mla(q, kv, scale=576 ** -0.5, lam=lam, num_splits=3)


@pytest.mark.parametrize("Hq", [16, 32, 64])
def test_mla_count_only_matches_the_full_launch(Hq):
    from block_sparse_attention_sm_gb300 import capi

    B, Lk, S = 4, 8192, 4
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
@pytest.mark.parametrize("name", ["mla_decode_32k", "mla_decode_32k_32h", "mla_decode_32k_64h"])
def test_mla_full_size_sampled(name):
    """The bench's workloads (128 sequences x 32K keys, 4 splits, 16 or 32
    heads) at lambda for 70% skipped tiles; the oracle checks the first, last
    and two random sequences."""
    import block_sparse_attention_sm_gb300 as ss
    from _parity import check_mla
    from block_sparse_attention_sm_gb300 import synth

    inp, cfg = synth.make(name, seed=0, device="cuda")
    a, _ = ss.calibrate("mla_decode", inp.q, inp.kv, None, scale=cfg["scale"], target_sparsity=0.7,
                        num_kv_splits=cfg["num_splits"])
    rng = np.random.default_rng(3)
    units = sorted({0, cfg["B"] - 1, *rng.choice(cfg["B"], size=2, replace=False).tolist()})
    check_mla(inp.q, inp.kv, scale=cfg["scale"], lam=min(1.0, a / cfg["Lk"]),
              num_splits=cfg["num_splits"], units=units)


def check_mla_paged(q, kv, lens, *, a, num_splits, spare_pages=3, seed=0):
    """Scatter each sequence's rows into shuffled pages of 128 (NaN in every
    unused page and in the rows past a sequence's end) and compare each
    sequence with the oracle on its own rows."""
    import oracle
    from _parity import Parity, _finish, check_output, compare_decisions, guarded
    from block_sparse_attention_sm_gb300 import capi

    B, Hq, dk = q.shape
    S = num_splits
    n_used = sum(-(-L // 128) for L in lens)
    num_pages = n_used + spare_pages
    max_pages = max(1, max(-(-L // 128) for L in lens))
    rng = np.random.default_rng(seed)
    phys = rng.permutation(num_pages)
    pages = torch.full((num_pages, 128, dk), float("nan"), dtype=kv.dtype, device=kv.device)
    table = np.full((B, max_pages), int(phys[0]), dtype=np.int32)
    nxt = 0
    for b, L in enumerate(lens):
        for j in range(-(-L // 128)):
            pg = int(phys[nxt])
            nxt += 1
            rows = min(128, L - 128 * j)
            pages[pg, :rows] = kv[b, 128 * j:128 * j + rows]
            table[b, j] = pg
    table_t = torch.from_numpy(table).to(q.device)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=q.device)
    ws_n = capi.ss_attn_mla_decode_workspace_size(B, Hq, 512, S)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=q.device)
    gbs = [guarded((B, Hq, 512), q.dtype, q.device, float("nan")),
           guarded((B * S,), torch.int32, q.device, -1),
           guarded((B, max_pages), torch.uint8, q.device, 7),
           guarded((B, max_pages), torch.float32, q.device, 12345.0)]
    o, counts, mask, margin = (g.t for g in gbs)
    st = capi.ss_attn_mla_decode_paged(q, pages, table_t, lens_t, o, B, Hq, num_pages, max_pages,
                                       512, dk - 512, SCALE, a, S, counts, ws, ws_n, mask, margin)
    assert st == capi.SS_OK, capi.ss_status_string(st)
    assert capi.ss_stream_status() == capi.SS_OK
    torch.cuda.synchronize()
    for g, what in zip(gbs, ("o", "skip_counts", "skip_mask", "vote_margin")):
        g.check(what)
    rec = Parity("mla_decode_paged", a)
    og = o.float().cpu().numpy()
    mh, gh = mask.cpu().numpy(), margin.cpu().numpy()
    ch = counts.cpu().numpy().reshape(B, S)
    for b, L in enumerate(lens):
        nT = -(-L // 128)
        assert (mh[b, nT:] == 2).all(), "tiles past the sequence end must be 'not evaluated'"
        if L == 0:
            assert (ch[b] == 0).all()
            np.testing.assert_array_equal(og[b], 0.0)
            continue
        lam = min(1.0, a / L) if a > 0 else 0.0
        T = -(-nT // S)
        qs, kvs = q[b:b + 1], kv[b:b + 1, :L]
        ref = oracle.mla_decode(qs, kvs, d_latent=512, scale=SCALE, lam=lam, num_splits=S)
        nd, row_dis = compare_decisions(mh[b:b + 1, :nT], gh[b:b + 1, :nT], ref.mask, ref.margin,
                                        lam)
        rec.units += 1
        rec.disagree += nd
        rec.add_decisions(mh[b:b + 1, :nT], ref.mask, ref.margin, lam)
        for sp in range(S):
            tiles = list(range(sp * T, min(nT, sp * T + T)))
            assert ch[b, sp] == (int((mh[b, tiles] == 1).sum()) if tiles else 0)
            if not row_dis[0]:
                assert ch[b, sp] == ref.counts[0, sp]
        over = oracle.mla_decode(qs, kvs, d_latent=512, scale=SCALE, lam=lam, num_splits=S,
                                 mask_override=(mh[b:b + 1, :nT] == 1).astype(np.uint8))
        rec.add_error(check_output(og[b], over.o[0], f"paged mla sequence {b} under GPU mask"),
                      False)
        if not row_dis[0]:
            rec.add_error(check_output(og[b], ref.o[0], f"paged mla sequence {b}"), True)
    return _finish(rec)


PAGED = [
    # B, Hq, lens, splits
    (4, 16, [1000, 0, 129, 3000], 3),   # ragged, an empty sequence, one row past a page
    (3, 12, [128, 5000, 1], 2),
    (2, 16, [4096, 2500], 1),
    (3, 32, [1000, 0, 3000], 3),        # two softmax warpgroups
    (2, 20, [129, 4096], 2),
    (3, 64, [1000, 0, 3000], 3),        # heads as MMA rows, two CTAs per split
    (2, 36, [129, 4096], 2),
]


@pytest.mark.parametrize("case", PAGED)
@pytest.mark.parametrize("a", [0.0, 1.0, 8.0])
def test_mla_paged(case, a):
    B, Hq, lens, S = case
    Lmax = max(128, -(-max(lens) // 128) * 128)
    inp = _inputs(B, Hq, Lmax, seed=6)
    check_mla_paged(inp.q, inp.kv, lens, a=a, num_splits=S, seed=4)
