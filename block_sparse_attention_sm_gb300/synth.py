"""Seeded synthetic inputs with the hot-tile structure skip-softmax exploits.

The "Skip-Softmax" design doc (§Motivation) observes that in long attention
rows the softmax weight concentrates on a small fraction of keys.  These
generators build that structure on purpose, with no trained model:

* a unit direction ``u`` (fp64, from the seed; one for all heads, or one per
  KV head shared by its query heads);
* queries ``Q = bf16(z + 12 u)``;
* keys in "hot" tiles ``K = bf16(z + 12 u)``, all other keys ``K = bf16(z)``;
  tile 0 (an attention sink) is always hot, plus ``round(f * (nT - 1))`` tiles
  drawn without replacement from the rest, per (batch, KV head);
* values ``V = bf16(z)``;

with ``z ~ N(0, 1)`` drawn by ``torch.randn`` from a generator seeded per
tensor, on the device the tensors live on.  Nothing here computes attention.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

TILE = 128
HOT_SHIFT = 12.0


@dataclass
class Inputs:
    q: torch.Tensor          # prefill [B,Hq,Lq,d] / decode [B,Hq,d], bf16
    k: torch.Tensor          # [B,Hkv,Lk,d] bf16
    v: torch.Tensor          # [B,Hkv,Lk,dv] bf16 (dv = d except for latent-attention prefill)
    hot: np.ndarray          # [B,Hkv,nT] bool: which key tiles were made hot
    u: np.ndarray            # [Hkv,d] fp64 unit directions


def hot_tiles(seed: int, B: int, Hkv: int, nT: int, frac: float) -> np.ndarray:
    """Tile 0 plus round(frac*(nT-1)) seeded distinct tiles from 1..nT-1."""
    n_extra = int(np.floor(frac * (nT - 1) + 0.5))
    hot = np.zeros((B, Hkv, nT), dtype=bool)
    for b in range(B):
        for h in range(Hkv):
            rng = np.random.default_rng([seed, 1, b, h])
            hot[b, h, 0] = True
            if n_extra > 0:
                hot[b, h, 1 + rng.permutation(nT - 1)[:n_extra]] = True
    return hot


def directions(seed: int, Hkv: int, d: int, per_head: bool) -> np.ndarray:
    """Unit vectors u (fp64): one per KV head, or one shared by all heads."""
    out = np.zeros((Hkv, d), np.float64)
    for h in range(Hkv):
        rng = np.random.default_rng([seed, 2, h if per_head else 0])
        x = rng.standard_normal(d)
        out[h] = x / np.linalg.norm(x)
    return out


def _randn(shape, seed: int, tensor_id: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + tensor_id)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _keys_values(seed, B, Hkv, Lk, d, hot, u, device, shift, dv=None):
    nT = -(-Lk // TILE)
    dv = d if dv is None else dv
    k = torch.empty((B, Hkv, Lk, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((B, Hkv, Lk, dv), dtype=torch.bfloat16, device=device)
    ut = torch.as_tensor(u, dtype=torch.float32, device=device)
    for b in range(B):  # per batch entry keeps the fp32 temporaries small
        kb = _randn((Hkv, Lk, d), seed * 100003 + b, 1, device)
        for h in range(Hkv):
            tiles = np.nonzero(hot[b, h])[0]
            rows = (tiles[:, None] * TILE + np.arange(TILE)[None, :]).ravel()
            rows = rows[rows < Lk]
            idx = torch.as_tensor(rows, device=device)
            kb[h].index_add_(0, idx, (shift * ut[h]).expand(len(rows), d))
        k[b] = kb.to(torch.bfloat16)
        del kb
        v[b] = _randn((Hkv, Lk, dv), seed * 100003 + b, 2, device).to(torch.bfloat16)
    assert hot.shape[2] == nT
    return k, v


def prefill_inputs(*, B, Hq, Hkv, Lq, Lk, d, hot_frac, seed=0, per_head_u=False,
                   device="cpu", shift=HOT_SHIFT, dv=None) -> Inputs:
    """Prefill tensors q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv] (dv = d
    unless given) in bf16 on `device`."""
    G = Hq // Hkv
    nT = -(-Lk // TILE)
    hot = hot_tiles(seed, B, Hkv, nT, hot_frac)
    u = directions(seed, Hkv, d, per_head_u)
    ut = torch.as_tensor(u, dtype=torch.float32, device=device)
    q = torch.empty((B, Hq, Lq, d), dtype=torch.bfloat16, device=device)
    for b in range(B):
        qb = _randn((Hq, Lq, d), seed * 100003 + b, 0, device)
        qb += shift * ut.repeat_interleave(G, dim=0)[:, None, :]
        q[b] = qb.to(torch.bfloat16)
        del qb
    k, v = _keys_values(seed, B, Hkv, Lk, d, hot, u, device, shift, dv)
    return Inputs(q, k, v, hot, u)


def decode_inputs(*, B, Hq, Hkv, Lk, d, hot_frac, seed=0, per_head_u=True, device="cpu",
                  shift=HOT_SHIFT) -> Inputs:
    """Decode tensors q [B,Hq,d] (one token per sequence), k/v [B,Hkv,Lk,d]."""
    G = Hq // Hkv
    nT = -(-Lk // TILE)
    hot = hot_tiles(seed, B, Hkv, nT, hot_frac)
    u = directions(seed, Hkv, d, per_head_u)
    ut = torch.as_tensor(u, dtype=torch.float32, device=device)
    q = _randn((B, Hq, d), seed * 100003, 3, device)
    q += shift * ut.repeat_interleave(G, dim=0)[None, :, :]
    q = q.to(torch.bfloat16)
    k, v = _keys_values(seed, B, Hkv, Lk, d, hot, u, device, shift)
    return Inputs(q, k, v, hot, u)


@dataclass
class MlaInputs:
    q: torch.Tensor          # [B,Hq,dk] bf16, dk = d_latent + d_rope
    kv: torch.Tensor         # [B,Lk,dk] bf16: latent part, then rotary part
    hot: np.ndarray          # [B,1,nT] bool
    u: np.ndarray            # [1,dk] fp64


def mla_decode_inputs(*, B, Hq, Lk, d_latent=512, d_rope=64, hot_frac, seed=0, device="cpu",
                      shift=HOT_SHIFT) -> MlaInputs:
    """Latent-attention decode: q [B,Hq,dk] and one latent cache kv [B,Lk,dk]
    shared by all heads; the same hot-tile structure over the full key width
    (the values are the latent part of the same rows)."""
    dk = d_latent + d_rope
    nT = -(-Lk // TILE)
    hot = hot_tiles(seed, B, 1, nT, hot_frac)
    u = directions(seed, 1, dk, False)
    ut = torch.as_tensor(u[0], dtype=torch.float32, device=device)
    q = _randn((B, Hq, dk), seed * 100003, 3, device)
    q += shift * ut
    q = q.to(torch.bfloat16)
    kv = torch.empty((B, Lk, dk), dtype=torch.bfloat16, device=device)
    for b in range(B):
        kb = _randn((Lk, dk), seed * 100003 + b, 4, device)
        tiles = np.nonzero(hot[b, 0])[0]
        rows = (tiles[:, None] * TILE + np.arange(TILE)[None, :]).ravel()
        rows = rows[rows < Lk]
        kb.index_add_(0, torch.as_tensor(rows, device=device), (shift * ut).expand(len(rows), dk))
        kv[b] = kb.to(torch.bfloat16)
        del kb
    return MlaInputs(q, kv, hot, u)


# The workloads, by what they are (shapes from the method's two target uses:
# video-DiT self-attention and Llama-3.1-8B-style GQA prefill/decode).
WORKLOADS = {
    "tiny_prefill": dict(kind="prefill", B=1, Hq=1, Hkv=1, Lq=1024, Lk=1024, d=64, causal=False,
                         scale=1.0 / 8.0, hot_frac=0.20, per_head_u=False),
    "dit_prefill_32k": dict(kind="prefill", B=1, Hq=24, Hkv=24, Lq=32768, Lk=32768, d=128,
                            causal=False, scale=128 ** -0.5, hot_frac=0.15, per_head_u=False),
    # the DiT shape with 64-wide heads
    "dit_prefill_32k_d64": dict(kind="prefill", B=1, Hq=24, Hkv=24, Lq=32768, Lk=32768, d=64,
                                causal=False, scale=64 ** -0.5, hot_frac=0.15, per_head_u=False),
    "llama_prefill_16k": dict(kind="prefill", B=1, Hq=32, Hkv=8, Lq=16384, Lk=16384, d=128,
                              causal=True, scale=128 ** -0.5, hot_frac=0.10, per_head_u=True),
    "llama_decode_32k": dict(kind="decode", B=64, Hq=32, Hkv=8, Lk=32768, d=128,
                             scale=128 ** -0.5, hot_frac=0.10, per_head_u=True, num_splits=8),
    # chunked prefill: 2048 new tokens of each of 4 sequences against a 32K
    # cache (keys of the earlier chunks plus the new ones), causal from the
    # bottom-right
    "llama_chunked_prefill_2k_on_32k": dict(kind="prefill", B=4, Hq=32, Hkv=8, Lq=2048,
                                            Lk=32768, d=128, causal=True, scale=128 ** -0.5,
                                            hot_frac=0.10, per_head_u=True),
    # latent-attention decode (absorbed form): 128 sequences, 16 query heads
    # sharing one latent head of 512 + 64 rotary dims (DeepSeek-V2-Lite's
    # heads, or DeepSeek-V3's 128 over 8 GPUs); softmax scale 1/sqrt(128 + 64)
    "mla_decode_32k": dict(kind="mla_decode", B=128, Hq=16, Lk=32768, d_latent=512, d_rope=64,
                           scale=192 ** -0.5, hot_frac=0.10, num_splits=4),
    # the same with 32 query heads (DeepSeek-V3's 128 heads over 4 GPUs)
    "mla_decode_32k_32h": dict(kind="mla_decode", B=128, Hq=32, Lk=32768, d_latent=512,
                               d_rope=64, scale=192 ** -0.5, hot_frac=0.10, num_splits=4),
    # the same with 64 query heads (DeepSeek-V3's 128 heads over 2 GPUs)
    "mla_decode_32k_64h": dict(kind="mla_decode", B=128, Hq=64, Lk=32768, d_latent=512,
                               d_rope=64, scale=192 ** -0.5, hot_frac=0.10, num_splits=4),
    # multi-query decode: 32 query heads on one KV head (a vote group of 32)
    "mqa_decode_32k": dict(kind="decode", B=64, Hq=32, Hkv=1, Lk=32768, d=128,
                           scale=128 ** -0.5, hot_frac=0.10, per_head_u=True, num_splits=8),
    # latent-attention prefill in its unabsorbed form: per head 128 non-rotary
    # + 64 rotary query/key entries and 128-wide values (DeepSeek-V2-Lite's 16
    # heads), causal
    "mla_prefill_16k": dict(kind="prefill", B=1, Hq=16, Hkv=16, Lq=16384, Lk=16384, d=192, dv=128,
                            causal=True, scale=192 ** -0.5, hot_frac=0.10, per_head_u=True),
    "long_prefill_128k": dict(kind="prefill", B=1, Hq=32, Hkv=8, Lq=131072, Lk=131072, d=128,
                              causal=True, scale=128 ** -0.5, hot_frac=0.05, per_head_u=True),
    "long_decode_128k": dict(kind="decode", B=8, Hq=32, Hkv=8, Lk=131072, d=128,
                             scale=128 ** -0.5, hot_frac=0.05, per_head_u=True, num_splits=16),
}


def make(workload: str, seed: int = 0, device="cpu", **overrides) -> tuple[Inputs, dict]:
    """Inputs for a named workload (shape fields may be overridden)."""
    cfg = dict(WORKLOADS[workload])
    cfg.update(overrides)
    if cfg["kind"] == "mla_decode":
        inp = mla_decode_inputs(B=cfg["B"], Hq=cfg["Hq"], Lk=cfg["Lk"], d_latent=cfg["d_latent"],
                                d_rope=cfg["d_rope"], hot_frac=cfg["hot_frac"], seed=seed,
                                device=device)
    elif cfg["kind"] == "prefill":
        inp = prefill_inputs(B=cfg["B"], Hq=cfg["Hq"], Hkv=cfg["Hkv"], Lq=cfg["Lq"], Lk=cfg["Lk"],
                             d=cfg["d"], hot_frac=cfg["hot_frac"], seed=seed,
                             per_head_u=cfg["per_head_u"], device=device, dv=cfg.get("dv"))
    else:
        inp = decode_inputs(B=cfg["B"], Hq=cfg["Hq"], Hkv=cfg["Hkv"], Lk=cfg["Lk"], d=cfg["d"],
                            hot_frac=cfg["hot_frac"], seed=seed, per_head_u=cfg["per_head_u"],
                            device=device)
    return inp, cfg
