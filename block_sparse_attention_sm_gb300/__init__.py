"""Skip-softmax (BLASST) attention for GB300 (sm_103a).

The product is the C-ABI library ``libssattn.so`` (``include/ssattn.h``);
:mod:`.capi` binds its entry points under the same names.  The helpers below
only allocate outputs with torch and forward to those entry points: every
step of the attention pass runs in the library's CUDA kernels, and there is
no CPU or eager fallback (a missing library raises).
"""
from __future__ import annotations

import math

from . import capi
from .capi import SSError

TILE = 128


def build(force: bool = False) -> str:
    from .builder import build as _build

    return _build(force=force)


def _check(st: int, what: str):
    if st != capi.SS_OK:
        raise SSError(st, what)


def _tensor(name, t, dtypes, ndim=None, min_numel=None, shape=None):
    """Check a tensor argument before its pointer reaches the library.

    The kernels read and write raw device addresses with the documented
    layout, so a strided view, another element type or a too small buffer
    would be read as something else.  The device is checked separately, after
    every argument's layout (``_on_cuda``), so that the layout checks can be
    exercised without a GPU."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: element type must be one of {[str(x) for x in dtypes]}, "
                         f"got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dimensions, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: needs at least {min_numel} elements, has {t.numel()}")
    return t


def _on_cuda(**tensors):
    """Every given tensor (None: absent) must live on one CUDA device: the
    library dereferences their addresses in its kernels."""
    devs = set()
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name}: must be a CUDA tensor, got device {t.device}")
        devs.add(t.device)
    if len(devs) > 1:
        raise ValueError(f"tensors on several devices: {sorted(str(d) for d in devs)}")


def _bf16():
    import torch

    return (torch.bfloat16,)


def _u32():
    import torch

    return (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _optional(name, t, dtypes, min_numel):
    if t is not None:
        _tensor(name, t, dtypes, min_numel=min_numel)


def _debug_outputs(skip_mask, vote_margin, n):
    import torch

    _optional("skip_mask", skip_mask, (torch.uint8,), n)
    _optional("vote_margin", vote_margin, (torch.float32,), n)


def _shape_prefill(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("prefill expects q [B,Hq,Lq,d] and k/v [B,Hkv,Lk,d]")
    B, Hq, Lq, d = q.shape
    Bk, Hkv, Lk, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("q and k disagree on batch or head dim")
    return B, Hq, Hkv, Lq, Lk, d


def units_prefill(B, Hq, Lq) -> int:
    return B * Hq * math.ceil(Lq / TILE)


def prefill(q, k, v, *, scale: float, causal: bool = False, lam: float = 0.0, counts=None,
            out=None, skip_mask=None, vote_margin=None, stream=None):
    """o = skip-softmax attention(q, k, v) for bf16 CUDA tensors.

    q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] contiguous.  Returns o [B,Hq,Lq,d].
    ``counts`` (uint32/int32 tensor of B*Hq*ceil(Lq/128)) receives the
    skipped tiles per query block; ``skip_mask``/``vote_margin`` the
    per-tile debug outputs."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _tensor(name, t, _bf16(), ndim=4)
    B, Hq, Hkv, Lq, Lk, d = _shape_prefill(q, k)
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("prefill expects v with the shape of k")
    units = units_prefill(B, Hq, Lq)
    _optional("counts", counts, _u32(), units)
    _debug_outputs(skip_mask, vote_margin, units * math.ceil(Lk / TILE))
    if out is not None:
        _tensor("out", out, _bf16(), shape=q.shape)
    _on_cuda(q=q, k=k, v=v, out=out, counts=counts, skip_mask=skip_mask, vote_margin=vote_margin)
    o = out if out is not None else torch.empty_like(q)
    if skip_mask is None and vote_margin is None:
        st = capi.ss_attn_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam, counts,
                                  stream)
    else:
        st = capi.ss_attn_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam,
                                     counts, skip_mask, vote_margin, False, stream)
    _check(st, "ss_attn_prefill")
    return o


def mla_prefill(q, k, v, *, scale: float, causal: bool = False, lam: float = 0.0, counts=None,
                out=None, skip_mask=None, vote_margin=None, stream=None):
    """Latent-attention prefill (unabsorbed form): q [B,Hq,Lq,192],
    k [B,Hkv,Lk,192], v [B,Hkv,Lk,128] bf16 CUDA tensors.  Returns
    o [B,Hq,Lq,128].  Counters and debug outputs as in :func:`prefill`."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _tensor(name, t, _bf16(), ndim=4)
    B, Hq, Hkv, Lq, Lk, d = _shape_prefill(q, k)
    dv = v.shape[3]
    if tuple(v.shape[:3]) != tuple(k.shape[:3]):
        raise ValueError("mla_prefill expects v [B,Hkv,Lk,d_v] with k's first three dims")
    units = units_prefill(B, Hq, Lq)
    _optional("counts", counts, _u32(), units)
    _debug_outputs(skip_mask, vote_margin, units * math.ceil(Lk / TILE))
    if out is not None:
        _tensor("out", out, _bf16(), shape=(B, Hq, Lq, dv))
    _on_cuda(q=q, k=k, v=v, out=out, counts=counts, skip_mask=skip_mask, vote_margin=vote_margin)
    o = out if out is not None else torch.empty((B, Hq, Lq, dv), dtype=q.dtype, device=q.device)
    if skip_mask is None and vote_margin is None:
        st = capi.ss_attn_mla_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, dv, scale, causal, lam,
                                      counts, stream)
    else:
        st = capi.ss_attn_mla_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, dv, scale, causal,
                                         lam, counts, skip_mask, vote_margin, False, stream)
    _check(st, "ss_attn_mla_prefill")
    return o


def decode_workspace(B, Hq, d, num_kv_splits, device):
    import torch

    n = capi.ss_attn_decode_workspace_size(B, Hq, d, num_kv_splits)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device), n


def decode(q, k, v, *, scale: float, lam: float = 0.0, num_kv_splits: int = 1, counts=None,
           out=None, workspace=None, skip_mask=None, vote_margin=None, stream=None):
    """Split-KV decode: q [B,Hq,d], k/v [B,Hkv,Lk,d] bf16 CUDA.  Returns o [B,Hq,d]."""
    import torch

    _tensor("q", q, _bf16(), ndim=3)
    _tensor("k", k, _bf16(), ndim=4)
    _tensor("v", v, _bf16(), shape=k.shape)
    B, Hq, d = q.shape
    Bk, Hkv, Lk, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("decode expects q [B,Hq,d] and k/v [B,Hkv,Lk,d]")
    _optional("counts", counts, _u32(), B * Hkv * max(1, int(num_kv_splits)))
    _debug_outputs(skip_mask, vote_margin, B * Hkv * math.ceil(Lk / TILE))
    if out is not None:
        _tensor("out", out, _bf16(), shape=q.shape)
    if workspace is not None:
        _tensor("workspace", workspace, (workspace.dtype,))
    _on_cuda(q=q, k=k, v=v, out=out, counts=counts, workspace=workspace, skip_mask=skip_mask,
             vote_margin=vote_margin)
    o = out if out is not None else torch.empty_like(q)
    if workspace is None:
        workspace, nbytes = decode_workspace(B, Hq, d, num_kv_splits, q.device)
    else:
        nbytes = workspace.numel() * workspace.element_size()
    if skip_mask is None and vote_margin is None:
        st = capi.ss_attn_decode(q, k, v, o, B, Hq, Hkv, Lk, d, scale, lam, num_kv_splits, counts,
                                 workspace, nbytes, stream)
    else:
        st = capi.ss_attn_decode_ex(q, k, v, o, B, Hq, Hkv, Lk, d, scale, lam, num_kv_splits,
                                    counts, workspace, nbytes, skip_mask, vote_margin, False,
                                    stream)
    _check(st, "ss_attn_decode")
    return o


MLA_LATENT, MLA_ROPE = 512, 64


def mla_workspace(B, Hq, num_kv_splits, device, d_latent=MLA_LATENT):
    import torch

    n = capi.ss_attn_mla_decode_workspace_size(B, Hq, d_latent, num_kv_splits)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device), n


def mla_decode(q, kv, *, scale: float, lam: float = 0.0, num_kv_splits: int = 1, counts=None,
               out=None, workspace=None, skip_mask=None, vote_margin=None, stream=None,
               d_latent: int = MLA_LATENT):
    """Latent-attention (MLA) split-KV decode: q [B,Hq,dk] and one latent
    cache kv [B,Lk,dk] (dk = d_latent + d_rope) bf16 CUDA; the values are
    kv[..., :d_latent].  Returns o [B,Hq,d_latent]."""
    import torch

    _tensor("q", q, _bf16(), ndim=3)
    _tensor("kv", kv, _bf16(), ndim=3)
    B, Hq, dk = q.shape
    Bk, Lk, dk2 = kv.shape
    if Bk != B or dk2 != dk:
        raise ValueError("mla_decode expects q [B,Hq,dk] and kv [B,Lk,dk]")
    _optional("counts", counts, _u32(), B * max(1, int(num_kv_splits)))
    _debug_outputs(skip_mask, vote_margin, B * math.ceil(Lk / TILE))
    if out is not None:
        _tensor("out", out, _bf16(), shape=(B, Hq, d_latent))
    if workspace is not None:
        _tensor("workspace", workspace, (workspace.dtype,))
    _on_cuda(q=q, kv=kv, out=out, counts=counts, workspace=workspace, skip_mask=skip_mask,
             vote_margin=vote_margin)
    o = out if out is not None else torch.empty((B, Hq, d_latent), dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace, nbytes = mla_workspace(B, Hq, num_kv_splits, q.device, d_latent)
    else:
        nbytes = workspace.numel() * workspace.element_size()
    if skip_mask is None and vote_margin is None:
        st = capi.ss_attn_mla_decode(q, kv, o, B, Hq, Lk, d_latent, dk - d_latent, scale, lam,
                                     num_kv_splits, counts, workspace, nbytes, stream)
    else:
        st = capi.ss_attn_mla_decode_ex(q, kv, o, B, Hq, Lk, d_latent, dk - d_latent, scale, lam,
                                        num_kv_splits, counts, workspace, nbytes, skip_mask,
                                        vote_margin, False, stream)
    _check(st, "ss_attn_mla_decode")
    return o


def calibrate(kind: str, q, k, v, *, scale: float, target_sparsity: float, causal: bool = False,
              num_kv_splits: int = 1, counts=None, stream=None):
    """Fit a (lambda = a / Lk) for a target tile sparsity.  Returns (a, achieved).

    kind: "prefill", "mla_prefill" (q/k 192 wide, v 128 wide), "decode" or
    "mla_decode" (k is then the latent cache [B,Lk,dk] and v is ignored)."""
    import torch

    if kind not in ("prefill", "decode", "mla_decode", "mla_prefill"):
        raise ValueError(f"calibrate: unknown kind {kind!r}")
    is_prefill = kind in ("prefill", "mla_prefill")
    _tensor("q", q, _bf16(), ndim=4 if is_prefill else 3)
    _tensor("k", k, _bf16(), ndim=3 if kind == "mla_decode" else 4)
    if kind == "mla_prefill":
        _tensor("v", v, _bf16(), ndim=4)
        if tuple(v.shape[:3]) != tuple(k.shape[:3]):
            raise ValueError("mla_prefill expects v [B,Hkv,Lk,d_v] with k's first three dims")
    elif kind != "mla_decode":
        _tensor("v", v, _bf16(), shape=k.shape)
    if is_prefill:
        B, Hq, Hkv, Lq, Lk, d = _shape_prefill(q, k)
        n = units_prefill(B, Hq, Lq)
        k_ = capi.SS_PREFILL if kind == "prefill" else capi.SS_MLA_PREFILL
    elif kind == "mla_decode":
        B, Hq, d = q.shape
        Lk = k.shape[1]
        Hkv, Lq = 1, 1
        n = B * num_kv_splits
        k_ = capi.SS_MLA_DECODE
        v = k
    else:
        B, Hq, d = q.shape
        _, Hkv, Lk, _ = k.shape
        Lq = 1
        n = B * Hkv * num_kv_splits
        k_ = capi.SS_DECODE
    if counts is not None:
        _tensor("counts", counts, _u32(), min_numel=n)
    _on_cuda(q=q, k=k, v=v, counts=counts)
    if counts is None:
        counts = torch.empty(n, dtype=torch.int32, device=q.device)
    prob = capi.ss_problem(k_, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Hq, Hkv, Lq, Lk, d,
                           float(scale), int(bool(causal)), int(num_kv_splits), counts.data_ptr(),
                           capi._stream(stream))
    st, a, achieved = capi.ss_calibrate(prob, target_sparsity)
    _check(st, "ss_calibrate")
    return a, achieved


def fit_factor(s, a):
    st, A, B = capi.ss_fit_factor(s, a)
    _check(st, "ss_fit_factor")
    return A, B


def lambda_of(A, B, s, L) -> float:
    return capi.ss_lambda(A, B, s, L)


def stream_status(stream=None) -> None:
    st = capi.ss_stream_status(stream)
    _check(st, "device status")
