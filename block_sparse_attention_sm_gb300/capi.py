"""ctypes binding of libssattn (include/ssattn.h): same names, marshalling only.

Every ``ss_*`` function here forwards to the C entry point of the same name.
Tensor arguments may be torch tensors (their ``data_ptr()`` is passed) or
plain integers (device addresses).  ``stream`` defaults to torch's current
CUDA stream.  Nothing here computes: if the shared library is missing the
import of a function fails loudly -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssattn.so")

SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED, SS_ERR_CUDA, SS_ERR_TIMEOUT, SS_ERR_WORKSPACE = range(6)
SS_PREFILL, SS_DECODE, SS_MLA_DECODE, SS_MLA_PREFILL = 0, 1, 2, 3

EXPORTS = (
    "ss_attn_prefill", "ss_attn_prefill_ex", "ss_attn_mla_prefill", "ss_attn_mla_prefill_ex",
    "ss_attn_decode_workspace_size", "ss_attn_decode",
    "ss_attn_decode_ex", "ss_attn_decode_noalloc", "ss_decode_static_scratch_bytes",
    "ss_attn_decode_paged",
    "ss_attn_mla_decode_workspace_size", "ss_attn_mla_decode", "ss_attn_mla_decode_ex",
    "ss_attn_mla_decode_paged",
    "ss_calibrate", "ss_fit_factor", "ss_lambda", "ss_status_string", "ss_stream_status",
)


class SSError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {ss_status_string(status)} (status {status})")


class ss_debug_opts(ctypes.Structure):
    _fields_ = [("skip_mask", ctypes.c_void_p), ("vote_margin", ctypes.c_void_p),
                ("count_only", ctypes.c_int), ("fault_inject", ctypes.c_int),
                ("vote_chunk_tiles", ctypes.c_int), ("prefill_kernel", ctypes.c_int)]


class ss_problem(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("q", ctypes.c_void_p), ("k", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("B", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("Lq", ctypes.c_int), ("Lk", ctypes.c_int),
                ("d", ctypes.c_int), ("scale", ctypes.c_float), ("causal", ctypes.c_int),
                ("num_kv_splits", ctypes.c_int), ("skip_counts", ctypes.c_void_p),
                ("stream", ctypes.c_void_p), ("fault_inject", ctypes.c_int)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libssattn.so (built by ``block_sparse_attention_sm_gb300.builder``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -m block_sparse_attention_sm_gb300.builder)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    pre = [P, P, P, P, I, I, I, I, I, I, F, I, F, P]
    lib.ss_attn_prefill.argtypes = pre + [P]
    lib.ss_attn_prefill_ex.argtypes = pre + [ctypes.POINTER(ss_debug_opts), P]
    mpre = [P, P, P, P, I, I, I, I, I, I, I, F, I, F, P]
    lib.ss_attn_mla_prefill.argtypes = mpre + [P]
    lib.ss_attn_mla_prefill_ex.argtypes = mpre + [ctypes.POINTER(ss_debug_opts), P]
    dec = [P, P, P, P, I, I, I, I, I, F, F, I, P, P, U]
    lib.ss_attn_decode.argtypes = dec + [P]
    lib.ss_attn_decode_ex.argtypes = dec + [ctypes.POINTER(ss_debug_opts), P]
    lib.ss_attn_decode_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, F, F, I, P, P]
    lib.ss_decode_static_scratch_bytes.argtypes = []
    lib.ss_decode_static_scratch_bytes.restype = U
    lib.ss_attn_decode_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, F, I, P, P, U,
                                         ctypes.POINTER(ss_debug_opts), P]
    lib.ss_attn_decode_workspace_size.argtypes = [I, I, I, I]
    lib.ss_attn_decode_workspace_size.restype = U
    mla = [P, P, P, I, I, I, I, I, F, F, I, P, P, U]
    lib.ss_attn_mla_decode.argtypes = mla + [P]
    lib.ss_attn_mla_decode_ex.argtypes = mla + [ctypes.POINTER(ss_debug_opts), P]
    lib.ss_attn_mla_decode_paged.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, F, I, P, P, U,
                                             ctypes.POINTER(ss_debug_opts), P]
    lib.ss_attn_mla_decode_workspace_size.argtypes = [I, I, I, I]
    lib.ss_attn_mla_decode_workspace_size.restype = U
    lib.ss_calibrate.argtypes = [ctypes.POINTER(ss_problem), F, ctypes.POINTER(F), ctypes.POINTER(F)]
    lib.ss_fit_factor.argtypes = [ctypes.POINTER(F), ctypes.POINTER(F), I, ctypes.POINTER(F),
                                  ctypes.POINTER(F)]
    lib.ss_lambda.argtypes = [F, F, F, I]
    lib.ss_lambda.restype = F
    lib.ss_status_string.argtypes = [I]
    lib.ss_status_string.restype = ctypes.c_char_p
    lib.ss_stream_status.argtypes = [P]
    for name in ("ss_attn_prefill", "ss_attn_prefill_ex", "ss_attn_mla_prefill",
                 "ss_attn_mla_prefill_ex", "ss_attn_decode", "ss_attn_decode_ex",
                 "ss_attn_decode_noalloc", "ss_attn_decode_paged", "ss_attn_mla_decode",
                 "ss_attn_mla_decode_ex", "ss_attn_mla_decode_paged", "ss_calibrate",
                 "ss_fit_factor", "ss_stream_status"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dbg(skip_mask=None, vote_margin=None, count_only=False, fault_inject=0, vote_chunk_tiles=0,
         prefill_kernel=0):
    return ss_debug_opts(_ptr(skip_mask), _ptr(vote_margin), int(bool(count_only)),
                         int(fault_inject), int(vote_chunk_tiles), int(prefill_kernel))


def ss_status_string(status: int) -> str:
    return load().ss_status_string(int(status)).decode()


def ss_attn_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam, skip_counts=None,
                    stream=None) -> int:
    return load().ss_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lq, Lk, d,
                                  float(scale), int(bool(causal)), float(lam), _ptr(skip_counts),
                                  _stream(stream))


def ss_attn_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lam, skip_counts=None,
                       skip_mask=None, vote_margin=None, count_only=False, stream=None,
                       vote_chunk_tiles=0, prefill_kernel=0) -> int:
    dbg = _dbg(skip_mask, vote_margin, count_only, vote_chunk_tiles=vote_chunk_tiles,
               prefill_kernel=prefill_kernel)
    return load().ss_attn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lq, Lk, d,
                                     float(scale), int(bool(causal)), float(lam),
                                     _ptr(skip_counts), ctypes.byref(dbg), _stream(stream))


def ss_attn_mla_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d_qk, d_v, scale, causal, lam,
                        skip_counts=None, stream=None) -> int:
    """Latent-attention prefill: q/k rows d_qk wide, v/o rows d_v wide."""
    return load().ss_attn_mla_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lq, Lk,
                                      d_qk, d_v, float(scale), int(bool(causal)), float(lam),
                                      _ptr(skip_counts), _stream(stream))


def ss_attn_mla_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d_qk, d_v, scale, causal, lam,
                           skip_counts=None, skip_mask=None, vote_margin=None, count_only=False,
                           stream=None) -> int:
    dbg = _dbg(skip_mask, vote_margin, count_only)
    return load().ss_attn_mla_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lq, Lk,
                                         d_qk, d_v, float(scale), int(bool(causal)), float(lam),
                                         _ptr(skip_counts), ctypes.byref(dbg), _stream(stream))


def ss_attn_decode_workspace_size(B, Hq, d, num_kv_splits) -> int:
    return int(load().ss_attn_decode_workspace_size(B, Hq, d, num_kv_splits))


def ss_attn_decode(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, lam, num_kv_splits,
                   skip_counts=None, workspace=None, workspace_bytes=0, stream=None) -> int:
    return load().ss_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), B, Hq, Hkv, Lk,
                                 d, float(scale), float(lam), int(num_kv_splits),
                                 _ptr(skip_counts), _ptr(workspace), int(workspace_bytes),
                                 _stream(stream))


def ss_attn_decode_ex(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, lam, num_kv_splits,
                      skip_counts=None, workspace=None, workspace_bytes=0, skip_mask=None,
                      vote_margin=None, count_only=False, stream=None, fault_inject=0) -> int:
    dbg = _dbg(skip_mask, vote_margin, count_only, fault_inject)
    return load().ss_attn_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), B, Hq, Hkv,
                                    Lk, d, float(scale), float(lam), int(num_kv_splits),
                                    _ptr(skip_counts), _ptr(workspace), int(workspace_bytes),
                                    ctypes.byref(dbg), _stream(stream))


def ss_attn_decode_noalloc(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, lam, num_kv_splits,
                           skip_counts=None, stream=None) -> int:
    """Decode without a workspace (partials in the library's static device array)."""
    return load().ss_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), B, Hq,
                                         Hkv, Lk, d, float(scale), float(lam), int(num_kv_splits),
                                         _ptr(skip_counts), _stream(stream))


def ss_attn_decode_paged(q, k_pages, v_pages, page_table, seq_lens, o, B, Hq, Hkv, num_pages,
                         max_pages, d, scale, lambda_a, num_kv_splits, skip_counts=None,
                         workspace=None, workspace_bytes=0, skip_mask=None, vote_margin=None,
                         count_only=False, stream=None) -> int:
    """Decode over a paged, variable-length KV cache (pages of 128 keys)."""
    dbg = _dbg(skip_mask, vote_margin, count_only)
    return load().ss_attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                       _ptr(seq_lens), _ptr(o), B, Hq, Hkv, num_pages, max_pages,
                                       d, float(scale), float(lambda_a), int(num_kv_splits),
                                       _ptr(skip_counts), _ptr(workspace), int(workspace_bytes),
                                       ctypes.byref(dbg), _stream(stream))


SS_DECODE_STATIC_SCRATCH_BYTES = 16 << 20  # the header's value; test_abi checks the library's


def ss_decode_static_scratch_bytes() -> int:
    """Size of ss_attn_decode_noalloc's built-in array in the loaded library."""
    return int(load().ss_decode_static_scratch_bytes())


def ss_attn_mla_decode_workspace_size(B, Hq, d_latent, num_kv_splits) -> int:
    return int(load().ss_attn_mla_decode_workspace_size(B, Hq, d_latent, num_kv_splits))


def ss_attn_mla_decode(q, kv, o, B, Hq, Lk, d_latent, d_rope, scale, lam, num_kv_splits,
                       skip_counts=None, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Latent-attention decode: q [B,Hq,dk], one latent cache kv [B,Lk,dk]."""
    return load().ss_attn_mla_decode(_ptr(q), _ptr(kv), _ptr(o), B, Hq, Lk, d_latent, d_rope,
                                     float(scale), float(lam), int(num_kv_splits),
                                     _ptr(skip_counts), _ptr(workspace), int(workspace_bytes),
                                     _stream(stream))


def ss_attn_mla_decode_ex(q, kv, o, B, Hq, Lk, d_latent, d_rope, scale, lam, num_kv_splits,
                          skip_counts=None, workspace=None, workspace_bytes=0, skip_mask=None,
                          vote_margin=None, count_only=False, stream=None) -> int:
    dbg = _dbg(skip_mask, vote_margin, count_only)
    return load().ss_attn_mla_decode_ex(_ptr(q), _ptr(kv), _ptr(o), B, Hq, Lk, d_latent, d_rope,
                                        float(scale), float(lam), int(num_kv_splits),
                                        _ptr(skip_counts), _ptr(workspace), int(workspace_bytes),
                                        ctypes.byref(dbg), _stream(stream))


def ss_calibrate(problem: ss_problem, target_sparsity: float):
    """Returns (status, a, achieved_sparsity)."""
    a = ctypes.c_float()
    ach = ctypes.c_float()
    st = load().ss_calibrate(ctypes.byref(problem), float(target_sparsity), ctypes.byref(a),
                             ctypes.byref(ach))
    return st, a.value, ach.value


def ss_fit_factor(s, a):
    """Least squares ln a = ln A + B s; returns (status, A, B)."""
    n = len(s)
    S = (ctypes.c_float * n)(*map(float, s))
    Av = (ctypes.c_float * n)(*map(float, a))
    A = ctypes.c_float()
    Bv = ctypes.c_float()
    st = load().ss_fit_factor(S, Av, n, ctypes.byref(A), ctypes.byref(Bv))
    return st, A.value, Bv.value


def ss_lambda(A, B, s, L) -> float:
    return float(load().ss_lambda(float(A), float(B), float(s), int(L)))


def ss_stream_status(stream=None) -> int:
    return load().ss_stream_status(_stream(stream))


def ss_attn_mla_decode_paged(q, kv_pages, page_table, seq_lens, o, B, Hq, num_pages, max_pages,
                             d_latent, d_rope, scale, lambda_a, num_kv_splits, skip_counts=None,
                             workspace=None, workspace_bytes=0, skip_mask=None, vote_margin=None,
                             count_only=False, stream=None) -> int:
    """Latent-attention decode over a paged latent cache (pages of 128 rows)."""
    dbg = _dbg(skip_mask, vote_margin, count_only)
    return load().ss_attn_mla_decode_paged(_ptr(q), _ptr(kv_pages), _ptr(page_table),
                                           _ptr(seq_lens), _ptr(o), B, Hq, num_pages, max_pages,
                                           d_latent, d_rope, float(scale), float(lambda_a),
                                           int(num_kv_splits), _ptr(skip_counts), _ptr(workspace),
                                           int(workspace_bytes), ctypes.byref(dbg),
                                           _stream(stream))
