"""fp64 CPU oracle for skip-softmax (BLASST) attention -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg use this package.  The product (``block_sparse_attention_sm_gb300``) never
imports it, and the two share no code: the oracle is plain C (``oracle.c``)
over bf16 bit patterns, compiled with gcc by :func:`build`.

The method follows the "Skip-Softmax" design doc (§The online-softmax pass,
§The skip test, §What this bounds, §The threshold) and the BLASST summary
(§Methodologie, §Calibratie); ``oracle.c`` cites each step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

KEPT, SKIPPED, NOT_EVALUATED = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc, OpenMP over units)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


class _Prefill(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("Lq", ctypes.c_int), ("Lk", ctypes.c_int), ("d", ctypes.c_int),
        ("scale", ctypes.c_double), ("causal", ctypes.c_int), ("lam", ctypes.c_double),
        ("Bq", ctypes.c_int), ("Bk", ctypes.c_int), ("dv", ctypes.c_int),
    ]


class _Decode(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("Lk", ctypes.c_int), ("d", ctypes.c_int), ("scale", ctypes.c_double),
        ("lam", ctypes.c_double), ("num_splits", ctypes.c_int), ("Bk", ctypes.c_int),
        ("dv", ctypes.c_int),
    ]


_lib = None


def _get():
    global _lib
    if _lib is None:
        # A test may point at a deliberately mutated copy of the oracle.
        override = os.environ.get("SSATTN_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        P = ctypes.c_void_p
        lib.orc_prefill.argtypes = [ctypes.POINTER(_Prefill), P, P, P, P, ctypes.c_int64, P, P, P, P, P]
        lib.orc_prefill.restype = ctypes.c_int
        lib.orc_decode.argtypes = [ctypes.POINTER(_Decode), P, P, P, P, ctypes.c_int64, P, P, P, P, P, P, P, P]
        lib.orc_decode.restype = ctypes.c_int
        lib.orc_calibrate.argtypes = [P, P, ctypes.c_int64, ctypes.c_double, ctypes.c_double, P, P, P]
        lib.orc_calibrate.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 input as a contiguous uint16 array of bit patterns.

    Accepts a uint16 numpy array or a torch bfloat16 tensor (any device)."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
        return np.ascontiguousarray(x)
    import torch  # local: the oracle itself does not need torch

    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bfloat16")
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@dataclass
class PrefillResult:
    o: np.ndarray        # [n, Bq, dv] fp64
    mask: np.ndarray     # [n, nT] uint8
    margin: np.ndarray   # [n, nT] fp64
    counts: np.ndarray   # [n] uint32
    units: np.ndarray    # [n] int64 unit ids


@dataclass
class DecodeResult:
    o: np.ndarray        # [n, G, dv]
    mask: np.ndarray     # [n, nT]
    margin: np.ndarray   # [n, nT]
    counts: np.ndarray   # [n, S]
    part_m: np.ndarray   # [n, G, S]
    part_l: np.ndarray   # [n, G, S]
    part_o: np.ndarray   # [n, G, S, dv]
    units: np.ndarray


def prefill(q, k, v, *, scale: float, causal: bool, lam: float, Bq: int = 128, Bk: int = 128,
            units=None, mask_override=None) -> PrefillResult:
    """Skip-softmax prefill over q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv]
    (bf16; dv may differ from d, as in the unabsorbed form of multi-head latent
    attention, which the BLASST summary lists among the supported kinds,
    §Belangrijkste Bijdragen item 4).  o is [n, Bq, dv]."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Lq, d = qb.shape
    _, Hkv, Lk, _ = kb.shape
    dv = vb.shape[-1]
    if vb.shape[:3] != kb.shape[:3]:
        raise ValueError("prefill: v must be [B, Hkv, Lk, dv] like k")
    nqb = -(-Lq // Bq)
    nT = -(-Lk // Bk)
    if units is None:
        units = np.arange(B * Hq * nqb, dtype=np.int64)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    n = len(units)
    o = np.zeros((n, Bq, dv), np.float64)
    mask = np.zeros((n, nT), np.uint8)
    margin = np.zeros((n, nT), np.float64)
    counts = np.zeros(n, np.uint32)
    ov = None
    if mask_override is not None:
        ov = np.ascontiguousarray(np.asarray(mask_override, dtype=np.uint8).reshape(n, nT))
    prob = _Prefill(B, Hq, Hkv, Lq, Lk, d, float(scale), int(bool(causal)), float(lam), Bq, Bk,
                    dv)
    rc = _get().orc_prefill(ctypes.byref(prob), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(units), n,
                            _ptr(ov), _ptr(o), _ptr(mask), _ptr(margin), _ptr(counts))
    if rc != 0:
        raise ValueError("orc_prefill rejected its arguments")
    return PrefillResult(o, mask, margin, counts, units)


def decode(q, k, v, *, scale: float, lam: float, num_splits: int, Bk: int = 128, units=None,
           mask_override=None) -> DecodeResult:
    """Skip-softmax split-KV decode over q [B,Hq,d], k [B,Hkv,Lk,d] and
    v [B,Hkv,Lk,dv] (bf16; dv may differ from d)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, d = qb.shape
    _, Hkv, Lk, dk = kb.shape
    dv = vb.shape[-1]
    if dk != d or vb.shape[:3] != kb.shape[:3]:
        raise ValueError("decode: q/k widths or k/v shapes disagree")
    G = Hq // Hkv
    S = int(num_splits)
    nT = -(-Lk // Bk)
    if units is None:
        units = np.arange(B * Hkv, dtype=np.int64)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    n = len(units)
    o = np.zeros((n, G, dv), np.float64)
    mask = np.zeros((n, nT), np.uint8)
    margin = np.zeros((n, nT), np.float64)
    counts = np.zeros((n, S), np.uint32)
    pm = np.zeros((n, G, S), np.float64)
    pl = np.zeros((n, G, S), np.float64)
    po = np.zeros((n, G, S, dv), np.float64)
    ov = None
    if mask_override is not None:
        ov = np.ascontiguousarray(np.asarray(mask_override, dtype=np.uint8).reshape(n, nT))
    prob = _Decode(B, Hq, Hkv, Lk, d, float(scale), float(lam), S, Bk, dv)
    rc = _get().orc_decode(ctypes.byref(prob), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(units), n,
                           _ptr(ov), _ptr(o), _ptr(mask), _ptr(margin), _ptr(counts),
                           _ptr(pm), _ptr(pl), _ptr(po))
    if rc != 0:
        raise ValueError("orc_decode rejected its arguments")
    return DecodeResult(o, mask, margin, counts, pm, pl, po, units)


def mla_decode(q, kv, *, d_latent: int, scale: float, lam: float, num_splits: int,
               Bk: int = 128, units=None, mask_override=None) -> DecodeResult:
    """Decode with multi-head latent attention over q [B,Hq,dk] and one
    latent cache kv [B,Lk,dk] (bf16) shared by every query head.

    Reading of the pages' "MLA" (the BLASST summary, §Belangrijkste
    Bijdragen item 4, lists it beside MHA, GQA and MQA among the attention
    kinds its prefill and decode kernels support, without giving its
    shapes): the absorbed
    form, in which the keys are the cache rows (latent part followed by the
    rotary part, dk wide) and the values are their first d_latent entries.
    All Hq heads share the one latent head, so they form the voting group.
    This is `decode` with Hkv = 1, k = kv and v = kv[..., :d_latent] (a copy
    of the inputs, no arithmetic)."""
    kb = _bits(kv)
    if kb.ndim != 3 or not 0 < d_latent <= kb.shape[-1]:
        raise ValueError("mla_decode: kv must be [B, Lk, dk] with d_latent <= dk")
    k = kb[:, None]
    v = np.ascontiguousarray(kb[:, None, :, :d_latent])
    return decode(q, k, v, scale=scale, lam=lam, num_splits=num_splits, Bk=Bk, units=units,
                  mask_override=mask_override)


def calibrate(margin: np.ndarray, mask: np.ndarray, target: float, L: float):
    """Order-statistic calibration: returns (a, skipped_at_a, evaluated)."""
    m = np.ascontiguousarray(margin, dtype=np.float64).ravel()
    k = np.ascontiguousarray(mask, dtype=np.uint8).ravel()
    a = ctypes.c_double()
    ko = ctypes.c_int64()
    no = ctypes.c_int64()
    rc = _get().orc_calibrate(_ptr(m), _ptr(k), m.size, float(target), float(L),
                              ctypes.cast(ctypes.byref(a), ctypes.c_void_p),
                              ctypes.cast(ctypes.byref(ko), ctypes.c_void_p),
                              ctypes.cast(ctypes.byref(no), ctypes.c_void_p))
    if rc != 0:
        raise ValueError("orc_calibrate rejected its arguments")
    return a.value, ko.value, no.value
