#!/usr/bin/env python3
"""Benchmark: skip-softmax (BLASST) attention forward on GB300.

One step = the whole hot path over one batch of synthetic inputs:
  * prefill "dit_prefill_32k": B1 H24 Lq=Lk=32768 d128 non-causal, lambda
    calibrated to 70% skipped tiles (ss_calibrate, before timing);
  * decode "llama_decode_32k": 64 sequences x Hq32/Hkv8, KV 32768, d128,
    8 KV splits, lambda calibrated to 70%.
Both kernels are timed with CUDA events on the launching stream.  `value` is
prefill TFLOP/s on the algorithm's FLOPs (QK^T on every evaluated tile + P.V
on kept tiles: the work the method executes); the MMA FLOPs the kernel
actually issues are reported beside them.  `decode` reports HBM GB/s on the
bytes the algorithm moves (all of K, kept V, Q and O).  Inputs exceed the 129 MB L2 (no flush needed).  Speedups are
against the library's own lambda = 0 path on the same inputs.

python bench.py [--gpus N --steps K --warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = "dit_prefill_32k"
DECODE = "llama_decode_32k"
TARGET = 0.7
METRIC = "prefill TFLOP/s & decode HBM GB/s at ~70% tile sparsity; speedup vs own dense"
TILE = 128


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        pk = json.load(open(path))
        return dict(hbm=pk["hbm_gbs"], bf16=pk["bf16_tflops"],
                    bf16_sust=pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def _src_hash(names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "block_sparse_attention_sm_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


PAIR_SOURCES = ["prefill_pair_sm103.cu", "ptx_pair_sm103.cuh", "ptx_sm103.cuh", "common.cuh"]
DECODE_SOURCES = ["decode_sm103.cu", "decode_rows.cuh", "ptx_sm103.cuh", "common.cuh"]


def _traffic(kernel, sources):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    ent = json.load(open(path)).get(kernel)
    if not ent or ent.get("source_sha256_16") != _src_hash(sources):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ssattn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines)


def parse_clock_samples(lines):
    """Summarise nvidia-smi samples (csv, noheader, nounits, in ClockSampler.FIELDS
    order): median SM clock over the samples above half the maximum (under
    load), the maximum, and every throttle reason seen active."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
        except ValueError:
            continue
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
    loaded = [r[0] for r in rows if r[0] > 0.5 * r[1]] or [r[0] for r in rows]
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, ws, device="cpu"):
    """The slowest rank sets the job's time: element-wise maximum over ranks
    (a process group must be initialised when ws > 1)."""
    if ws <= 1:
        return [float(x) for x in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(work_per_rank, ws, ms):
    """Whole-job throughput of N independent replicas (weak scaling): every
    rank processes the same work, and the job takes the slowest rank's time."""
    return work_per_rank * ws / ms


def prefill_flops(B, Hq, nqb, nT_eval, kept, d):
    """Algorithmic FLOPs: Q K^T on every evaluated tile, P.V on kept tiles."""
    return 2 * TILE * TILE * d * (nT_eval + kept)


def prefill_mma_flops(nT_eval, pair_union_tiles, d):
    """MMA FLOPs the CTA-pair prefill kernel issues: Q K^T once on every
    evaluated tile, and P.V for both query blocks of a pair on every tile
    that either block keeps (the pair's P.V covers both blocks; a block that
    skipped the tile contributes zero rows).  `pair_union_tiles` counts, per
    pair of query blocks, the tiles kept by either block."""
    return 2 * TILE * TILE * d * (nT_eval + 2 * pair_union_tiles)


def pair_union(mask, nqb):
    """Tiles kept (mask 0) by either query block of each pair (blocks 2p and
    2p + 1 of one head): mask is [B*Hq*nqb, nT] uint8 with units in
    (b, h, query block) order.  A last, unpaired block counts alone."""
    import torch

    kept = (mask == 0).view(-1, nqb, mask.shape[1])
    if nqb % 2:
        kept = torch.cat([kept, torch.zeros_like(kept[:, :1])], dim=1)
    return int((kept[:, 0::2] | kept[:, 1::2]).sum())


def read_stream_gbs(dev, gib=4, reps=5):
    """A read-only HBM stream measured in the same process: the best
    CUDA-event time (of `reps`) of torch reductions that read a `gib` GiB
    buffer once (int64 max, fp32 sum and fp32 amax over the same bytes).  The
    decode kernel is almost pure reads, which a read+write copy does not
    measure.  Returns (GB/s, which reduction)."""
    import torch

    x = torch.ones(gib << 29, dtype=torch.bfloat16, device=dev)
    cands = {"int64 max": lambda: x.view(torch.int64).max(),
             "fp32 sum": lambda: x.view(torch.float32).sum(),
             "fp32 amax": lambda: x.view(torch.float32).amax()}
    best, which = None, None
    for name, fn in cands.items():
        fn()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            if best is None or ms < best:
                best, which = ms, name
    nbytes = x.numel() * x.element_size()
    del x
    torch.cuda.empty_cache()
    return nbytes / best / 1e6, which


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, the vendor's nominal figure (context only)


def run_native(args):
    import torch
    import torch.distributed as dist

    import block_sparse_attention_sm_gb300 as ss
    from block_sparse_attention_sm_gb300 import capi, synth

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ss.build()
    capi.load()
    peaks = _peaks()

    # ---------------------------------------------------------------- inputs
    pin, pcfg = synth.make(PREFILL, seed=rank, device=dev,
                           **({"Hq": args.prefill_heads, "Hkv": args.prefill_heads}
                              if args.prefill_heads else {}))
    q, k, v = pin.q, pin.k, pin.v
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    nqb, nT = -(-Lq // TILE), -(-Lk // TILE)
    p_units = B * Hq * nqb
    p_eval = p_units * nT  # non-causal: every tile evaluated
    o = torch.empty_like(q)
    p_cnt = torch.zeros(p_units, dtype=torch.int32, device=dev)

    din, dcfg = synth.make(args.decode_workload if args.profile else DECODE, seed=rank, device=dev,
                           **({"B": args.decode_batch} if args.decode_batch else {}))
    dq, dk, dv = din.q, din.k, din.v
    dB, dHq, dd = dq.shape
    dHkv, dLk = dk.shape[1], dk.shape[2]
    S = dcfg["num_splits"]
    dnT = -(-dLk // TILE)
    d_eval = dB * dHkv * dnT
    do = torch.empty_like(dq)
    d_cnt = torch.zeros(dB * dHkv * S, dtype=torch.int32, device=dev)
    wsb, wsn = ss.decode_workspace(dB, dHq, dd, S, dev)

    # ---------------------------------------------------------------- calibration
    t0 = time.time()
    a_p, ach_p = ss.calibrate("prefill", q, k, v, scale=pcfg["scale"], target_sparsity=TARGET)
    t_cal_p = time.time() - t0
    t0 = time.time()
    a_d, ach_d = ss.calibrate("decode", dq, dk, dv, scale=dcfg["scale"], target_sparsity=TARGET,
                              num_kv_splits=S)
    t_cal_d = time.time() - t0
    lam_p, lam_d = a_p / Lk, a_d / dLk

    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def prefill_call(lam):
        st = capi.ss_attn_prefill(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, pcfg["scale"], 0, lam, p_cnt, sh)
        if st != capi.SS_OK:
            raise SystemExit(f"ss_attn_prefill: {capi.ss_status_string(st)}")

    def decode_call(lam):
        st = capi.ss_attn_decode(dq, dk, dv, do, dB, dHq, dHkv, dLk, dd, dcfg["scale"], lam, S,
                                 d_cnt, wsb, wsn, sh)
        if st != capi.SS_OK:
            raise SystemExit(f"ss_attn_decode: {capi.ss_status_string(st)}")

    def barrier():
        if ws > 1:
            dist.barrier()

    def timed_loop(lam_p_, lam_d_, steps, warmup):
        for _ in range(warmup):
            prefill_call(lam_p_)
            decode_call(lam_d_)
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            ev[i][0].record(stream)
            prefill_call(lam_p_)
            ev[i][1].record(stream)
            decode_call(lam_d_)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        barrier()
        tp = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
        td = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
        return tp, td

    # ---------------------------------------------------------------- timed region
    clocks = ClockSampler(local)
    clocks.start()
    if args.profile and args.profile_dense:
        lam_p, lam_d = 0.0, 0.0
    tp, td = timed_loop(lam_p, lam_d, args.steps, args.warmup)
    clk = clocks.stop()
    st = capi.ss_stream_status(sh)
    if st != capi.SS_OK:
        raise SystemExit(f"device status: {capi.ss_status_string(st)}")
    p_skip = int(p_cnt.sum())
    d_skip = int(d_cnt.sum())
    p_kept = p_eval - p_skip
    d_kept = d_eval - d_skip
    ms_p = sum(tp) / len(tp)
    ms_d = sum(td) / len(td)
    ms_step = ms_p + ms_d

    if args.profile:
        # profiling run (under ncu): no extras, no JSON line
        return
    # dense (lambda = 0) path of the same library, same inputs, same protocol
    tpd, tdd = timed_loop(0.0, 0.0, max(5, args.steps // 4), 2)
    ms_p0 = sum(tpd) / len(tpd)
    ms_d0 = sum(tdd) / len(tdd)

    flops_p = prefill_flops(B, Hq, nqb, p_eval, p_kept, d)
    flops_dense_eq = 4.0 * B * Hq * Lq * Lk * d  # FA convention, lambda = 0 problem
    bytes_d = dB * dHkv * dLk * dd * 2 + d_kept * TILE * dd * 2 + 2 * dB * dHq * dd * 2
    bytes_d_part = 2 * dB * dHq * S * (dd + 2) * 4

    # max over ranks
    ms_p, ms_d, ms_step = max_over_ranks([ms_p, ms_d, ms_step], ws, dev)
    tflops = job_rate(flops_p, ws, ms_p) / 1e9
    gbs = job_rate(bytes_d, ws, ms_d) / 1e6

    # ---------------------------------------------------------------- end to end (host buffers)
    # One e2e step is the same work as one timed step -- a prefill and a
    # decode through the C ABI -- with each step's inputs copied in from
    # pinned host memory and its outputs copied out.  Prefill's inputs are its
    # q, k and v; decode's are the 64 new query tokens and the newest key and
    # value row of every (sequence, KV head), appended into the KV cache that
    # stays resident on the device between steps (loaded from the host once,
    # before timing).  Steps are pipelined over two device buffer sets on
    # three streams (copy in, compute, copy out): step i+1's copies overlap
    # step i's kernels.  A buffer set is refilled only after the step that
    # used it has been computed and copied out.
    # As many steps as the device-timed loop (the pipeline's fill and drain,
    # one input copy and one output copy, are spread over the same count).
    e2e_steps = max(3, args.steps)
    hq_, hk_, hv_ = (t_.cpu().pin_memory() for t_ in (q, k, v))
    ho_ = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    e_dk, e_dv = torch.empty_like(dk), torch.empty_like(dv)
    e_dk.copy_(dk.cpu())  # the resident cache, uploaded from the host once
    e_dv.copy_(dv.cpu())
    h_dq = dq.cpu().pin_memory()
    h_knew = dk[:, :, dLk - 1:dLk].cpu().pin_memory()  # the step's new key / value rows
    h_vnew = dv[:, :, dLk - 1:dLk].cpu().pin_memory()
    hdo_ = [torch.empty(do.shape, dtype=do.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t_.numel() * t_.element_size() for t_ in (hq_, hk_, hv_, h_dq, h_knew, h_vnew))
    d2h = ho_[0].numel() * ho_[0].element_size() + hdo_[0].numel() * hdo_[0].element_size()
    bufs = [(q, k, v, o), tuple(torch.empty_like(t_) for t_ in (q, k, v, o))]
    # (device buffers: empty_like of the pinned host rows would give pageable
    # host tensors, whose copies block the host and serialise the pipeline)
    dbufs = [tuple(torch.empty(t_.shape, dtype=t_.dtype, device=dev)
                   for t_ in (dq, h_knew, h_vnew, do)) for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in, ev_done, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        b = i % 2
        bq, bk, bv, bo = bufs[b]
        eq, ekn, evn, eo = dbufs[b]
        s_in.wait_event(ev_done[b])  # the step two back has read this set's inputs
        with torch.cuda.stream(s_in):
            bq.copy_(hq_, non_blocking=True)
            bk.copy_(hk_, non_blocking=True)
            bv.copy_(hv_, non_blocking=True)
            eq.copy_(h_dq, non_blocking=True)
            ekn.copy_(h_knew, non_blocking=True)
            evn.copy_(h_vnew, non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        s_cmp.wait_event(ev_out[b])  # the step two back has copied this set's outputs out
        st_ = capi.ss_attn_prefill(bq, bk, bv, bo, B, Hq, Hkv, Lq, Lk, d, pcfg["scale"], 0, lam_p,
                                   p_cnt, s_cmp.cuda_stream)
        if st_ != capi.SS_OK:
            raise SystemExit(f"ss_attn_prefill: {capi.ss_status_string(st_)}")
        with torch.cuda.stream(s_cmp):  # append the new rows (in stream order with decode)
            e_dk[:, :, dLk - 1:dLk].copy_(ekn)
            e_dv[:, :, dLk - 1:dLk].copy_(evn)
        st_ = capi.ss_attn_decode(eq, e_dk, e_dv, eo, dB, dHq, dHkv, dLk, dd, dcfg["scale"], lam_d,
                                  S, d_cnt, wsb, wsn, s_cmp.cuda_stream)
        if st_ != capi.SS_OK:
            raise SystemExit(f"ss_attn_decode: {capi.ss_status_string(st_)}")
        ev_done[b].record(s_cmp)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            ho_[b].copy_(bo, non_blocking=True)
            hdo_[b].copy_(eo, non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    # The host<->device copies share the host's memory and link with other
    # jobs on the machine, and a single run has shown copies stalled for
    # ~10 ms: the e2e figure is the median of three timed runs (all reported).
    e2e_runs = []
    for _ in range(3):
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        s_out.wait_stream(s_cmp)
        s_out.wait_stream(s_in)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_runs.append(e0.elapsed_time(e1) / e2e_steps)
    ms_e2e = statistics.median(e2e_runs)
    (ms_e2e,) = max_over_ranks([ms_e2e], ws, dev)
    st = capi.ss_stream_status(sh)
    if st != capi.SS_OK:
        raise SystemExit(f"device status after the end-to-end steps: {capi.ss_status_string(st)}")
    e2e_o_match = bool(torch.equal(ho_[(e2e_steps - 1) % 2], bufs[(e2e_steps - 1) % 2][3].cpu()))
    del bufs, dbufs, e_dk, e_dv, hq_, hk_, hv_
    torch.cuda.empty_cache()

    # ---------------------------------------------------------------- outputs for the parity sample
    # The timed configuration (plain entry points at the timed lambdas) and the
    # debug call with skip masks and vote margins (same kernels, same result),
    # outside the timed region.  The oracle side of the comparison runs in the
    # CPU-baseline leg below.
    p_mask = torch.empty((p_units, nT), dtype=torch.uint8, device=dev)
    p_margin = torch.empty((p_units, nT), dtype=torch.float32, device=dev)
    o_dbg = torch.empty_like(q)
    cnt_dbg = torch.empty_like(p_cnt)
    prefill_call(lam_p)
    st = capi.ss_attn_prefill_ex(q, k, v, o_dbg, B, Hq, Hkv, Lq, Lk, d, pcfg["scale"], 0, lam_p,
                                 cnt_dbg, p_mask, p_margin, stream=sh)
    dnT_ = dnT
    d_mask = torch.empty((dB * dHkv, dnT_), dtype=torch.uint8, device=dev)
    d_margin = torch.empty((dB * dHkv, dnT_), dtype=torch.float32, device=dev)
    do_dbg = torch.empty_like(do)
    dcnt_dbg = torch.empty_like(d_cnt)
    decode_call(lam_d)
    st2 = capi.ss_attn_decode_ex(dq, dk, dv, do_dbg, dB, dHq, dHkv, dLk, dd, dcfg["scale"], lam_d,
                                 S, dcnt_dbg, wsb, wsn, d_mask, d_margin, stream=sh)
    if st != capi.SS_OK or st2 != capi.SS_OK or capi.ss_stream_status(sh) != capi.SS_OK:
        raise SystemExit("debug launches failed")
    debug_same = bool(torch.equal(o, o_dbg) and torch.equal(p_cnt, cnt_dbg)
                      and torch.equal(do, do_dbg) and torch.equal(d_cnt, dcnt_dbg))
    gpu_out = {"prefill": {"o": o, "counts": p_cnt, "mask": p_mask, "margin": p_margin},
               "decode": {"o": do, "counts": d_cnt, "mask": d_mask, "margin": d_margin},
               "debug_call_equals_timed_call": debug_same}

    read_gbs, read_kind = read_stream_gbs(dev)

    line = None
    if rank == 0:
        peak_t = peaks["bf16"]
        achieved_p = flops_p / ms_p / 1e9
        achieved_d = bytes_d / ms_d / 1e6
        flops_mma = prefill_mma_flops(p_eval, pair_union(p_mask, nqb), d)
        line = {
            "metric": METRIC,
            "value": round(tflops, 2),
            "unit": "TFLOP/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded hot-tile generator; no model weights)",
            "config": {
                "workload": f"{PREFILL}: B1 H24 Lq=Lk=32768 d128 non-causal + {DECODE}: 64 seq "
                            "x Hq32/Hkv8 KV32768 d128 8 splits; lambda = a/L calibrated to 70% "
                            "skipped tiles",
                "prefill": {"B": B, "Hq": Hq, "Hkv": Hkv, "Lq": Lq, "Lk": Lk, "d": d,
                            "causal": False, "a": a_p, "lambda": lam_p,
                            "sparsity": p_skip / p_eval, "calibration_s": round(t_cal_p, 3)},
                "decode": {"B": dB, "Hq": dHq, "Hkv": dHkv, "Lk": dLk, "d": dd, "splits": S,
                           "a": a_d, "lambda": lam_d, "sparsity": d_skip / d_eval,
                           "calibration_s": round(t_cal_d, 3)},
                "l2": "inputs larger than L2 (prefill 604 MB, decode 8.6 GB); no flush",
                "parallelism": f"replicas x{ws} (independent units, no collective)",
                "value_from": "prefill kernel events inside each step",
            },
            "decode": {
                "value": round(gbs, 1), "unit": "GB/s", "ms": round(ms_d, 4),
                "tokens_per_s": round(dB * ws / ms_d * 1e3, 1),
                "bytes_per_launch": bytes_d, "partials_bytes_overhead": bytes_d_part,
            },
            "prefill": {"ms": round(ms_p, 4),
                        "tflops_algorithmic": round(tflops, 2),
                        "tflops_mma_issued": round(flops_mma * ws / ms_p / 1e9, 2),
                        "mma_issued_frac_of_peak": round(flops_mma / ms_p / 1e9 / peak_t, 4),
                        "tflops_dense_equivalent": round(flops_dense_eq * ws / ms_p / 1e9, 2),
                        "flops_algorithmic": flops_p, "flops_mma_issued": flops_mma,
                        "flops_note": "algorithmic = QK^T on every evaluated tile + P.V on kept "
                                      "tiles; mma_issued = what the CTA-pair kernel runs: QK^T on "
                                      "every evaluated tile, P.V for both blocks of a pair on every "
                                      "tile either block keeps"},
            "speedup_vs_dense": {"prefill": round(ms_p0 / ms_p, 3), "decode": round(ms_d0 / ms_d, 3),
                                 "prefill_dense_ms": round(ms_p0, 4),
                                 "decode_dense_ms": round(ms_d0, 4),
                                 "ideal_prefill_2_over_2_minus_s": round(2 / (2 - p_skip / p_eval), 3)},
            "roofline": {
                "bound": "tensor", "achieved": round(achieved_p, 2), "peak": peak_t,
                "unit": "TFLOP/s", "frac": round(achieved_p / peak_t, 4),
                "traffic": _traffic("prefill_pair", PAIR_SOURCES),
                "kernel": "prefill_pair_kernel<128,128,Sparse>",
                "peak_kind": f"bf16 burst ({peaks['src']})",
            },
            "roofline_decode": {
                "bound": "hbm", "achieved": round(achieved_d, 1), "peak": peaks["hbm"],
                "unit": "GB/s", "frac": round(achieved_d / peaks["hbm"], 4),
                "traffic": _traffic("decode", DECODE_SOURCES),
                "kernel": "decode_kernel<128,4,Sparse> + decode_merge_kernel",
                "peak_kind": f"HBM copy, read+write ({peaks['src']})",
                "read_stream_gbs": round(read_gbs, 1),
                "frac_of_read_stream": round(achieved_d / read_gbs, 4),
                "read_stream_kind": f"best torch reduction over 4 GiB ({read_kind}), CUDA events, "
                                    "best of 5 each, same process",
                "nominal_gbs": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved_d / NOMINAL_HBM_GBS, 4),
            },
            "clocks": clk,
            "e2e": {"value": round(job_rate(flops_p, ws, ms_e2e) / 1e9, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(ms_e2e, 4),
                    "runs_ms_per_step": [round(x, 4) for x in e2e_runs],
                    "output_copied_back_matches_device": e2e_o_match,
                    "what": "one prefill + one decode per step through the C ABI, like the timed "
                            "step: H2D of prefill q,k,v and of decode's 64 query tokens and "
                            "new K/V rows (appended into the device-resident KV cache), both "
                            "kernels, D2H of both outputs; steps pipelined over two buffer sets "
                            "(copies overlap the previous step's kernels). value = prefill's "
                            "algorithmic FLOPs / the whole step's time (prefill + decode), "
                            "comparable with ms_per_step; median of three timed runs"},
            "gpu_launches": args.steps * 3,
        }
    # CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only); the
    # same oracle results give the parity block against the GPU outputs.
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        base, par = cpu_baseline(q, k, v, pcfg, lam_p, args.cpu_seconds, gpu_out,
                                 decode=(dq, dk, dv, dcfg, lam_d))
        line["cpu_baseline"] = base
        line["parity"] = par
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()


def _time_ms(fn, iters=6, warmup=3, batches=5):
    """Median over `batches` of the mean device time of `iters` back-to-back
    calls (CUDA events on the current stream).  Back to back, the host's
    per-call work (argument checks, marshalling, launch) overlaps the previous
    call's kernels instead of leaving the GPU idle between two events."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(batches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / iters)
    ts.sort()
    return ts[len(ts) // 2]


def run_suite(args):
    """Every workload of the plan: calibrated sparsity points, dense path,
    (A, B) fits, and the calibration-stability sweep.  One JSON line each."""
    import numpy as np
    import torch

    import block_sparse_attention_sm_gb300 as ss
    from block_sparse_attention_sm_gb300 import capi, synth

    ss.build()
    peaks = _peaks()
    dev = torch.device("cuda", 0)

    def emit(d):
        print(json.dumps(d), flush=True)

    def prefill_points(name, targets):
        inp, cfg = synth.make(name, seed=0, device=dev)
        q, k, v = inp.q, inp.k, inp.v
        B, Hq, Lq, d = q.shape
        Lk = k.shape[2]
        nqb, nT = -(-Lq // TILE), -(-Lk // TILE)
        cnt = torch.zeros(B * Hq * nqb, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        # evaluated (unit, tile) pairs: causal blocks stop at the diagonal
        per_head = 0
        for qb in range(nqb):
            rows = min(TILE, Lq - qb * TILE)
            last = qb * TILE + rows - 1 + (Lk - Lq)
            per_head += (min(nT, last // TILE + 1) if cfg["causal"] else nT) if last >= 0 else 0
        n_eval = per_head * B * Hq
        dense_eq = 4.0 * B * Hq * Lq * Lk * d * (0.5 if cfg["causal"] else 1.0)
        fit_s, fit_a, dense_ms = [], [], None
        for s_t in targets:
            a = 0.0
            if s_t > 0:
                a, _ = ss.calibrate("prefill", q, k, v, scale=cfg["scale"], target_sparsity=s_t,
                                    causal=cfg["causal"])
            lam = min(1.0, a / Lk)
            ms = _time_ms(lambda: ss.prefill(q, k, v, scale=cfg["scale"], causal=cfg["causal"],
                                             lam=lam, counts=cnt, out=o))
            sk = int(cnt.sum())
            kept = n_eval - sk
            flops = 2.0 * TILE * TILE * d * (n_eval + kept)
            if s_t == 0:
                dense_ms = ms
            if s_t > 0 and a > 0:
                fit_s.append(sk / n_eval)
                fit_a.append(a)
            # at d = 64 and 128 both prefill kernels run every mode: time each
            # one explicitly beside the library's own choice
            per_kernel = {}
            if d in (64, 128):
                for kname, kid in (("one_cta", 1), ("pair", 2)):
                    def run(kid=kid):
                        st = capi.ss_attn_prefill_ex(q, k, v, o, B, Hq, k.shape[1], Lq, Lk, d,
                                                     cfg["scale"], cfg["causal"], lam, cnt,
                                                     prefill_kernel=kid)
                        if st != 0:
                            raise RuntimeError(capi.ss_status_string(st))
                    per_kernel[kname] = round(_time_ms(run), 4)
            emit({"suite": name, "kind": "prefill", "target": s_t, "a": a, "lambda": lam,
                  "sparsity": round(sk / n_eval, 4), "ms": round(ms, 4),
                  "tflops_executed": round(flops / ms / 1e9, 1),
                  "tflops_dense_equivalent": round(dense_eq / ms / 1e9, 1),
                  "frac_of_peak": round(flops / ms / 1e9 / peaks["bf16"], 4),
                  "speedup_vs_dense": round(dense_ms / ms, 3) if dense_ms else None,
                  "ms_by_kernel": per_kernel or None})
        if len(fit_s) >= 2:
            A, Bc = ss.fit_factor(fit_s, fit_a)
            emit({"suite": name, "kind": "fit", "A": A, "B": Bc, "points": list(zip(fit_s, fit_a))})
        del q, k, v, o, inp
        torch.cuda.empty_cache()

    def decode_points(name, targets):
        inp, cfg = synth.make(name, seed=0, device=dev)
        q, k, v = inp.q, inp.k, inp.v
        B, Hq, d = q.shape
        Hkv, Lk = k.shape[1], k.shape[2]
        S = cfg["num_splits"]
        nT = -(-Lk // TILE)
        cnt = torch.zeros(B * Hkv * S, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        wsb, _ = ss.decode_workspace(B, Hq, d, S, dev)
        n_eval = B * Hkv * nT
        fit_s, fit_a, dense_ms = [], [], None
        for s_t in targets:
            a = 0.0
            if s_t > 0:
                a, _ = ss.calibrate("decode", q, k, v, scale=cfg["scale"], target_sparsity=s_t,
                                    num_kv_splits=S)
            lam = min(1.0, a / Lk)
            ms = _time_ms(lambda: ss.decode(q, k, v, scale=cfg["scale"], lam=lam, num_kv_splits=S,
                                            counts=cnt, out=o, workspace=wsb))
            sk = int(cnt.sum())
            kept = n_eval - sk
            byts = B * Hkv * Lk * d * 2 + kept * TILE * d * 2 + 2 * B * Hq * d * 2
            if s_t == 0:
                dense_ms = ms
            if s_t > 0 and a > 0:
                fit_s.append(sk / n_eval)
                fit_a.append(a)
            emit({"suite": name, "kind": "decode", "target": s_t, "a": a, "lambda": lam,
                  "sparsity": round(sk / n_eval, 4), "ms": round(ms, 4),
                  "gbs": round(byts / ms / 1e6, 1), "frac_of_peak": round(byts / ms / 1e6 / peaks["hbm"], 4),
                  "tokens_per_s": round(B / ms * 1e3, 1),
                  "speedup_vs_dense": round(dense_ms / ms, 3) if dense_ms else None})
        if len(fit_s) >= 2:
            A, Bc = ss.fit_factor(fit_s, fit_a)
            emit({"suite": name, "kind": "fit", "A": A, "B": Bc, "points": list(zip(fit_s, fit_a))})
        del q, k, v, o, inp
        torch.cuda.empty_cache()

    def stability(target=0.7, ref_L=32768):
        """Calibrate a at one length, then hold a (lambda = a/L) or hold lambda
        fixed and measure the skipped fraction at other lengths.  Count-only."""
        from block_sparse_attention_sm_gb300 import capi

        Ls = [4096, 8192, 16384, 32768, 65536, 131072]
        res = {}
        for L in Ls:
            inp = synth.decode_inputs(B=8, Hq=32, Hkv=8, Lk=L, d=128, hot_frac=0.10, seed=3,
                                      device=dev)
            res[L] = inp
        q, k, v = res[ref_L].q, res[ref_L].k, res[ref_L].v
        scale = 128 ** -0.5
        a, _ = ss.calibrate("decode", q, k, v, scale=scale, target_sparsity=target, num_kv_splits=1)
        lam_fixed = a / ref_L
        for L in Ls:
            inp = res[L]
            nT = -(-L // TILE)
            cnt = torch.zeros(8 * 8, dtype=torch.int32, device=dev)
            out = {}
            for tag, lam in (("lambda_a_over_L", min(1.0, a / L)), ("fixed_lambda", lam_fixed)):
                st = capi.ss_attn_decode_ex(inp.q, inp.k, inp.v, None, 8, 32, 8, L, 128, scale, lam,
                                            1, cnt, None, 0, count_only=True)
                assert st == capi.SS_OK
                torch.cuda.synchronize()
                out[tag] = round(int(cnt.sum()) / (64 * nT), 4)
            emit({"suite": "calibration_stability", "L": L, "a": a, "calibrated_at": ref_L,
                  "target": target, **out})
        del res
        torch.cuda.empty_cache()

    def mla_points(name, targets):
        """Latent-attention decode: the cache is read once (the values are its
        latent part, already on chip); bytes = cache + q + o."""
        inp, cfg = synth.make(name, seed=0, device=dev,
                              **({"B": args.mla_batch} if args.mla_batch else {}))
        q, kv = inp.q, inp.kv
        B, Hq, dk = q.shape
        Lk = kv.shape[1]
        S = cfg["num_splits"]
        nT = -(-Lk // TILE)
        cnt = torch.zeros(B * S, dtype=torch.int32, device=dev)
        o = torch.empty(B, Hq, cfg["d_latent"], dtype=q.dtype, device=dev)
        wsb, _ = ss.mla_workspace(B, Hq, S, dev)
        n_eval = B * nT
        byts = B * Lk * dk * 2 + B * Hq * (dk + cfg["d_latent"]) * 2
        flops_tile = 2.0 * TILE * Hq * dk  # scores of one tile; P.V adds 2*128*Hq*512 if kept
        fit_s, fit_a, dense_ms = [], [], None
        for s_t in targets:
            a = 0.0
            if s_t > 0:
                a, _ = ss.calibrate("mla_decode", q, kv, None, scale=cfg["scale"],
                                    target_sparsity=s_t, num_kv_splits=S)
            lam = min(1.0, a / Lk)
            ms = _time_ms(lambda: ss.mla_decode(q, kv, scale=cfg["scale"], lam=lam, num_kv_splits=S,
                                                counts=cnt, out=o, workspace=wsb))
            sk = int(cnt.sum())
            kept = n_eval - sk
            if s_t == 0:
                dense_ms = ms
            if s_t > 0 and a > 0:
                fit_s.append(sk / n_eval)
                fit_a.append(a)
            flops = flops_tile * n_eval + 2.0 * TILE * Hq * cfg["d_latent"] * kept
            emit({"suite": name, "kind": "mla_decode", "target": s_t, "a": a, "lambda": lam,
                  "sparsity": round(sk / n_eval, 4), "ms": round(ms, 4),
                  "gbs": round(byts / ms / 1e6, 1), "frac_of_peak": round(byts / ms / 1e6 / peaks["hbm"], 4),
                  "tflops_executed": round(flops / ms / 1e9, 1),
                  "tokens_per_s": round(B / ms * 1e3, 1),
                  "speedup_vs_dense": round(dense_ms / ms, 3) if dense_ms else None})
        if len(fit_s) >= 2:
            A, Bc = ss.fit_factor(fit_s, fit_a)
            emit({"suite": name, "kind": "fit", "A": A, "B": Bc, "points": list(zip(fit_s, fit_a))})
        del q, kv, o, inp
        torch.cuda.empty_cache()

    def sdpa_points(name):
        """Sanity check of the dense denominator: PyTorch's
        scaled_dot_product_attention (its default backend on this GPU) against
        this library's lambda = 0 path, same bf16 inputs and shapes."""
        import torch.nn.functional as F

        inp, cfg = synth.make(name, seed=0, device=dev)
        q, k, v = inp.q, inp.k, inp.v
        B, Hq, Lq, d = q.shape
        Hkv, Lk = k.shape[1], k.shape[2]
        causal = cfg["causal"]
        flops = 4.0 * B * Hq * Lq * Lk * d * (0.5 if causal else 1.0)
        o = torch.empty_like(q)
        ms_own = _time_ms(lambda: ss.prefill(q, k, v, scale=cfg["scale"], causal=causal, lam=0.0, out=o))
        kw = {"enable_gqa": True} if Hkv != Hq else {}
        ms_sdpa = _time_ms(lambda: F.scaled_dot_product_attention(q, k, v, is_causal=causal,
                                                                   scale=cfg["scale"], **kw))
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=cfg["scale"], **kw)
        diff = (ref.float() - o.float()).abs()
        emit({"suite": name, "kind": "sdpa_sanity", "own_dense_ms": round(ms_own, 4),
              "own_dense_tflops": round(flops / ms_own / 1e9, 1), "sdpa_ms": round(ms_sdpa, 4),
              "sdpa_tflops": round(flops / ms_sdpa / 1e9, 1),
              "own_vs_sdpa": round(ms_sdpa / ms_own, 3),
              "max_abs_diff": round(float(diff.max()), 5), "mean_abs_diff": float(diff.mean())})
        del q, k, v, o, ref, inp
        torch.cuda.empty_cache()

    def mla_paged_points():
        """Paged, ragged latent-attention decode: 128 sequences of 8K..32K
        rows in shuffled pages of 128, lambda_b = a / L_b with the a
        calibrated for 70% on the contiguous 32K cache of the same data."""
        from block_sparse_attention_sm_gb300 import capi

        B, Hq, S, Lmax = (args.mla_batch or 128), 16, 4, 32768
        rng = np.random.default_rng(9)
        lens = [int(x) for x in rng.integers(8192, Lmax + 1, size=B)]
        inp = synth.mla_decode_inputs(B=B, Hq=Hq, Lk=Lmax, hot_frac=0.10, seed=0, device=dev)
        q, kv = inp.q, inp.kv
        scale = 192 ** -0.5
        a, _ = ss.calibrate("mla_decode", q, kv, None, scale=scale, target_sparsity=0.7,
                            num_kv_splits=S)
        npg = [-(-L // TILE) for L in lens]
        num_pages, max_pages = sum(npg), max(npg)
        perm = torch.from_numpy(rng.permutation(num_pages)).to(dev)
        pages = torch.empty(num_pages, TILE, kv.shape[2], dtype=kv.dtype, device=dev)
        table = torch.zeros(B, max_pages, dtype=torch.int32, device=dev)
        off = 0
        for b, n in enumerate(npg):
            pg = perm[off:off + n]
            off += n
            pages[pg] = kv[b, :n * TILE].reshape(n, TILE, kv.shape[2])
            table[b, :n] = pg.to(torch.int32)
        del inp, kv
        torch.cuda.empty_cache()
        lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
        cnt = torch.zeros(B * S, dtype=torch.int32, device=dev)
        o = torch.empty(B, Hq, 512, dtype=q.dtype, device=dev)
        wsn = capi.ss_attn_mla_decode_workspace_size(B, Hq, 512, S)
        ws = torch.empty(wsn, dtype=torch.uint8, device=dev)
        n_eval = num_pages
        byts = sum(lens) * 576 * 2 + B * Hq * (576 + 512) * 2
        dense_ms = None
        for tag, aa in (("dense", 0.0), ("a_for_70pct_at_32k", a)):
            def run():
                st = capi.ss_attn_mla_decode_paged(q, pages, table, lens_t, o, B, Hq, num_pages,
                                                   max_pages, 512, 64, scale, aa, S, cnt, ws, wsn)
                if st != capi.SS_OK:
                    raise SystemExit(capi.ss_status_string(st))
            ms = _time_ms(run)
            sk = int(cnt.sum())
            if aa == 0.0:
                dense_ms = ms
            emit({"suite": "mla_paged_decode_ragged", "kind": "mla_decode", "point": tag, "a": aa,
                  "lens": [min(lens), max(lens), sum(lens) // B], "pages": num_pages,
                  "sparsity": round(sk / n_eval, 4), "ms": round(ms, 4),
                  "gbs": round(byts / ms / 1e6, 1), "frac_of_peak": round(byts / ms / 1e6 / peaks["hbm"], 4),
                  "tokens_per_s": round(B / ms * 1e3, 1),
                  "speedup_vs_dense": round(dense_ms / ms, 3) if dense_ms else None})
        del q, pages, o
        torch.cuda.empty_cache()

    def paged_points():
        """Paged, ragged decode: 64 sequences of 8K..32K keys in shuffled pages
        of 128 keys, lambda_b = a / L_b per sequence with the a calibrated for
        70% on the contiguous 32K cache of the same data; dense and sparse."""
        from block_sparse_attention_sm_gb300 import capi

        B, Hq, Hkv, d, S, Lmax = 64, 32, 8, 128, 8, 32768
        rng = np.random.default_rng(7)
        lens = [int(x) for x in rng.integers(8192, Lmax + 1, size=B)]
        inp = synth.decode_inputs(B=B, Hq=Hq, Hkv=Hkv, Lk=Lmax, d=d, hot_frac=0.10, seed=0,
                                  device=dev)
        q, k, v = inp.q, inp.k, inp.v
        scale = d ** -0.5
        a, _ = ss.calibrate("decode", q, k, v, scale=scale, target_sparsity=0.7, num_kv_splits=S)
        npg = [-(-L // TILE) for L in lens]
        num_pages, max_pages = sum(npg), max(npg)
        perm = torch.from_numpy(rng.permutation(num_pages)).to(dev)
        kp = torch.empty(num_pages, Hkv, TILE, d, dtype=k.dtype, device=dev)
        vp = torch.empty_like(kp)
        table = torch.zeros(B, max_pages, dtype=torch.int32, device=dev)
        off = 0
        for b, n in enumerate(npg):
            pg = perm[off:off + n]
            off += n
            kp[pg] = k[b, :, :n * TILE].reshape(Hkv, n, TILE, d).permute(1, 0, 2, 3)
            vp[pg] = v[b, :, :n * TILE].reshape(Hkv, n, TILE, d).permute(1, 0, 2, 3)
            table[b, :n] = pg.to(torch.int32)
        del inp, k, v
        torch.cuda.empty_cache()
        lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
        cnt = torch.zeros(B * Hkv * S, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        wsn = capi.ss_attn_decode_workspace_size(B, Hq, d, S)
        ws = torch.empty(wsn, dtype=torch.uint8, device=dev)
        n_eval = Hkv * num_pages
        dense_ms = None
        for tag, aa in (("dense", 0.0), ("a_for_70pct_at_32k", a)):
            def run():
                st = capi.ss_attn_decode_paged(q, kp, vp, table, lens_t, o, B, Hq, Hkv, num_pages,
                                               max_pages, d, scale, aa, S, cnt, ws, wsn)
                if st != capi.SS_OK:
                    raise SystemExit(capi.ss_status_string(st))
            ms = _time_ms(run)
            sk = int(cnt.sum())
            kept = n_eval - sk
            byts = Hkv * sum(lens) * d * 2 + kept * TILE * d * 2 + 2 * B * Hq * d * 2
            if aa == 0.0:
                dense_ms = ms
            emit({"suite": "paged_decode_ragged", "kind": "decode", "point": tag, "a": aa,
                  "lens": [min(lens), max(lens), sum(lens) // B], "pages": num_pages,
                  "sparsity": round(sk / n_eval, 4), "ms": round(ms, 4),
                  "gbs": round(byts / ms / 1e6, 1), "frac_of_peak": round(byts / ms / 1e6 / peaks["hbm"], 4),
                  "tokens_per_s": round(B / ms * 1e3, 1),
                  "speedup_vs_dense": round(dense_ms / ms, 3) if dense_ms else None})
        del q, kp, vp, o
        torch.cuda.empty_cache()

    parts = set(filter(None, args.suite_only.split(","))) or {"prefill", "chunked", "decode", "paged",
                                                                  "mla", "sdpa", "stability"}
    if "prefill" in parts:
        prefill_points("tiny_prefill", [0.0, 0.5, 0.75])
        prefill_points("dit_prefill_32k", [0.0, 0.5, 0.7])
        prefill_points("dit_prefill_32k_d64", [0.0, 0.5, 0.7])
        prefill_points("llama_prefill_16k", [0.0, 0.5, 0.7])
    if "chunked" in parts:
        prefill_points("llama_chunked_prefill_2k_on_32k", [0.0, 0.5, 0.7, 0.9])
    if "decode" in parts:
        decode_points("llama_decode_32k", [0.0, 0.5, 0.7])
        decode_points("mqa_decode_32k", [0.0, 0.5, 0.7])
    if "prefill" in parts:
        prefill_points("long_prefill_128k", [0.0, 0.5, 0.7, 0.9])
    if "decode" in parts:
        decode_points("long_decode_128k", [0.0, 0.5, 0.7, 0.9])
    if "paged" in parts:
        paged_points()
    if "mla" in parts:
        mla_points("mla_decode_32k", [0.0, 0.5, 0.7, 0.9])
        mla_points("mla_decode_32k_32h", [0.0, 0.7])
        mla_points("mla_decode_32k_64h", [0.0, 0.7])
        mla_paged_points()
    if "sdpa" in parts:
        sdpa_points("dit_prefill_32k")
        sdpa_points("llama_prefill_16k")
    if "stability" in parts:
        stability()


def _parity_units(rng, n, k=6):
    """First, last and k random indices of range(n), in that order."""
    rest = [int(x) for x in rng.permutation(np.arange(1, max(1, n - 1)))[:k]] if n > 2 else []
    return list(dict.fromkeys([0, n - 1] + rest))


def _compare_unit(stats, g_mask, g_margin, g_count, g_o, res_mask, res_margin, res_count, res_o,
                  lam):
    """Fold one unit's GPU-vs-oracle comparison into `stats` (acceptance of the
    parity tests: decisions exact outside the near-margin band, counts exact
    and outputs within max-abs / mean-abs on units whose decisions agree)."""
    ln_lam = math.log(lam) if lam > 0 else -math.inf
    ev = res_mask != 2
    near = ev & (np.abs(res_margin - ln_lam) < 1e-2)
    dis = (g_mask.astype(np.int64) != res_mask.astype(np.int64))
    stats["units"] += 1
    stats["tiles"] += int(ev.sum())
    stats["skipped"] += int((g_mask == 1).sum())
    stats["near_margin_tiles"] += int(near.sum())
    stats["near_margin_disagreements"] += int((dis & near).sum())
    stats["other_disagreements"] += int((dis & ~near).sum())
    if not dis.any():
        stats["count_mismatches"] += int(np.any(np.asarray(g_count) != np.asarray(res_count)))
        err = np.abs(g_o.astype(np.float64) - res_o)
        stats["max_abs"] = max(stats["max_abs"], float(err.max(initial=0.0)))
        stats["mean_abs"] = max(stats["mean_abs"], float(err.mean()) if err.size else 0.0)


def _new_stats(lam):
    return {"lambda": lam, "units": 0, "tiles": 0, "skipped": 0, "near_margin_tiles": 0,
            "near_margin_disagreements": 0, "other_disagreements": 0, "count_mismatches": 0,
            "max_abs": 0.0, "mean_abs": 0.0}


def cpu_baseline(q, k, v, cfg, lam, seconds_budget, gpu_out=None, decode=None):
    """Time the fp64 oracle (as it stands) on whole query blocks of the
    prefill workload; report TFLOP/s on the same algorithmic FLOP count.

    The same oracle results are compared with the GPU's outputs of the timed
    launch (gpu_out: o, counters, skip mask and vote margins) on those query
    blocks -- the first, the last, then random ones of head 0 -- and, with
    `decode`, on eight sampled (sequence, KV head) units of the decode
    workload; that comparison is returned as the parity block."""
    import oracle

    oracle.build()
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    h = 0
    qs, ks, vs = q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1]
    qb_h = oracle._bits(qs)
    kb_h = oracle._bits(ks)
    vb_h = oracle._bits(vs)
    Lk = k.shape[2]
    nT = -(-Lk // TILE)
    d = q.shape[3]
    nqb = q.shape[2] // TILE
    rng = np.random.default_rng(2024)
    order = _parity_units(rng, nqb, k=nqb)  # first, last, then the rest shuffled
    gp = None
    if gpu_out is not None:
        gp = {key: (val.cpu().numpy() if key != "o" else val[0, h].float().cpu().numpy())
              for key, val in gpu_out["prefill"].items()}
    pstats = _new_stats(lam)
    # probe one unit per core to size the sample to the budget
    n = cores
    done_units, done_s, done_flops = 0, 0.0, 0.0
    while True:
        units = np.array(order[done_units:done_units + n])
        t0 = time.time()
        res = oracle.prefill(qb_h, kb_h, vb_h, scale=cfg["scale"], causal=False, lam=lam,
                             units=units)
        dt = time.time() - t0
        kept = int((res.mask == 0).sum())
        done_flops += 2 * TILE * TILE * d * (len(units) * nT + kept)
        done_units += len(units)
        done_s += dt
        if gp is not None:
            for i, qb in enumerate(units.tolist()):
                gid = h * nqb + qb
                _compare_unit(pstats, gp["mask"][gid], gp["margin"][gid], gp["counts"][gid],
                              gp["o"][qb * TILE:(qb + 1) * TILE], res.mask[i], res.margin[i],
                              res.counts[i], res.o[i], lam)
        if done_s > seconds_budget * 0.5 or done_units >= nqb:
            break
        n = max(cores, int(n * max(1.0, (seconds_budget - done_s) / max(dt, 1e-3) * 0.8)))
        n = min(n, nqb - done_units)
        if n <= 0:
            break
    base = {"value": round(done_flops / done_s / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{done_units} query blocks (128 rows x 32768 keys, head 0: the first, "
                      f"the last, then seeded random ones) of {PREFILL} at the same lambda, "
                      f"{done_s:.1f} s wall"}
    if gpu_out is None:
        return base, None
    par = {"prefill": pstats,
           "debug_call_equals_timed_call": gpu_out["debug_call_equals_timed_call"],
           "tolerance": {"max_abs": 2e-2, "mean_abs": 2e-3, "near_margin_log": 1e-2}}
    if decode is not None:
        dq, dk, dv, dcfg, lam_d = decode
        dB, dHq, _ = dq.shape
        dHkv = dk.shape[1]
        G = dHq // dHkv
        S = dcfg["num_splits"]
        gd = {key: val.cpu().numpy() if key != "o" else val.float().cpu().numpy()
              for key, val in gpu_out["decode"].items()}
        dstats = _new_stats(lam_d)
        for u in _parity_units(rng, dB * dHkv):
            b, kvh = divmod(u, dHkv)
            res = oracle.decode(dq[b:b + 1, kvh * G:(kvh + 1) * G], dk[b:b + 1, kvh:kvh + 1],
                                dv[b:b + 1, kvh:kvh + 1], scale=dcfg["scale"], lam=lam_d,
                                num_splits=S)
            _compare_unit(dstats, gd["mask"][u], gd["margin"][u],
                          gd["counts"].reshape(dB * dHkv, S)[u], gd["o"][b, kvh * G:(kvh + 1) * G],
                          res.mask[0], res.margin[0], res.counts[0], res.o[0], lam_d)
        par["decode"] = dstats
    par["pass"] = all(st_["other_disagreements"] == 0 and st_["count_mismatches"] == 0
                      and st_["max_abs"] <= 2e-2 and st_["mean_abs"] <= 2e-3
                      for key, st_ in par.items() if key in ("prefill", "decode"))
    return base, par


def run_reference(args):
    """The oracle as the reference arm: same workload, metric and unit."""
    import numpy as np
    import torch

    import oracle
    from block_sparse_attention_sm_gb300 import synth

    ws, rank, _ = _dist()
    if rank != 0:
        return
    oracle.build()
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    # Same generator, one head on the host (the oracle runs per query block).
    inp = synth.prefill_inputs(B=1, Hq=1, Hkv=1, Lq=32768, Lk=32768, d=128, hot_frac=0.15,
                               seed=0, per_head_u=False, device="cpu")
    cfg = synth.WORKLOADS[PREFILL]
    qb_h, kb_h, vb_h = (oracle._bits(t) for t in (inp.q, inp.k, inp.v))
    # lambda: the oracle's own order-statistic calibration to 70% on a sample
    nT = 256
    cal_units = np.arange(0, 256, 32)
    r0 = oracle.prefill(qb_h, kb_h, vb_h, scale=cfg["scale"], causal=False, lam=0.0,
                        units=cal_units)
    a, _, _ = oracle.calibrate(r0.margin, r0.mask, TARGET, 32768)
    lam = a / 32768
    per_step = max(1, cores)
    times, flops = [], []
    step = 0
    for i in range(args.warmup + args.steps):
        units = (np.arange(per_step) + i * per_step) % 256
        t0 = time.time()
        res = oracle.prefill(qb_h, kb_h, vb_h, scale=cfg["scale"], causal=False, lam=lam,
                             units=units)
        dt = time.time() - t0
        if i >= args.warmup:
            kept = int((res.mask == 0).sum())
            times.append(dt)
            flops.append(2 * TILE * TILE * 128 * (len(units) * nT + kept))
            step += 1
    value = sum(flops) / sum(times) / 1e12
    ms = sum(times) / len(times) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded generator)",
        "config": {"workload": f"{PREFILL} (one head on the host), lambda from the oracle's "
                               f"order-statistic calibration to {TARGET}",
                   "units_per_step": per_step},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{per_step} query blocks (128 x 32768 keys) per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite-only", default="",
                    help="with --suite: run only the named parts (comma-separated: prefill, chunked, decode, paged, mla, sdpa, stability)")
    ap.add_argument("--suite", action="store_true",
                    help="measure every workload (calibrated sweeps, fits, stability); JSON lines")
    ap.add_argument("--profile", action="store_true",
                    help="run calibration + the timed loop only (for ncu); prints nothing")
    ap.add_argument("--profile-dense", action="store_true",
                    help="with --profile: run the timed loop at lambda = 0 (the dense path)")
    ap.add_argument("--prefill-heads", type=int, default=0,
                    help="profiling: shrink the prefill workload to this many heads")
    ap.add_argument("--decode-workload", default=DECODE, choices=[DECODE, "mqa_decode_32k"],
                    help="with --profile: the decode workload to run (multi-query: 32 heads on one KV head)")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="profiling: shrink the decode workload to this many sequences")
    ap.add_argument("--mla-batch", type=int, default=0,
                    help="profiling: shrink the latent-attention suite workloads to this many sequences")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.suite:
        run_suite(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
