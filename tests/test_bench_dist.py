"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

One process per GPU runs an independent replica of the workload (the units
shard with no exchange), the job time is the slowest rank's, and the whole-job
rate is the ranks' total work over that time.  These tests run the same
host code on CPU processes instead of GPUs.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    assert bench._dist() == (ws, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    # rank r was slower on the first value, faster on the second
    got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.5], ws)
    out[rank] = torch.tensor(got + [bench.job_rate(100.0, ws, got[0])], dtype=torch.float64)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo_world_size_2():
    ws = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, out)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(ws):
        t = out[r].tolist()
        assert t[:3] == [2.0, 5.0, 2.5]       # element-wise maximum over the ranks
        assert t[3] == pytest.approx(100.0 * ws / 2.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3, 4], 1) == [3.0, 4.0]
    assert bench.job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun the oracle baseline runs on rank 0 only; other ranks
    print nothing and exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_clock_samples_summary():
    """The clocks record of the bench line: median SM clock under load, the
    maximum, and the throttle reasons seen active (what decides whether a
    number is kept)."""
    sys.path.insert(0, ROOT)
    import bench

    na = "Not Active"
    lines = [
        f"0, 2070, 2070, 900.1, 0x0, {na}, {na}, {na}, {na}\n",
        f"0, 1980, 2070, 1390.0, 0x4, {na}, {na}, {na}, Active\n",
        f"0, 2010, 2070, 1385.2, 0x4, {na}, {na}, {na}, Active\n",
        f"0, 345, 2070, 120.0, 0x1, {na}, {na}, {na}, {na}\n",  # idle sample: not under load
        "garbled line\n",
    ]
    got = bench.parse_clock_samples(lines)
    assert got["sm_mhz"] == 2010 and got["sm_max_mhz"] == 2070 and got["samples"] == 4
    assert got["reasons"] == ["sw_power_cap"]
    hot = bench.parse_clock_samples([f"0, 1500, 2070, 1400, 0x40, Active, {na}, Active, {na}\n"])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples([])["reasons"] == ["no samples"]


def test_clock_sampler_with_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """ClockSampler start/stop end to end, with a stand-in nvidia-smi on PATH
    that prints two samples and then waits to be terminated."""
    sys.path.insert(0, ROOT)
    import bench

    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 2055, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    cs = bench.ClockSampler(0)
    cs.start()
    got = cs.stop()
    assert got == {"sm_mhz": 2062.5, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 2}
    assert not os.path.exists(cs.path)


def test_reference_arm_line_on_the_host():
    """The reference arm (the oracle on host cores) prints one JSON line with
    the native arm's metric and unit, its core count and zero-byte e2e."""
    import json

    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench

    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["warmup"] >= 3
    assert d["cpu_baseline"]["cores"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]


def test_bench_parity_bookkeeping():
    """The bench's parity block (built in its CPU-baseline leg from the oracle
    results it times) counts near-margin disagreements apart from others, and
    compares counts and outputs only on units whose decisions agree."""
    import numpy as np

    import bench

    lam = 0.01
    ln = np.log(lam)
    st = bench._new_stats(lam)
    mask_o = np.array([0, 1, 1, 2], np.uint8)
    margin_o = np.array([np.inf, ln - 0.5, ln - 0.005, np.nan])
    o_ref = np.zeros((4, 8))
    # unit 1: identical decisions, small output error
    bench._compare_unit(st, mask_o.copy(), margin_o, [2], o_ref + 1e-3, mask_o, margin_o, [2],
                        o_ref, lam)
    # unit 2: the near-margin tile (third) kept by the GPU: counted, output not compared
    g = mask_o.copy()
    g[2] = 0
    bench._compare_unit(st, g, margin_o, [1], o_ref + 1.0, mask_o, margin_o, [2], o_ref, lam)
    assert st["units"] == 2 and st["tiles"] == 6 and st["near_margin_tiles"] == 2
    assert st["near_margin_disagreements"] == 1 and st["other_disagreements"] == 0
    assert st["count_mismatches"] == 0 and abs(st["max_abs"] - 1e-3) < 1e-12
    # unit 3: a disagreement far from the margin is reported as such
    g = mask_o.copy()
    g[1] = 0
    bench._compare_unit(st, g, margin_o, [1], o_ref, mask_o, margin_o, [2], o_ref, lam)
    assert st["other_disagreements"] == 1
    rng = np.random.default_rng(0)
    u = bench._parity_units(rng, 10)
    assert u[:2] == [0, 9] and len(u) == 8 and len(set(u)) == 8
    assert bench._parity_units(rng, 1) == [0]


def test_pair_union_counts_tiles_kept_by_either_block_of_a_pair():
    """The MMA-issued FLOP count of the CTA-pair prefill kernel needs, per
    pair of query blocks (2p, 2p + 1 of one head), the tiles either block
    keeps; an unpaired last block counts alone."""
    import torch

    sys.path.insert(0, ROOT)
    import bench

    # 1 head, 3 query blocks (pair (0, 1) and block 2 alone), 4 tiles;
    # mask values: 0 kept, 1 skipped, 2 not evaluated.
    mask = torch.tensor([[0, 1, 1, 2],
                         [1, 0, 1, 2],
                         [0, 0, 1, 1]], dtype=torch.uint8)
    assert bench.pair_union(mask, 3) == 2 + 2
    # two heads of 2 blocks: union per head
    mask2 = torch.tensor([[0, 1], [0, 1], [1, 1], [1, 0]], dtype=torch.uint8)
    assert bench.pair_union(mask2, 2) == 1 + 1
    assert bench.prefill_mma_flops(10, 3, 128) == 2 * 128 * 128 * 128 * (10 + 6)
