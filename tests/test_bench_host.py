"""Host-side logic of bench.py: byte accounting, the multi-rank reduction (gloo, 2 ranks on
CPU) and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_match_the_scope_table():
    wl = workloads.config(1)
    P = wl.N * wl.T * wl.R
    ab = bench.algorithmic_bytes(wl, P, P)
    assert ab["pack"] == wl.N * wl.T * (1 + wl.R) * 2 * wl.H == 132_120_576
    assert ab["scatter"] == ab["unpack"] == 2 * P * 2 * wl.H == 234_881_024
    assert ab["combine_pack"] + ab["combine_scatter"] == 469_762_048
    assert ab["combine_reduce"] == wl.N * wl.T * (wl.R + 1) * 2 * wl.H
    # the one-kernel phases: one read of each row, every write of the kernels they stand for
    assert ab["dispatch_fused"] == ab["pack"] + ab["scatter"] + ab["unpack"] - 2 * P * 2 * wl.H
    assert ab["combine_fused"] == (ab["combine_pack"] + ab["combine_scatter"] + ab["combine_reduce"]
                                   - 2 * P * 2 * wl.H)
    f = workloads.config(3)
    Pf = f.N * f.T * f.R
    abf = bench.algorithmic_bytes(f, Pf, Pf)
    assert abf["pack"] == f.N * f.T * (1 + f.R) * 7392 == 136_249_344
    assert abf["combine_reduce"] == f.N * f.T * (f.R + 1) * 2 * f.H == 264_241_152
    assert abf["quant_dispatch_fused"] == abf["quant_pack"] + 2 * Pf * 7392


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    d = bench.dist_init("gloo")
    v = bench.max_over_ranks(1.5 + rank, d)
    bench.barrier(d)
    q.put((rank, v))
    d.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_cpu_baseline_reports_single_thread_and_all_cores():
    wl = workloads.config(0)
    inp = workloads.make_inputs(wl)
    cb = bench.cpu_baseline(wl, inp, 0.2)
    out = cb.pop("out")
    assert out.shape == (wl.N, wl.T, wl.H)
    assert cb["cores"] == 1 and cb["value"] > 0
    ac = cb["all_cores"]
    assert ac["kind"] == "oracle" and ac["cores"] >= 1 and ac["value"] > 0
    assert f"{ac['cores']} threads" in ac["sample"]
