"""Host-side logic of bench.py, on CPU: cross-rank reductions under gloo with two
ranks, and the reference (oracle) arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mx = bench.max_over_ranks(1.5 + rank, world, "cpu")
        sm = bench.sum_over_ranks(10.0 * (rank + 1), world, "cpu")
        results[rank] = (mx, sm)
    finally:
        dist.destroy_process_group()


def test_cross_rank_reductions_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert results[0] == results[1] == (2.5, 30.0)


def test_single_rank_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.sum_over_ranks(4.0, 1, "cpu") == 4.0


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object as the GPU arm's line (152 SMs assumed without a GPU, one of
    # them kept for the next batch's loads and plan)
    sys.path.insert(0, ROOT)
    import bench
    from load_balancing_gb300 import workloads as W

    w = W.WORKLOADS[bench.WORKLOAD]
    mask_np = W.make_mask(w)
    assert d["config"] == bench.bench_config(w, bench.attention_workers(152), bench.dense_blocks(mask_np, w.causal))
    assert d["config"]["n_workers"] == 151


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("PATH", "/nonexistent")
    s = bench.ClockSampler(0)
    s.start()
    out = s.stop()
    assert out["sm_mhz"] is None
