"""bench.py host logic on the CPU: multi-rank max timing over gloo
(world_size 2), whole-job throughput, and the reference (oracle) arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 19.0][rank]          # the slow rank decides the job time
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        dist.barrier()
        value = bench.job_tflops(1e12, ms, world)
        out.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 19.0
        assert value == pytest.approx(2 * 1e12 / 19e-3 / 1e12)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(2e12, 1000.0, 1) == pytest.approx(2.0)


def test_workload_lookup_and_flops():
    w = bench.workload_by_name("long-64k")
    assert (w.T, w.Hq, w.Hk, w.d, w.L) == (65536, 16, 4, 128, 48)
    assert w.flops() == 4 * 128 * 16 * (65536 * 65537 / 2 + 65536 * 48)
    with pytest.raises(SystemExit):
        bench.workload_by_name("nope")


def test_reference_arm_prints_contract_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "2", "--warmup", "1", "--cpu-seconds", "0.3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_reference_arm_other_ranks_exit_quietly():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.1"]
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""
