"""The multi-rank path of bench.py on CPU: two gloo ranks agree on the
slowest rank's time, the job throughput counts every rank's keys, ranks draw
disjoint inputs, and the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as tdist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(True)
        ms = [3.0, 7.5][rank]  # this rank's timed region
        out[rank] = bench.max_over_ranks_of(ms, True, "cpu")
        bench.rank_barrier(True)
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        assert dict(out) == {0: 7.5, 1: 7.5}


def test_single_rank_keeps_its_time():
    assert bench.max_over_ranks_of(4.25, False, "cpu") == 4.25


def test_job_throughput_counts_every_rank():
    # each of 4 ranks scans 1e9 keys in the timed region; the slowest takes 250 ms
    assert bench.job_throughput(1e9, 4, 250.0) == 16e9
    assert bench.job_throughput(1e9, 1, 250.0) == 4e9


def test_ranks_draw_disjoint_inputs():
    seeds = {bench.rank_seed(r, li) for r in range(8) for li in range(8)}
    assert len(seeds) == 64


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny-4k",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "keys/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["cpu_model"]
    assert line["cpu_baseline"]["single_thread"]["cores"] == 1 and line["cpu_baseline"]["single_thread"]["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
