"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The decode GEMV and the MoE layer are independent per GPU: with N GPUs the
benchmark runs N replicas of the same workload (weak scaling, no collective on
the data path).  What crosses ranks is host-side only: the rendezvous, the
barriers around the timed region, the maximum of the ranks' times and the
whole-job value built from it.  These tests run that logic as two gloo ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w = bench.dist_init(world)
    bench.barrier(w)
    # rank-dependent "times": every rank must see the slowest one
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)
    value = bench.job_gbps(1e9, w, slowest)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": slowest, "value": value}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, g in enumerate(got):
        assert g["rank"] == r and g["world"] == world
        assert g["max"] == pytest.approx(15.0)  # rank 1's 15 ms, seen by both ranks
        # 1 GB per rank per step, two ranks, 15 ms per step -> 2 GB / 15 ms
        assert g["value"] == pytest.approx(2.0 / 0.015)


def test_job_value_is_weak_scaling_over_the_slowest_rank():
    sys.path.insert(0, ROOT)
    import bench

    one = bench.job_gbps(735838208, 1, 0.25)
    assert one == pytest.approx(735838208 / 0.25e-3 / 1e9)
    assert bench.job_gbps(735838208, 4, 0.25) == pytest.approx(4 * one)
    # a slower step lowers the job value in proportion
    assert bench.job_gbps(735838208, 4, 0.5) == pytest.approx(2 * one)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the
    oracle and prints the one JSON line, the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the contract's keys
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["steps"] == 1 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and "workload" in line["config"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    cb = line["cpu_baseline"]
    assert cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
