"""The N > 1 path of bench.py on the CPU: two gloo ranks (127.0.0.1), each
with its own step time, agree on the slowest one, and the job throughput
counts every replica's work against that time; `bench.py --gpus 2` started
without torchrun starts both ranks itself, each on its own device index, and
only rank 0 prints; a --gpus that disagrees with WORLD_SIZE is refused."""
import json
import subprocess
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank            # rank 1 is slower
    m = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = (m, bench.job_throughput(1e12, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        ctx = mp.get_context("spawn")
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 replicas x 1 TFLOP in 15 ms
    assert res[0][1] == pytest.approx(2e12 / 15e-3 / 1e12)


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(2e12, 1, 2.0) == pytest.approx(1000.0)


def _bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_bench_starts_its_own_ranks_without_torchrun():
    r = _bench(["--gpus", "2", "--probe-ranks", "--backend", "gloo"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["backend"] == "gloo"
    ranks = sorted(line["ranks"], key=lambda x: x["rank"])
    assert [x["rank"] for x in ranks] == [0, 1]
    assert [x["device_index"] for x in ranks] == [0, 1]  # one GPU per rank (LOCAL_RANK)
    assert ranks[0]["pid"] != ranks[1]["pid"]


def test_single_gpu_probe_needs_no_process_group():
    r = _bench(["--probe-ranks"])
    assert r.returncode == 0, r.stderr
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert line["n_gpus"] == 1 and line["ranks"][0]["device_index"] == 0


def test_gpus_must_match_world_size():
    r = _bench(["--gpus", "3", "--probe-ranks", "--backend", "gloo"],
               {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0
    assert "does not match WORLD_SIZE" in r.stderr
