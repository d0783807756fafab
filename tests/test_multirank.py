"""The multi-process side of bench.py without a GPU: two ranks on the gloo
backend (127.0.0.1) agree on the slowest rank's time, and under two ranks the
reference arm prints exactly one line, from rank 0; the all-cores oracle
baseline's spawned processes report or fail fast."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms per step and (20 - r) ms end to end
        got = bench.max_over_ranks(torch, [10.0 + rank, 20.0 - rank], world, device="cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [11.0, 20.0]


def test_max_over_ranks_one_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, [3, 4.5], 1) == [3.0, 4.5]


@pytest.mark.parametrize("workload", ["tiny", "int8-linear"])
def test_reference_arm_prints_once_under_two_ranks(workload):
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                            "--workload", workload, "--steps", "1", "--warmup", "0",
                            "--cpu-budget", "1"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append([ln for ln in r.stdout.splitlines() if ln.strip()])
    assert outs[1] == []
    assert len(outs[0]) == 1
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_all_cores_oracle_baseline():
    """The all-cores CPU baseline: every spawned process reports, and one that
    fails (here: a workload its process cannot build) ends the measurement at
    once with that process's error instead of leaving the others waiting."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from paged_kv_cache_240_gb300 import inputs as I
    oracle.build()
    w = I.make_workload("tiny", seed=0)
    value, procs = bench.cpu_baseline_all_cores(w, 0.5, procs=2)
    assert procs == 2 and value > 0
    with pytest.raises(RuntimeError, match="decoding sequences"):
        bench.cpu_baseline_all_cores(w, 0.5, num_seqs=7, procs=2)
