"""The N > 1 path of bench.py on the CPU, with two gloo ranks.

The hot path partitions by (batch, head) slice with no exchange, so N GPUs run
N independent replicas: each rank draws its own inputs, the step time is the
slowest rank's (a MAX all-reduce after a barrier), the whole-job rate counts
the tokens of every rank, and the reference arm runs on rank 0 alone.  These
tests run that host logic in two processes over gloo (no GPU, no collective on
the data path)."""
import contextlib
import io
import json
import os
import socket
import types

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    from gaussian_mixture_sequence_gb300 import workloads

    w, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        # the slowest rank's step time, seen by every rank
        ms = bench.max_over_ranks(dist, 1.0 + 0.5 * r, torch.device("cpu"))
        rate = bench.whole_job_rate(w, 1000, ms)
        # every rank's replica has its own inputs
        wl = workloads.WORKLOADS["tiny"].with_(B=1, H=2, N=24)
        q, _, _ = workloads.full_inputs(wl, bench.replica_seed(wl, r))
        # the reference arm: rank 0 times the oracle and prints one line, the others print nothing
        buf = io.StringIO()
        args = types.SimpleNamespace(steps=1, warmup=0)
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args, wl, w, r)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"world": w, "rank": r, "local": local, "ms": ms, "rate": rate,
                       "q0": float(q.reshape(-1)[0]), "printed": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_timing_and_reference_arm(tmp_path):
    import oracle
    oracle.build()   # compiled once here, not concurrently by the two ranks
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert (x["world"], x["rank"], x["local"]) == (world, r, r)
        assert x["ms"] == 1.5                              # the max over ranks, on every rank
        assert x["rate"] == pytest.approx(world * 1000 / 1.5e-3)
    assert res[0]["q0"] != res[1]["q0"]                    # independent replicas
    line = json.loads(res[0]["printed"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert res[1]["printed"] == ""


def test_one_rank_helpers():
    import bench
    from gaussian_mixture_sequence_gb300 import workloads
    assert bench.max_over_ranks(None, 2.5, None) == 2.5
    assert bench.whole_job_rate(1, 500, 2.0) == pytest.approx(250000.0)
    wl = workloads.WORKLOADS["tiny"]
    assert bench.replica_seed(wl, 0) == wl.seed and bench.replica_seed(wl, 3) == wl.seed + 3
    a = workloads.full_inputs(wl.with_(N=8), bench.replica_seed(wl, 0))[2]
    b = workloads.full_inputs(wl.with_(N=8), bench.replica_seed(wl, 1))[2]
    assert not np.array_equal(a, b)
