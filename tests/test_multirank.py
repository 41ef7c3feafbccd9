"""The benchmark's multi-rank host path on CPU: two gloo ranks on 127.0.0.1.

Sequences are independent, so N GPUs run N replicas with no data-path
collective: each rank decodes its own sequences (same shapes, another seed),
the job's time is the slowest rank's (a max all-reduce) and the whole-job
rate counts every rank's steps.  Nothing here needs a GPU.
"""
import json
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.rank_workload(synth.WORKLOADS["batched"], rank, world)
    mine = {"seed": w.seed, "shape": [w.B, w.V, w.K, w.N, w.Hq, w.Hkv, w.d],
            "prefix": [int(x) for x in w.prefix_lengths()],
            "root": [int(x) for x in synth.initial_roots(w)]}
    every = [None] * world
    dist.all_gather_object(every, mine)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")   # rank r took 10 + 5r ms
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"every": every, "slowest": slowest}, f)


def test_two_gloo_ranks_replicas(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(os.path.join(tmp_path, "rank%d.json" % r))) for r in range(world)]
    every = res[0]["every"]
    assert res[1]["every"] == every
    # same shapes, different sequences on each rank
    assert every[0]["shape"] == every[1]["shape"]
    assert every[0]["seed"] != every[1]["seed"]
    assert every[0]["prefix"] != every[1]["prefix"] or every[0]["root"] != every[1]["root"]
    # the job's time is the slowest rank's, on every rank
    assert res[0]["slowest"] == res[1]["slowest"] == 15.0
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 16 steps of their own batches in 15 ms
    assert np.isclose(bench.job_rate(world, 16, 15.0), 2 * 16 / 0.015)
    assert np.isclose(bench.job_rate(1, 16, 15.0), 16 / 0.015)
