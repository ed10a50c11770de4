"""The multi-rank path on CPU: two gloo ranks aggregate work and time the way
bench.py reports a job (sum of work, max of time); replica inputs differ."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from random_feature_gb300.replicas import job_aggregate, replica_seed


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units, ms = job_aggregate(units=1000 * (rank + 1), ms=10.0 + 5 * rank)
        out[rank] = (units, ms)
    finally:
        dist.destroy_process_group()


def test_job_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (3000.0, 15.0)


def test_job_aggregate_single_process():
    assert job_aggregate(12.0, 3.5) == (12.0, 3.5)


def test_replica_inputs_differ_per_rank():
    from synth import CONFIGS, make_workload
    w = CONFIGS["tiny_f32"]
    a = make_workload(w, replica_seed(0, 0))[1]
    b = make_workload(w, replica_seed(0, 1))[1]
    assert replica_seed(0, 0) != replica_seed(0, 1)
    assert not np.array_equal(a, b)
