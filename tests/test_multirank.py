"""The N > 1 bench path on CPU: two gloo ranks (world size 2).

The path has no exchange step, so `bench.py --gpus N` runs N independent
replicas; what the ranks share is host logic -- each rank's own workload
seed, the job time as the slowest rank's (max over ranks), the job
throughput as every rank's samples over that time, and a reference arm that
only rank 0 runs.  These run here with the gloo backend, no GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.env_rank()
        t_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(t_ms, dist, "cpu")
        value = bench.job_throughput(7, w, job_ms)
        p = workloads.minibatch_priorities(seed=bench.rank_seed(r))
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), r, w) if r != 0 else None
        q.put((r, w, lr, job_ms, value, float(p[:8].sum()), ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_host_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, t0, v0, s0, ref0), (r1, w1, l1, t1, v1, s1, ref1) = out
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    # the job time is the slowest rank's, on every rank
    assert t0 == t1 == 15.0
    # whole-job throughput: both ranks' samples over that time
    want = 7 * bench.ROUNDS * bench.B * 2 / 15.0e-3
    assert v0 == v1 == pytest.approx(want, rel=1e-12)
    # each replica draws its own buffer
    assert s0 != s1
    # the reference arm does no work off rank 0
    assert ref1 is None


def test_single_process_helpers_without_a_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2, 1, 1000.0) == 2 * bench.ROUNDS * bench.B
    assert bench.rank_seed(0) == workloads.MINIBATCH["seed"]
    a = workloads.minibatch_priorities(seed=bench.rank_seed(0))
    b = workloads.minibatch_priorities(seed=bench.rank_seed(0))
    assert np.array_equal(a, b)
