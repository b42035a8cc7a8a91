"""The multi-GPU path of bench.py, on CPU with two gloo ranks.

The path has no data exchange: every rank runs a full replica of the workload
(weak scaling) and only the timing is reduced -- the job takes as long as the
slowest rank, and throughput counts every rank's units.  Here each rank runs a
small replica through the CPU oracle (standing in for its GPU), with a
different amount of simulated time, and both ranks must agree on the result."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth_inputs as SI


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = SI.gqa_prompt(40, seed=7 + rank, hq=4, hkv=2, dim=16)
        out, _, sizes = oracle.chunked_prefill(q.double().numpy(), k.double().numpy(), v.double().numpy(), 16)
        ok = np.isfinite(out).all() and sizes == [16, 16, 8]
        local_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
        total_ms, value = bench.job_throughput(local_ms, 40, 5, world)
        dist.barrier()
        out_q.put((rank, bool(ok), total_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok, total_ms, value in res:
        assert ok
        assert total_ms == 20.0                      # the slowest rank's time
        assert abs(value - 2 * 40 * 5 / 0.020) < 1e-6  # units of both ranks / that time
