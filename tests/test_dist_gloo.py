"""The multi-rank host path of the benchmark on CPU (gloo, world size 2).

The decode path shards by sequence with no exchange, so N GPUs run N
independent replicas; the only cross-rank steps are the barrier around the
timed region and the MAX reduction of the elapsed time.  Two gloo ranks run
those steps here, each also advancing its own replica of a small workload
with the oracle (seeded by rank), and the job value is checked.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    import oracle as orc
    from recurrent_state_gb300 import inputs as gen

    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        # each rank: its own replica (seed = rank), no data crosses ranks
        w = gen.decode_workload(B=2, Hk=1, Hv=2, d=16, steps=2, per_channel=False,
                                in_dtype="f32", seed=rank)
        pool = w.state0.copy()
        for t in range(w.steps):
            orc.decode_f32(pool, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        bench._barrier(world)
        dt = 0.25 * (rank + 1)                     # rank 1 is the slowest
        dt_max = bench._max_over_ranks(dt, world)
        value = bench.job_value(world, 10, w.B * w.Hv, dt_max)
        out.put((rank, dt_max, value, float(np.abs(pool).sum())))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, v0, s0), (r1, m1, v1, s1) = res
    assert m0 == m1 == 0.5                         # MAX over ranks
    assert v0 == v1 == pytest.approx(2 * 10 * 4 / 0.5)
    assert s0 != s1                                # independent replicas
