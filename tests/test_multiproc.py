"""The N > 1 host logic of bench.py on CPU with gloo, world size 2: each rank
runs its own seeded replica (no data exchange), timings are max-reduced and
the reported rate is the aggregate over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import numpy as np
    import torch.distributed as dist

    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = bench.replica_spec("tiny_ragged_fp32", rank, world)
    x = spec.build()
    out = oracle.sparse_attention(x)
    fake_ms = 10.0 * (rank + 1)  # rank 1 is the slower one
    ms = bench.max_over_ranks(fake_ms, world)
    q.put((rank, spec.seed, float(np.abs(out).sum()), ms, bench.aggregate_rate(x.total_q, world, ms)))
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_timing():
    import oracle

    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, a0, ms0, v0), (r1, s1, a1, ms1, v1) = res
    assert s0 != s1 and a0 != a1          # independent replicas
    assert ms0 == ms1 == 20.0             # both see the slowest rank
    assert v0 == v1 == pytest.approx(2 * 8 / 0.020)  # 2 ranks x 8 rows / 20 ms
