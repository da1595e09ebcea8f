"""The N > 1 path on CPU: two gloo ranks.

The BitDelta linear partitions along output rows with no exchange (per-row
alpha lives with its rows).  Each rank computes its row block of y with the
oracle and an all_gather along rows must reproduce the unsharded result
exactly.  The benchmark's multi-GPU timing reduction (slowest rank wins) is
checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from bit_weight_delta_bd_gb300 import synth

        oracle.set_threads(1)
        d_out, d_in, T = 70, 256, 5
        wb, wf, x = synth.single_problem(123, d_out, d_in, T)
        bounds = np.linspace(0, d_out, world + 1).astype(int)
        r0, r1 = bounds[rank], bounds[rank + 1]
        s, a = oracle.compress(wb[r0:r1], wf[r0:r1], per_row=True)
        y_part = oracle.linear(x, wb[r0:r1], s, a, per_row=True)
        parts = [None] * world
        dist.all_gather_object(parts, y_part)
        y = np.concatenate(parts, axis=1)
        s_all, a_all = oracle.compress(wb, wf, per_row=True)
        ok_shard = bool(np.array_equal(y, oracle.linear(x, wb, s_all, a_all, per_row=True)))
        t = torch.tensor([10.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        q.put((rank, ok_shard, float(t.item())))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_row_sharding_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [True, True]
    assert [r[2] for r in res] == [11.0, 11.0]
