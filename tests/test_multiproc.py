"""The N > 1 path on CPU: two gloo ranks.

The BitDelta linear partitions along output rows with no exchange (per-row
alpha lives with its rows).  Each rank computes its row block of y with the
oracle and an all_gather along rows must reproduce the unsharded result
exactly.  The benchmark's multi-GPU timing reduction (slowest rank wins) is
checked the same way.  A per-matrix alpha under row sharding is the one
exchange (``shard.per_matrix_alpha_allreduce``): it must match the unsharded
alpha within the 1e-6 relative bound, and a rank that never reaches it must
turn into BD_ERR_TIMEOUT on the others, not a hang (gloo; under NCCL the
watchdog handles a timed-out collective instead).
"""
import os
import socket
import time
from datetime import timedelta

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


def _alpha_rank(rank, world, port, q, d_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from bit_weight_delta_bd_gb300 import shard, synth

        oracle.set_threads(1)
        d_in = 256
        wb, wf, _ = synth.single_problem(7, d_out, d_in, 1)
        r0, r1 = shard.row_bounds(d_out, world, rank)
        if r1 > r0:
            _, a = oracle.compress(wb[r0:r1], wf[r0:r1], per_row=False)
        else:  # no rows: the compression writes no alpha, so the buffer holds whatever it held
            a = np.array([np.nan], np.float32)
        alpha = shard.per_matrix_alpha_allreduce(torch.from_numpy(a), r1 - r0, d_out)
        _, a_all = oracle.compress(wb, wf, per_row=False)
        q.put((rank, float(alpha.item()), float(a_all[0]), r1 - r0))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
@pytest.mark.parametrize("world,d_out", [(2, 70), (3, 70), (3, 2)])
def test_per_matrix_alpha_under_row_sharding(world, d_out):
    """d_out = 2 over 3 ranks leaves one rank without rows; its NaN alpha
    buffer must not reach the others."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_alpha_rank, args=(r, world, port, q, d_out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sum(r[3] for r in res) == d_out
    assert all(np.isfinite(r[1]) for r in res)
    alphas = {r[1] for r in res}
    assert len(alphas) == 1  # every rank holds the same alpha
    got, ref = alphas.pop(), res[0][2]
    assert abs(got - ref) <= 1e-6 * ref


def _silent_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=3))
    try:
        if rank == 1:  # never reaches the all-reduce
            time.sleep(12)
            q.put((rank, "slept", 0.0))
            return
        from bit_weight_delta_bd_gb300 import bitdelta as bd
        from bit_weight_delta_bd_gb300 import shard

        t0 = time.time()
        try:
            shard.per_matrix_alpha_allreduce(torch.ones(1), 5, 10)
            q.put((rank, "returned", time.time() - t0))
        except bd.BitDeltaError as e:
            q.put((rank, f"error {e.status}", time.time() - t0))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001 -- the group may already be unusable after the timeout
            pass


@pytest.mark.timeout(300)
def test_alpha_allreduce_rank_that_never_arrives_times_out():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_silent_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res[0][1] == "error 7"  # BD_ERR_TIMEOUT, after about the group's 3 s timeout
    assert res[0][2] < 11.0
    assert res[1][1] == "slept"


def test_row_bounds_partition():
    from bit_weight_delta_bd_gb300 import shard

    for d_out in (0, 1, 7, 70, 28672):
        for world in (1, 2, 3, 8):
            spans = [shard.row_bounds(d_out, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == d_out
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.row_bounds(10, 2, 2)


def _gather_rank(rank, world, port, q, d_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        T = 3
        y_full = torch.arange(T * d_out, dtype=torch.float32).reshape(T, d_out)
        r0, r1 = bench.row_span(d_out, world, rank)
        y = bench.gather_rows(y_full[:, r0:r1].contiguous(), d_out, world, rank)
        q.put((rank, bool(torch.equal(y, y_full))))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
@pytest.mark.parametrize("world,d_out", [(2, 8), (3, 7), (3, 2)])
def test_benchmark_row_gather_reassembles_y(world, d_out):
    """The benchmark's exchange step under the output-row partition: each
    rank's y columns, gathered (shards padded to equal size), give the full y
    on every rank, also for ragged and empty shards."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_rank, args=(r, world, port, q, d_out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [True] * world
