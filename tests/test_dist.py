"""The multi-process path of the benchmark on CPU: two gloo ranks.  Each rank
draws its own batch (weak scaling) and the step time is the maximum over
ranks; nothing else crosses ranks."""
import os
import socket

import torch
import torch.distributed as td
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import kda_inputs
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench._dist()
        mx = bench.max_over_ranks([1.0 + r, 10.0 - r], "cpu")
        x = kda_inputs.fixed(1, 8, 2, 64, seed=bench.rank_seed(r))
        q.put((r, w, mx, float(x.v.float().sum())))
        td.barrier()
    finally:
        td.destroy_process_group()


def test_two_rank_timing_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, mx0, s0), (r1, w1, mx1, s1) = out
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert mx0 == mx1 == [2.0, 10.0]      # slowest rank's time, seen by every rank
    assert s0 != s1                       # each rank draws its own batch
    assert bench_seed_is_workload_seed()


def bench_seed_is_workload_seed():
    import bench
    return bench.rank_seed(0) == 1001
