"""The multi-process paths on CPU, as two gloo ranks:

* the benchmark's replicas: each rank draws its own batch (weak scaling) and the
  step time is the maximum over ranks;
* the partition of one batch across ranks (by sequence, longest first, or by
  head), each rank computing only its own chains with the float64 oracle; the
  gathered results must equal the unsharded run.  Nothing but the results'
  check crosses ranks."""
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


# partition of one batch across ranks ------------------------------------------------

def _shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import kda_inputs
    import oracle
    from kda_delta_rule_fwd_gb300 import shard
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lens = [300, 0, 65, 1, 200, 64, 130, 7, 520]
        x = kda_inputs.packed(lens, 3, 64, dtype=torch.bfloat16, seed=78, h0_std=0.1)
        run = lambda s: oracle.recurrent(s.q, s.k, s.v, s.g, s.beta, cu_seqlens=s.cu_seqlens,
                                         h0=s.h0, n_threads=1)
        # by sequence (LPT): this rank's sequences only
        parts = shard.lpt_by_sequence(lens, world)
        mine = shard.take_sequences(x, parts[rank])
        o, h = run(mine)
        by_seq = [None] * world
        td.all_gather_object(by_seq, (mine.seqs, o, h))
        # by head: this rank's head range of every sequence
        h0, h1 = shard.heads_by_rank(3, world)[rank]
        o2, hh2 = run(shard.take_heads(x, h0, h1))
        by_head = [None] * world
        td.all_gather_object(by_head, ((h0, h1), o2, hh2))
        if rank == 0:
            q.put((lens, parts, by_seq, by_head))
        td.barrier()
    finally:
        td.destroy_process_group()


def test_two_rank_partition_of_one_batch():
    """One packed batch split across two gloo ranks, by sequence (LPT) and by head:
    every (sequence, head) chain is computed by exactly one rank, the larger rank's
    work is within the greedy bound, and the ranks' outputs put back in place equal
    the unsharded run exactly (chains are independent; no exchange is needed)."""
    import numpy as np
    import oracle
    import kda_inputs
    from kda_delta_rule_fwd_gb300 import shard
    oracle.build()
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    lens, parts, by_seq, by_head = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every sequence exactly once; work balanced within the list-scheduling bound
    assert sorted(i for r in parts for i in r) == list(range(len(lens)))
    work = [sum(shard.chunk_work(lens[i]) for i in r) for r in parts]
    total, biggest = sum(work), max(shard.chunk_work(n) for n in lens)
    assert max(work) <= total / world + biggest
    # reassembled outputs equal the whole batch's
    x = kda_inputs.packed(lens, 3, 64, dtype=torch.bfloat16, seed=78, h0_std=0.1)
    o_ref, h_ref = oracle.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                    h0=x.h0, n_threads=1)
    cu = x.cu_seqlens.tolist()
    o = np.zeros_like(o_ref)
    h = np.zeros_like(h_ref)
    for seqs, o_r, h_r in by_seq:
        at = 0
        for j, i in enumerate(seqs):
            n = cu[i + 1] - cu[i]
            o[:, cu[i]:cu[i + 1]] = o_r[:, at:at + n]
            h[i] = h_r[j]
            at += n
    assert np.array_equal(o, o_ref) and np.array_equal(h, h_ref)
    o = np.zeros_like(o_ref)
    h = np.zeros_like(h_ref)
    covered = []
    for (h0, h1), o_r, h_r in by_head:
        o[:, :, h0:h1] = o_r
        h[:, h0:h1] = h_r
        covered += list(range(h0, h1))
    assert sorted(covered) == [0, 1, 2]
    assert np.array_equal(o, o_ref) and np.array_equal(h, h_ref)


def test_partition_helpers():
    from kda_delta_rule_fwd_gb300 import shard
    assert shard.heads_by_rank(32, 3) == [(0, 11), (11, 22), (22, 32)]
    assert shard.heads_by_rank(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    lens = [8192, 128, 4000, 4000, 0, 64, 8000]
    parts = shard.lpt_by_sequence(lens, 3)
    assert sorted(sum(parts, [])) == list(range(len(lens)))
    assert parts[0] == [0]  # the longest sequence alone, first
    assert shard.lpt_by_sequence(lens, 1) == [list(range(len(lens)))]
    # more ranks than sequences: the extra ranks get nothing
    assert shard.lpt_by_sequence([5, 6], 4)[2:] == [[], []]
