"""Partition of one batch across ranks (one process per GPU), with no exchange.

Every (sequence, head) chain of the KDA forward is independent: the state
resets at each packed-sequence boundary ("Kimi K3 NPU Training", section 定长与
TND) and each head keeps its own state.  A batch therefore splits across GPUs
with no collective on the data path, in either of two ways:

* by sequence -- longest-processing-time first (LPT): sequences in order of
  decreasing length, each to the rank with the least work so far, work being
  the 64-token chunks it will run (its chains' serial length);
* by head -- contiguous head ranges, the tensor-parallel split of the attention
  layer ("Kimi K3 NPU Training", section 模型与并行改造, TP row: KDA sharded by
  head).

Each rank then calls the forward on its own shard; its outputs are its own
sequences' (or heads') rows.  The helpers here only decide the assignment and
slice tensors; every step of the computation stays in the CUDA kernels.
"""
from __future__ import annotations

import dataclasses

import torch

CHUNK = 64


def chunk_work(length: int) -> int:
    """Serial work of one sequence's chains: its 64-token chunks."""
    return (int(length) + CHUNK - 1) // CHUNK


def lpt_by_sequence(lengths, world: int):
    """Per-rank lists of sequence indices (each list ascending).

    Sequences go in order of decreasing work (ties: lower index first), each to
    the rank with the least work assigned so far (ties: lower rank).  Every
    sequence, an empty one included, is assigned to exactly one rank, so its
    final state is written exactly once.  Greedy list scheduling bounds the
    largest rank's work by total / world + the largest sequence's work.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    lengths = [int(x) for x in lengths]
    order = sorted(range(len(lengths)), key=lambda i: (-chunk_work(lengths[i]), i))
    load = [0] * world
    ranks = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda j: (load[j], j))
        ranks[r].append(i)
        load[r] += chunk_work(lengths[i])
    return [sorted(r) for r in ranks]


def heads_by_rank(H: int, world: int):
    """Contiguous head ranges ``(h0, h1)`` per rank, sizes differing by at most one."""
    if world < 1:
        raise ValueError("world must be >= 1")
    base, extra = divmod(int(H), world)
    out, h = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((h, h + n))
        h += n
    return out


def _lengths(cu):
    cu = [int(x) for x in cu]
    return [b - a for a, b in zip(cu[:-1], cu[1:])]


@dataclasses.dataclass
class Shard:
    """A rank's part of a batch: its inputs and where its rows sit in the whole."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor | None
    h0: torch.Tensor | None
    seqs: list          # sequence indices of the whole batch, in shard order
    heads: tuple        # (h0, h1) head range of the whole batch


def take_sequences(x, idx) -> Shard:
    """The packed sub-batch of sequences ``idx`` (in that order) of the packed
    batch ``x`` (``[1, T, H, d]`` with ``cu_seqlens``): token rows gathered, the
    offsets rebased, start states ``h0[idx]``."""
    cu = x.cu_seqlens.detach().cpu().tolist()
    lens = _lengths(cu)
    dev = x.q.device
    rows = [torch.arange(cu[i], cu[i + 1], dtype=torch.int64) for i in idx]
    rows = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.int64)
    rows = rows.to(dev)
    sel = lambda t: t.index_select(1, rows).contiguous()
    new_cu = [0]
    for i in idx:
        new_cu.append(new_cu[-1] + lens[i])
    h0 = None
    if x.h0 is not None:
        h0 = x.h0.index_select(0, torch.as_tensor(list(idx), dtype=torch.int64,
                                                  device=x.h0.device)).contiguous()
    H = x.q.shape[2]
    return Shard(sel(x.q), sel(x.k), sel(x.v), sel(x.g), sel(x.beta),
                 torch.tensor(new_cu, dtype=torch.int32, device=dev), h0, list(idx), (0, H))


def take_heads(x, h0: int, h1: int) -> Shard:
    """Heads ``[h0, h1)`` of every sequence of ``x`` (fixed-length or packed)."""
    sl = lambda t: t[:, :, h0:h1].contiguous()
    st = None if x.h0 is None else x.h0[:, h0:h1].contiguous()
    n = x.q.shape[0] if x.cu_seqlens is None else x.cu_seqlens.numel() - 1
    return Shard(sl(x.q), sl(x.k), sl(x.v), sl(x.g), x.beta[:, :, h0:h1].contiguous(),
                 x.cu_seqlens, st, list(range(n)), (h0, h1))


def place_sequences(total_tokens: int, cu, shards, outs, states):
    """Reassemble per-rank results of a sequence partition: ``outs[r]`` the
    ``[1, T_r, H, dv]`` output and ``states[r]`` the ``[N_r, H, dk, dv]`` final
    states of ``shards[r]``.  Returns the whole batch's ``(o, hT)``."""
    cu = [int(x) for x in cu]
    o = None
    hT = None
    for sh, o_r, h_r in zip(shards, outs, states):
        if o is None:
            o = o_r.new_zeros((1, total_tokens) + tuple(o_r.shape[2:]))
            hT = h_r.new_zeros((len(cu) - 1,) + tuple(h_r.shape[1:]))
        at = 0
        for j, i in enumerate(sh.seqs):
            n = cu[i + 1] - cu[i]
            o[:, cu[i]:cu[i + 1]] = o_r[:, at:at + n]
            hT[i] = h_r[j]
            at += n
    return o, hT
