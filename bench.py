"""Benchmark of the KDA forward on GB300.

Default workload (one "step" = one kda_fwd call over the whole batch):
    fixed-length prefill, B=4, T=4096, H=32, dk=dv=128, bf16 q/k/v/g/beta,
    float32 state and output, chunk 64, h0 = 0.
Timed in the same run and reported in sub-objects: the decode pool (1024
sequences, H=32, d=128, float32 states resident in HBM; T_step = 1 and an
8-token replay step) under "decode", the packed 16-sequence prefill under
"prefill_packed", the 1,048,576-token prefill (B=1, H=32) under "prefill_long",
a packed batch holding one 2^18-token sequence under "prefill_packed_long", and
the rows beyond the hot path under "next_rows".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --case NAME     (one kernel's workload, for an ncu capture)

Prints one JSON line.  Under torchrun every rank runs its own batch of the
headline workload (weak scaling, no data-path collective); the packed batch is
also partitioned across the ranks by sequence, longest first, and timed as one
job ("prefill_packed_sharded").  The barrier and the max over ranks of the
timed regions are the only communication.  ``--impl reference`` times the
float64 CPU oracle on the host's cores on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, T, H, D = 4, 4096, 32, 128
CHUNK = 64
# algorithmic work per token per head (chunk 64, d = 128): dense 64x64 tiles
FLOP_PER_TOKEN_HEAD = 10 * CHUNK * D + 6 * D * D          # 180,224
# minimum HBM bytes per token per head: q, k, v, g bf16 + beta bf16 + o float32
BYTES_PER_TOKEN_HEAD = 4 * D * 2 + 2 + D * 4               # 1,538
STATE_BYTES = D * D * 4                                    # one head's float32 state
# backward: q, k, v, g bf16 + beta bf16 + dout fp32 in; dq, dk, dv, dg, dbeta fp32 out
BWD_BYTES_PER_TOKEN_HEAD = 4 * D * 2 + 2 + D * 4 + 4 * D * 4 + 4   # 3,590
WORKLOAD = "KDA prefill, fixed length: B=4, T=4096, H=32, dk=dv=128, bf16 in, fp32 state/out, chunk 64"
METRIC = "KDA fwd tokens/s at H=32,d=128 (prefill+decode); % of tensor/HBM roofline"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def profiled_traffic():
    """DRAM bytes per prefill launch from the committed ncu summary, or None when
    the kernel source (with its headers) has changed since those counters were taken."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "kda_delta_rule_fwd_gb300", "csrc")
    srcs = [os.path.join(csrc, f) for f in ("kda_prefill_bf16.cu", "kda_prefill_common.cuh",
                                            "kda_internal.cuh", "kda_mma_sync.cuh",
                                            "kda_sm100.cuh")]
    prof = os.path.join(ROOT, "profiles", "prefill_bf16_B4_T4096_H32.txt")
    try:
        txt = open(prof).read()
        h = hashlib.sha256()
        for f in srcs:  # the kernel's source and the headers it includes
            h.update(open(f, "rb").read())
        digest = h.hexdigest()[:16]
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256_16: (\w+)", txt)
    b = re.search(r"dram_bytes_per_launch: (\d+)", txt)
    if m and b and m.group(1) == digest:
        return int(b.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"kda_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for name, val in zip(names, r[5:9]):
                    if val.strip() == "Active":
                        reasons.add(name)
            except (ValueError, IndexError):
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(rank):
    """Seed of a rank's batch: rank 0 runs the workload's own seed, every other
    rank an independent batch of the same shape (weak scaling: per-rank work is
    fixed, no data crosses ranks)."""
    return 1001 + 97 * rank


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the step
    time).  The only collective the benchmark makes besides its barriers."""
    import torch
    import torch.distributed as td
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if td.is_available() and td.is_initialized() and td.get_world_size() > 1:
        td.all_reduce(t, op=td.ReduceOp.MAX)
    return t.tolist()


def _cpu_baseline(x, budget_s=20.0):
    """The float64 oracle on the host's cores: whole sequences of the first few
    heads, as many heads as fit the time budget (estimated from one head)."""
    import numpy as np
    import torch
    import oracle
    cores = oracle.max_threads()
    # sample: batch element 0, one head, first 1024 tokens -> per-token-head rate
    t0 = time.perf_counter()
    sl = lambda a: a[:1, :1024, :1].contiguous()
    oracle.recurrent(sl(x.q), sl(x.k), sl(x.v), sl(x.g), x.beta[:1, :1024, :1].contiguous(),
                     n_threads=1)
    rate1 = 1024 / (time.perf_counter() - t0)          # token-heads/s on one core
    heads = max(1, min(H, int(budget_s * rate1 * cores / (B * T))))
    sub = lambda a: a[:, :, :heads].contiguous()
    args = (sub(x.q), sub(x.k), sub(x.v), sub(x.g), x.beta[:, :, :heads].contiguous())
    # whole passes over the sample until at least half the budget has elapsed (the
    # oracle may finish all heads well inside it), at most 30
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.recurrent(*args, n_threads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= 0.5 * budget_s or passes >= 30:
            break
    head_tokens_per_s = passes * B * T * heads / dt
    return {"value": head_tokens_per_s / H, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"B={B}, T={T}, {heads} of {H} heads, all tokens, {passes} passes "
                      f"({dt:.1f} s); tokens/s = head-tokens/s / H"}


def _time_steps(fn, steps, warmup, stream, dist_on):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist_on:
        import torch.distributed as td
        td.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist_on:
        td.barrier()
    return e0.elapsed_time(e1) / steps


def _hbm_line(nbytes, ms, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak}


E2E_SEQ_PARTS = 4   # the headline batch's sequences, each its own stream of kernels
E2E_TIME_PARTS = 2  # each sequence cut in time (the later part starts from the earlier's hT)


def make_e2e_step(kda, x, dev, seq_parts=E2E_SEQ_PARTS, time_parts=E2E_TIME_PARTS):
    """One end-to-end step through the public API with HOST buffers: pinned host
    inputs in, o and hT back to pinned host memory.  The batch is cut by sequence
    into `seq_parts` and in time into `time_parts` contiguous pieces.  Every piece's
    inputs go down in turn on one copy stream; each sequence's pieces run kda_fwd in
    order on a stream of their own, a piece starting from the previous piece's final
    state (h0 = its hT; chunk boundaries stay at multiples of 64, so the results are
    those of one call), as soon as its inputs have landed; its o (and the last
    piece's hT) come back on a third stream.  The copies overlap the kernels and
    each other (the two directions of the link are independent).
    Returns (step, h2d_bytes, d2h_bytes, buffers)."""
    import torch
    pin = lambda t: t.cpu().pin_memory()
    hin = [pin(t) for t in (x.q, x.k, x.v, x.g, x.beta)]
    din = [torch.empty_like(t) for t in (x.q, x.k, x.v, x.g, x.beta)]
    o = torch.empty(B, T, H, D, device=dev)
    hT = torch.empty(B, H, D, D, device=dev)
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hh = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
    per, tl = B // seq_parts, T // time_parts
    mid = [[torch.empty(per, H, D, D, device=dev) for _ in range(time_parts - 1)]
           for _ in range(seq_parts)]
    shape = kda.make_shape(x.q[:per, :tl], x.v[:per, :tl])
    wss = [kda.new_workspace(shape, dev) for _ in range(seq_parts)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s_run = [torch.cuda.Stream(device=dev) for _ in range(seq_parts)]

    def step():
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(seq_parts):
            bs = slice(i * per, (i + 1) * per)
            for j in range(time_parts):
                ts = slice(j * tl, (j + 1) * tl)
                last = j == time_parts - 1
                landed, done = torch.cuda.Event(), torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    for d_, h_ in zip(din, hin):
                        d_[bs, ts].copy_(h_[bs, ts], non_blocking=True)
                    landed.record(s_in)
                s_run[i].wait_event(landed)
                with torch.cuda.stream(s_run[i]):
                    kda.fwd(*(d_[bs, ts] for d_ in din), h0=mid[i][j - 1] if j else None,
                            out=o[bs, ts], hT=hT[bs] if last else mid[i][j], workspace=wss[i])
                    done.record(s_run[i])
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    ho[bs, ts].copy_(o[bs, ts], non_blocking=True)
                    if last:
                        hh[bs].copy_(hT[bs], non_blocking=True)
        cur.wait_stream(s_out)

    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = ho.numel() * ho.element_size() + hh.numel() * hh.element_size()
    return step, h2d, d2h, (o, hT, ho, hh, mid)


def bench_long(kda, args, dev, stream, dist_on, hbm_peak):
    """The 1,048,576-token prefill (B=1, H=32): one step is the whole call (the
    long-chain split's transition, scan and output passes included)."""
    import torch
    import kda_inputs
    x = kda_inputs.workload(3, device=dev)
    shape = kda.make_shape(x.q, x.v)
    ws = kda.new_workspace(shape, dev)
    o = torch.empty_like(x.v, dtype=torch.float32)
    hT = torch.empty(1, H, D, D, device=dev)
    fn = lambda: kda.fwd(x.q, x.k, x.v, x.g, x.beta, out=o, hT=hT, workspace=ws)
    ms = _time_steps(fn, max(3, args.steps // 4), 2, stream, dist_on)
    st = kda.read_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.status_string(st)}")
    tok = x.q.shape[1]
    nbytes = tok * H * BYTES_PER_TOKEN_HEAD + H * STATE_BYTES
    del x, o, hT, ws
    torch.cuda.empty_cache()
    ms = max_over_ranks([ms], dev)[0]
    return {
        "workload": "KDA prefill, long context: B=1, T=1,048,576, H=32, dk=dv=128, bf16 in, "
                    "fp32 state/out, chunk 64, h0 = 0",
        "tokens": tok, "ms_per_step": ms, "tokens_per_s": tok * _dist()[1] / (ms * 1e-3),
        "workspace_bytes": int(kda.workspace_size(shape)),
        "roofline": _hbm_line(nbytes, ms, hbm_peak),
    }


def bench_packed_long(kda, args, dev, stream, dist_on, hbm_peak):
    """A packed batch holding one long sequence, [2^18, 300, 1, 5000] tokens at H=32
    (the device-planned split cuts the long sequence into segments), beside the
    fixed-length B=1, T=2^18 batch of that length alone (the host-planned split)."""
    import torch
    import kda_inputs
    lens = [1 << 18, 300, 1, 5000]
    out = {}
    for name, x in (("packed", lambda: kda_inputs.packed(lens, H, D, device=dev, seed=1006,
                                                        h0_std=0.1)),
                    ("fixed", lambda: kda_inputs.fixed(1, 1 << 18, H, D, device=dev,
                                                      seed=1006))):
        x = x()
        n = 4 if name == "packed" else 1
        shape = kda.make_shape(x.q, x.v, packed_seqs=n if name == "packed" else None)
        ws = kda.new_workspace(shape, dev)
        o = torch.empty_like(x.v, dtype=torch.float32)
        hT = torch.empty(n, H, D, D, device=dev)
        fn = lambda: kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                             out=o, hT=hT, workspace=ws)
        ms = _time_steps(fn, max(3, args.steps // 4), 3, stream, dist_on)
        st = kda.read_device_status(ws)
        if st != kda.KDA_OK:
            raise RuntimeError(f"device status {kda.status_string(st)}")
        tok = x.q.shape[1]
        nbytes = tok * H * BYTES_PER_TOKEN_HEAD + n * H * 2 * STATE_BYTES
        ms = max_over_ranks([ms], dev)[0]
        out[name] = {"tokens": tok, "ms_per_step": ms, "tokens_per_s": tok / (ms * 1e-3),
                     "roofline": _hbm_line(nbytes, ms, hbm_peak)}
        del x, o, hT, ws
        torch.cuda.empty_cache()
    out["workload"] = ("packed [2^18, 300, 1, 5000] tokens, H=32, d=128, bf16, h0; against "
                       "fixed-length B=1, T=2^18, H=32")
    out["time_per_token_packed_over_fixed"] = (
        out["packed"]["ms_per_step"] / out["packed"]["tokens"]) / (
        out["fixed"]["ms_per_step"] / out["fixed"]["tokens"])
    return out


def bench_packed_sharded(kda, args, dev, stream, dist_on, hbm_peak):
    """The packed 16-sequence batch partitioned across the ranks by sequence,
    longest first: each rank runs only its own sequences; the job's time is the
    slowest rank's and its tokens are the whole batch's (one batch, strong
    scaling)."""
    import torch
    import kda_inputs
    from kda_delta_rule_fwd_gb300 import shard
    rank, world, _ = _dist()
    y = kda_inputs.workload(2, device=dev)
    lens = (y.cu_seqlens[1:] - y.cu_seqlens[:-1]).tolist()
    mine = shard.take_sequences(y, shard.lpt_by_sequence(lens, world)[rank])
    n = len(mine.seqs)
    if n:
        ws = kda.new_workspace(kda.make_shape(mine.q, mine.v, packed_seqs=n), dev)
        o = torch.empty_like(mine.v, dtype=torch.float32)
        hT = torch.empty(n, H, D, D, device=dev)
        fn = lambda: kda.fwd(mine.q, mine.k, mine.v, mine.g, mine.beta,
                             cu_seqlens=mine.cu_seqlens, h0=mine.h0, out=o, hT=hT, workspace=ws)
    else:
        fn = lambda: None
    ms = _time_steps(fn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    ms = max_over_ranks([ms], dev)[0]
    tok = y.q.shape[1]
    nbytes = tok * H * BYTES_PER_TOKEN_HEAD + len(lens) * H * 2 * STATE_BYTES
    return {"workload": "16 packed sequences (as prefill_packed) split across the ranks by "
                        "sequence, longest first", "ranks": world, "tokens": tok,
            "ms_per_step": ms, "tokens_per_s": tok / (ms * 1e-3),
            "roofline_per_job": _hbm_line(nbytes, ms, hbm_peak * world)}


def run_ours(args):
    import torch
    import kda_inputs
    import kda_delta_rule_fwd_gb300 as kda

    rank, world, local = _dist()
    dist_on = world > 1
    if dist_on:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    hbm_peak, bf16_peak, peak_kind = _peaks()

    x = kda_inputs.workload(1, device=dev)
    if rank:  # each rank its own batch of the same shape
        x = kda_inputs.fixed(B, T, H, D, device=dev, seed=rank_seed(rank))
    shape = kda.make_shape(x.q, x.v)
    ws = kda.new_workspace(shape, dev)
    o = torch.empty(B, T, H, D, device=dev)
    hT = torch.empty(B, H, D, D, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        kda.fwd(x.q, x.k, x.v, x.g, x.beta, out=o, hT=hT, workspace=ws)

    clocks = ClockSampler(local)  # spans every timed region below
    clocks.start()
    ms = _time_steps(step, args.steps, args.warmup, stream, dist_on)
    st = kda.read_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.status_string(st)}")

    # end to end through the public API with host buffers (pipelined by sequence)
    e2e_step, h2d, d2h, keep = make_e2e_step(kda, x, dev)
    ms_e2e = _time_steps(e2e_step, max(3, args.steps // 4), 2, stream, dist_on)
    # the same with one part: copies in, kernel, copies out in sequence
    e2e_serial, _, _, keep1 = make_e2e_step(kda, x, dev, seq_parts=1, time_parts=1)
    ms_e2e1 = _time_steps(e2e_serial, max(3, args.steps // 4), 2, stream, dist_on)
    del keep, keep1, e2e_step, e2e_serial

    # decode pool: T_step = 1 and 8, states resident in HBM (updated in place)
    dec = {}
    for T_step in (1, 8):
        y = kda_inputs.decode_pool(num_seqs=1024, H=H, d=D, T_step=T_step, device=dev,
                                   seed=1004 + 13 * rank)
        state = y.h0
        out_d = torch.empty(1024, T_step, H, D, device=dev)
        dshape = kda.make_shape(y.q, y.v)
        dws = kda.new_workspace(dshape, dev)
        fn = lambda: kda.decode(y.q, y.k, y.v, y.g, y.beta, state, out=out_d, workspace=dws)
        dms = _time_steps(fn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
        nbytes = 1024 * H * (2 * STATE_BYTES + T_step * BYTES_PER_TOKEN_HEAD)
        dec[f"T{T_step}"] = {"tokens_per_s": 1024 * T_step * world / (dms * 1e-3),
                             "ms_per_step": dms, "roofline": _hbm_line(nbytes, dms, hbm_peak)}
        dec[f"T{T_step}"]["roofline"]["traffic"] = None
        del y, state, out_d

    # packed prefill: 16 sequences of 128..8192 tokens with h0 (a second prefill workload)
    y = kda_inputs.workload(2, device=dev) if rank == 0 else kda_inputs.packed(
        kda_inputs.seq_lengths(16, 128, 8192, 1002), H, D, device=dev, seed=rank_seed(rank),
        h0_std=0.1)
    n_seq = y.cu_seqlens.numel() - 1
    py_o = torch.empty_like(y.v, dtype=torch.float32)
    py_h = torch.empty(n_seq, H, D, D, device=dev)
    pws = kda.new_workspace(kda.make_shape(y.q, y.v, packed_seqs=n_seq), dev)
    pfn = lambda: kda.fwd(y.q, y.k, y.v, y.g, y.beta, cu_seqlens=y.cu_seqlens, h0=y.h0,
                          out=py_o, hT=py_h, workspace=pws)
    pms = _time_steps(pfn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    ptok = y.q.shape[1]
    pbytes = ptok * H * BYTES_PER_TOKEN_HEAD + n_seq * H * 2 * STATE_BYTES
    pms = max_over_ranks([pms], dev)[0]
    packed_line = {
        "workload": "16 packed sequences, lengths uniform in [128, 8192], H=32, d=128, bf16, h0",
        "tokens": ptok, "ms_per_step": pms, "tokens_per_s": ptok * world / (pms * 1e-3),
        "roofline": _hbm_line(pbytes, pms, hbm_peak),
    }
    del y, py_o, py_h

    long_line = None if args.no_long else bench_long(kda, args, dev, stream, dist_on, hbm_peak)
    plong_line = None if args.no_long else bench_packed_long(kda, args, dev, stream, dist_on,
                                                             hbm_peak)
    sharded_line = bench_packed_sharded(kda, args, dev, stream, dist_on, hbm_peak) \
        if dist_on else None

    # rows beyond the hot path: prefix-cache checkpoints every 512 tokens on the
    # fixed-length batch, and the decode step with per-sequence commit counts
    ck_rows = B * (T // 512)
    ck = torch.empty(ck_rows, H, D, D, device=dev)
    cfn = lambda: kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, interval=512, out=o, hT=hT,
                                      ckpt=ck, workspace=ws)
    cms = _time_steps(cfn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    cbytes = B * T * H * BYTES_PER_TOKEN_HEAD + B * H * STATE_BYTES + ck_rows * H * STATE_BYTES
    del ck
    y = kda_inputs.decode_pool(num_seqs=1024, H=H, d=D, T_step=8, device=dev,
                               seed=1004 + 13 * rank)
    counts = torch.randint(0, 9, (1024,), generator=torch.Generator().manual_seed(7),
                           dtype=torch.int32).to(dev)
    out_d = torch.empty(1024, 8, H, D, device=dev)
    dws = kda.new_workspace(kda.make_shape(y.q, y.v), dev)
    kfn = lambda: kda.decode_commit(y.q, y.k, y.v, y.g, y.beta, y.h0, counts, out=out_d,
                                    workspace=dws)
    kms = _time_steps(kfn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    kbytes = 1024 * H * (2 * STATE_BYTES + 8 * BYTES_PER_TOKEN_HEAD)  # upper bound: all commit
    del y, out_d
    # fused input preprocessing on raw inputs of the same shapes, against the same
    # preprocessing done by torch ops followed by the plain prefill
    r = kda_inputs.draw_raw((B, T), H, D, D, device=dev, seed=1001 + 13 * rank)
    rfn = lambda: kda.fwd_preproc(r.q, r.k, r.v, r.g, r.beta, out=o, hT=hT, workspace=ws)
    rms = _time_steps(rfn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    st = kda.read_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.status_string(st)}")

    def unfused():
        f = torch.nn.functional
        qn = f.normalize(r.q.float(), dim=-1).to(r.q.dtype)
        kn = f.normalize(r.k.float(), dim=-1).to(r.k.dtype)
        gn = (-f.softplus(r.g.float())).to(r.g.dtype)
        bn = torch.sigmoid(r.beta.float()).to(r.beta.dtype)
        kda.fwd(qn, kn, r.v, gn, bn, out=o, hT=hT, workspace=ws)

    ums = _time_steps(unfused, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    del r
    y = kda_inputs.draw_raw((1024, 1), H, D, D, device=dev, seed=1004 + 13 * rank,
                            num_states=1024, h0_std=0.1)
    out_d = torch.empty(1024, 1, H, D, device=dev)
    dws = kda.new_workspace(kda.make_shape(y.q, y.v), dev)
    qfn = lambda: kda.decode_preproc(y.q, y.k, y.v, y.g, y.beta, y.h0, out=out_d,
                                     workspace=dws)
    qms = _time_steps(qfn, max(5, args.steps), max(3, args.warmup), stream, dist_on)
    qbytes = 1024 * H * (2 * STATE_BYTES + BYTES_PER_TOKEN_HEAD)
    del y, out_d
    # backward on the fixed-length batch: gradients of sum(o * dout), dout ~ N(0, 1)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1005 + 13 * rank)
    dout = torch.randn(B, T, H, D, generator=gen, device=dev)
    bshape = kda.make_shape(x.q, x.v)
    bws = torch.empty(kda.bwd_workspace_size(bshape), dtype=torch.uint8, device=dev)
    bfn = lambda: kda.bwd(x.q, x.k, x.v, x.g, x.beta, dout, want_dh0=False, workspace=bws)
    bms = _time_steps(bfn, max(3, args.steps // 4), 2, stream, dist_on)
    st = kda.read_device_status(bws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"device status {kda.status_string(st)}")
    del dout, bws
    bbytes = B * T * H * BWD_BYTES_PER_TOKEN_HEAD
    cms, kms, rms, ums, qms, bms = max_over_ranks([cms, kms, rms, ums, qms, bms], dev)
    fbytes = B * T * H * BYTES_PER_TOKEN_HEAD + B * H * STATE_BYTES
    next_rows = {
        "prefill_checkpoints_512": {
            "workload": WORKLOAD + "; state checkpoint every 512 tokens (32 per chain)",
            "ms_per_step": cms, "overhead_vs_prefill": cms / ms - 1.0,
            "roofline": _hbm_line(cbytes, cms, hbm_peak)},
        "decode_commit_T8": {
            "workload": "decode pool 1024 x 32 heads, T_step=8, commit counts uniform 0..8",
            "ms_per_step": kms, "tokens_per_s": 1024 * 8 * world / (kms * 1e-3),
            "roofline": dict(_hbm_line(kbytes, kms, hbm_peak),
                             note="bytes counted as if every sequence commits")},
        "prefill_preproc": {
            "workload": WORKLOAD.replace("bf16", "bf16 raw") +
            "; q/k L2 norm, -softplus gate, sigmoid beta fused",
            "ms_per_step": rms, "overhead_vs_prefill": rms / ms - 1.0,
            "unfused_ms_per_step": ums,
            "roofline": _hbm_line(fbytes, rms, hbm_peak)},
        "backward": {
            "workload": WORKLOAD + "; gradients dq, dk, dv, dg, dbeta of sum(o * dout), "
            "dout float32",
            "ms_per_step": bms, "vs_prefill": bms / ms,
            "tokens_per_s": B * T * H * world / H / (bms * 1e-3),
            "roofline": dict(_hbm_line(bbytes, bms, hbm_peak),
                             note="algorithmic bytes (inputs, dout, gradients); the sub-chunk "
                                  "states add 8 KB per token and head of workspace traffic")},
        "decode_preproc_T1": {
            "workload": "decode pool 1024 x 32 heads, T_step=1, raw inputs, preprocessing fused",
            "ms_per_step": qms, "tokens_per_s": 1024 * world / (qms * 1e-3),
            "roofline": _hbm_line(qbytes, qms, hbm_peak)},
    }
    clk = clocks.stop()

    ms, ms_e2e, ms_e2e1 = max_over_ranks([ms, ms_e2e, ms_e2e1], dev)
    for key in dec:
        dec[key]["ms_per_step"] = max_over_ranks([dec[key]["ms_per_step"]], dev)[0]

    tokens = B * T * world
    alg_bytes = B * T * H * BYTES_PER_TOKEN_HEAD + B * H * STATE_BYTES
    alg_flops = B * T * H * FLOP_PER_TOKEN_HEAD
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": tokens / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1); v N(0,1); g=-softplus(N(0,1)); "
                "beta=sigmoid(N(0,1)))",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "H": H, "dk": D, "dv": D,
                   "chunk": CHUNK, "tokens_per_rank": B * T,
                   "l2": "inputs and outputs (~0.8 GB) exceed L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic(),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "kda_prefill (one launch per step)",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "tensor_tflops_algorithmic": alg_flops / (ms * 1e-3) / 1e12,
                     "tensor_frac_of_bf16_peak": alg_flops / (ms * 1e-3) / 1e12 / bf16_peak},
        "e2e": {"value": tokens / (ms_e2e * 1e-3), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": f"pinned host inputs -> device -> kda_fwd -> o, hT to pinned host, "
                       f"pipelined in {E2E_SEQ_PARTS} sequences x {E2E_TIME_PARTS} time parts "
                       f"(copies in on one stream, a stream per sequence's kernels, each time "
                       f"part starting from the previous part's hT, copies out on another)",
                "serial_ms_per_step": ms_e2e1},
        "gpu_launches": args.steps,
        "clocks": clk,
        "decode": dec,
        "prefill_packed": packed_line,
        "next_rows": next_rows,
    }
    if long_line is not None:
        result["prefill_long"] = long_line
    if plong_line is not None:
        result["prefill_packed_long"] = plong_line
    if sharded_line is not None:
        result["prefill_packed_sharded"] = sharded_line
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = _cpu_baseline(kda_inputs.workload(1, device=dev))
    if dist_on:
        td.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_case(name):
    """One kernel's workload, run twice (a warm-up launch, then the one to
    capture: ``ncu -s 1 -c 1``), seeded and synthetic:

      prefill   the headline batch, B=4, T=4096, H=32, d=128, bf16
      packed    the 16-sequence packed batch with h0
      long      B=1, T=65,536, H=32 (one chain per head split into segments)
      long1m    B=1, T=1,048,576, H=32: the long-context call (segment split)
      decode1   1-token decode on a pool of 256 sequences x 32 heads
      decode8   8-token decode on the same pool
      bwd       the backward on B=1, T=512, H=4, d=128, bf16, with h0
    """
    import torch
    import kda_inputs
    import kda_delta_rule_fwd_gb300 as kda
    dev = torch.device("cuda:0")
    if name in ("prefill", "packed", "long", "long1m"):
        x = (kda_inputs.workload(1, device=dev) if name == "prefill" else
             kda_inputs.workload(2, device=dev) if name == "packed" else
             kda_inputs.workload(3, device=dev) if name == "long1m" else
             kda_inputs.fixed(1, 1 << 16, H, D, device=dev, seed=1003))
        for _ in range(2):
            out = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    elif name in ("decode1", "decode8"):
        x = kda_inputs.decode_pool(num_seqs=256, H=H, d=D, T_step=int(name[-1]), device=dev,
                                   seed=15)
        state = x.h0.clone()
        for _ in range(2):
            out = (kda.decode(x.q, x.k, x.v, x.g, x.beta, state), state)
    elif name == "bwd":
        x = kda_inputs.fixed(1, 512, 4, D, dtype=torch.bfloat16, device=dev, seed=5, h0_std=0.1)
        gen = torch.Generator(device=dev)
        gen.manual_seed(6)
        dout = torch.randn(x.v.shape, generator=gen, device=dev)
        for _ in range(2):
            out = kda.bwd(x.q, x.k, x.v, x.g, x.beta, dout, h0=x.h0)
    else:
        raise SystemExit(f"unknown case {name}")
    torch.cuda.synchronize()
    print(name, "ok", float(out[0].float().abs().sum()))


def run_reference(args):
    """The float64 oracle, as it stands, on the host's cores.  Each step is a
    bounded sample of the workload: the whole batch (B=4, T=4096) on a subset of
    heads sized from a one-head probe so the run stays within minutes."""
    rank, world, _ = _dist()
    if rank != 0:
        return
    import kda_inputs
    import oracle
    x = kda_inputs.workload(1, device="cpu")
    cores = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.recurrent(x.q[:1, :512, :1].contiguous(), x.k[:1, :512, :1].contiguous(),
                     x.v[:1, :512, :1].contiguous(), x.g[:1, :512, :1].contiguous(),
                     x.beta[:1, :512, :1].contiguous(), n_threads=1)
    rate1 = 512 / (time.perf_counter() - t0)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    heads = max(1, min(H, int(per_step_budget * rate1 * cores / (B * T))))
    sub = lambda a: a[:, :, :heads].contiguous()
    args_ = (sub(x.q), sub(x.k), sub(x.v), sub(x.g), x.beta[:, :, :heads].contiguous())
    for _ in range(args.warmup):
        oracle.recurrent(*args_, n_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrent(*args_, n_threads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = B * T * heads / dt / H
    sample = f"B={B}, T={T}, {heads} of {H} heads per step; tokens/s = head-tokens/s / H"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "H": H, "dk": D, "dv": D},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the 1M-token prefill")
    ap.add_argument("--case", help="run one kernel's workload (see run_case) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args.case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
