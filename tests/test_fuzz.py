"""Seeded random configurations (48 prefill, 24 decode), each compared with the
float64 oracle element by element: the prefill (both input dtypes, both head sizes,
fixed-length and packed batches with empty, one-token and chunk-edge lengths, with and
without a start state, gates from the workloads' strength to ones that send whole chunks
to the exact token path, alpha = 0 on some channels) and the decode (pool sizes, step
counts, commit counts, both dtypes and head sizes).  The draws come from fixed seeds, so
every run checks the same cases."""
import numpy as np
import pytest
import torch

import kda_inputs
from _util import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.float32: TOL_F32, torch.bfloat16: TOL_BF16}
EDGE_LENGTHS = [0, 1, 2, 63, 64, 65, 127, 128, 129, 191, 256, 320]


def _prefill_case(i):
    rng = np.random.default_rng(9000 + i)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    d = 128 if dtype == torch.bfloat16 and rng.random() < 0.8 else int(rng.choice([64, 128]))
    H = int(rng.integers(1, 4))
    gate_mult = float(rng.choice([1.0, 1.0, 3.0, 10.0, 40.0]))
    h0_std = 0.1 if rng.random() < 0.6 else None
    if rng.random() < 0.5:
        n = int(rng.integers(1, 7))
        lens = [int(rng.choice(EDGE_LENGTHS)) if rng.random() < 0.5 else int(rng.integers(0, 400))
                for _ in range(n)]
        x = kda_inputs.packed(lens, H, d, dtype=dtype, device=DEV, seed=9100 + i,
                              h0_std=h0_std)
        desc = f"packed {lens}"
    else:
        B, T = int(rng.integers(1, 4)), int(rng.integers(1, 400))
        x = kda_inputs.fixed(B, T, H, d, dtype=dtype, device=DEV, seed=9100 + i, h0_std=h0_std)
        desc = f"fixed B={B} T={T}"
    g = x.g.float() * gate_mult
    alpha0 = rng.random() < 0.2
    if alpha0:  # alpha = 0 on one channel of one head, on every token
        g[..., int(rng.integers(0, H)), int(rng.integers(0, d))] = float("-inf")
    x.g = g.to(dtype).contiguous()
    out_bf16 = dtype == torch.bfloat16 and rng.random() < 0.2
    return x, dtype, out_bf16, (f"{desc} H={H} d={d} {dtype} gates x{gate_mult} "
                                f"alpha0={alpha0} h0={h0_std}")


@pytest.mark.parametrize("i", range(48))
def test_prefill_random_case(kda, oracle_mod, i):
    x, dtype, out_bf16, desc = _prefill_case(i)
    out_dtype = torch.bfloat16 if out_bf16 else torch.float32
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                    out_dtype=out_dtype)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    tol = TOL[dtype]
    if o_ref.size:
        if out_bf16:  # plus the output rounding itself: half a bf16 ulp of |o|
            diff = np.abs(o.float().cpu().numpy() - o_ref)
            bound = tol * np.sqrt(np.mean(o_ref ** 2)) + np.abs(o_ref) * 2.0 ** -8
            assert np.all(diff <= bound), desc
        else:
            assert rel_err(o, o_ref) <= tol, desc
    assert rel_err(hT, h_ref) <= tol, desc


def _decode_case(i):
    rng = np.random.default_rng(9500 + i)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    d = int(rng.choice([64, 128]))
    num_seqs, H = int(rng.integers(1, 41)), int(rng.integers(1, 5))
    T_step = int(rng.integers(1, 9))
    x = kda_inputs.decode_pool(num_seqs=num_seqs, H=H, d=d, T_step=T_step, dtype=dtype,
                               device=DEV, seed=9600 + i)
    gate_mult = float(rng.choice([1.0, 5.0, 30.0]))
    x.g = (x.g.float() * gate_mult).to(dtype).contiguous()
    counts = ([int(c) for c in rng.integers(0, T_step + 1, num_seqs)]
              if rng.random() < 0.4 else None)
    return x, dtype, counts, (f"pool {num_seqs} H={H} d={d} T_step={T_step} {dtype} "
                              f"gates x{gate_mult} counts={counts}")


@pytest.mark.parametrize("i", range(24))
def test_decode_random_case(kda, oracle_mod, i):
    x, dtype, counts, desc = _decode_case(i)
    state = x.h0.clone()
    if counts is None:
        o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    else:
        o = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                              torch.tensor(counts, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    tol = TOL[dtype]
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= tol, desc
    if counts is None:
        assert rel_err(state, h_ref) <= tol, desc
        return
    for n, c in enumerate(counts):  # the state after the accepted prefix
        if c == 0:
            assert torch.equal(state[n], x.h0[n]), desc
            continue
        sl = lambda t: t[n:n + 1, :c].contiguous()
        _, h = oracle_mod.recurrent(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta),
                                    h0=x.h0[n:n + 1].contiguous())
        assert rel_err(state[n], h[0]) <= tol, desc
