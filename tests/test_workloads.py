"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses, against the float64 oracle:

* fixed-length prefill B=4, T=4096, H=32, d=128 (bf16): every element;
* packed prefill, 16 sequences of 128..8192 tokens with h0 ~ N(0, 0.1^2): every element;
* long context B=1, T=1,048,576, H=32: two seeded, sampled heads over the full length;
* decode pool of 1024 sequences (T_step 1 and 8): a seeded sample of 64 sequences.

Tolerance: max|err| / rms(ref) <= 1e-2 for bf16 inputs with float32 state,
per output tensor.
"""
import numpy as np
import pytest
import torch

import kda_inputs
from _util import TOL_BF16, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _report(name, eo, eh):
    print(f"{name}: max|err|/rms  o {eo:.3e}  hT {eh:.3e}")


def test_fixed_length_prefill_full(kda, oracle_mod):
    x = kda_inputs.workload(1, device=DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta)
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    _report("B=4 T=4096 H=32", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16


def test_packed_varlen_prefill_full(kda, oracle_mod):
    x = kda_inputs.workload(2, device=DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    _report(f"packed 16 seqs ({x.q.shape[1]} tokens)", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16


def test_long_context_prefill_sampled_heads(kda, oracle_mod):
    x = kda_inputs.workload(3, device=DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(1003)
    heads = torch.randperm(32, generator=gen)[:2].tolist()
    sub = lambda t: t[:, :, heads].contiguous().cpu()
    q, k, v, g, b = (sub(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    o_s = o[:, :, heads].cpu()
    h_s = hT[:, heads].cpu()
    del x, o, hT
    torch.cuda.empty_cache()
    o_ref, h_ref = oracle_mod.recurrent(q, k, v, g, b)
    eo, eh = rel_err(o_s, o_ref), rel_err(h_s, h_ref)
    _report(f"T=1,048,576 heads {heads}", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16


@pytest.mark.parametrize("T_step", [1, 8])
def test_decode_pool_sampled_sequences(kda, oracle_mod, T_step):
    x = kda_inputs.decode_pool(num_seqs=1024, H=32, d=128, T_step=T_step, device=DEV)
    state = x.h0.clone()
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(2000 + T_step)
    seqs = torch.randperm(1024, generator=gen)[:64].sort().values
    pick = lambda t: t[seqs.to(t.device)].contiguous().cpu()
    o_ref, h_ref = oracle_mod.recurrent(pick(x.q), pick(x.k), pick(x.v), pick(x.g),
                                        pick(x.beta), h0=pick(x.h0))
    eo, eh = rel_err(pick(o), o_ref), rel_err(pick(state), h_ref)
    _report(f"decode T_step={T_step} (64 of 1024 sequences)", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16
