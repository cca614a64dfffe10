"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses, against the float64 oracle:

* fixed-length prefill B=4, T=4096, H=32, d=128 (bf16): every element;
* packed prefill, 16 sequences of 128..8192 tokens with h0 ~ N(0, 0.1^2): every element;
* long context B=1, T=1,048,576, H=32: two seeded, sampled heads over the full length;
* decode pool of 1024 sequences (T_step 1 and 8): every element;
* the fused preprocessing on the fixed-length batch: every element;
* the backward of the fixed-length batch: exact zeros past the cotangent's support and
  two sampled (sequence, head) chains (tolerance 1e-4, float32 throughout).

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
def test_decode_pool_full(kda, oracle_mod, T_step):
    """Every element of o and of the updated state, all 1024 sequences x 32 heads.  The
    oracle runs 128 sequences at a time (host memory); max|err| and the rms of the
    reference are accumulated over the whole pool, so the metric is the pool's."""
    x = kda_inputs.decode_pool(num_seqs=1024, H=32, d=128, T_step=T_step, device=DEV)
    state = x.h0.clone()
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    torch.cuda.synchronize()
    acc = {"o": [0.0, 0.0, 0], "h": [0.0, 0.0, 0]}  # max|err|, sum ref^2, count

    def add(key, got, ref):
        got = got.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        a = acc[key]
        a[0] = max(a[0], float(np.max(np.abs(got - ref))))
        a[1] += float(np.sum(ref * ref))
        a[2] += ref.size

    for s0 in range(0, 1024, 128):
        sl = lambda t: t[s0:s0 + 128].contiguous().cpu()
        o_ref, h_ref = oracle_mod.recurrent(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta),
                                            h0=sl(x.h0))
        add("o", o[s0:s0 + 128], o_ref)
        add("h", state[s0:s0 + 128], h_ref)
        del o_ref, h_ref
    eo, eh = (acc[k][0] / np.sqrt(acc[k][1] / acc[k][2]) for k in ("o", "h"))
    _report(f"decode T_step={T_step} (all 1024 sequences)", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16


def test_fused_preprocessing_full(kda, oracle_mod):
    """The fixed-length batch on raw inputs with all three preprocessing steps fused,
    the bench's launch: every element against the oracle's preprocessing and
    recurrence."""
    r = kda_inputs.draw_raw((4, 4096), 32, 128, 128, device=DEV, seed=1001)
    o, hT = kda.fwd_preproc(r.q, r.k, r.v, r.g, r.beta)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(r.q, r.k, r.g, r.beta)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, r.v, fg, fb)
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    _report("fused preprocessing B=4 T=4096 H=32", eo, eh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16


def test_backward_full_sampled(kda, oracle_mod):
    """The backward on the full B=4, T=4096, H=32 batch (the bench's launch) with
    dout nonzero on the first 512 tokens only.  Every gradient past token 512 must
    then be exactly zero, and on two seeded (sequence, head) samples the first 512
    tokens' gradients match the oracle's autograd (which needs only those tokens)."""
    x = kda_inputs.workload(1, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1005)
    do = torch.randn(x.v.shape, generator=gen, device=DEV)
    do[:, 512:] = 0
    grads = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do)
    torch.cuda.synchronize()
    for gr in grads[:5]:
        assert torch.count_nonzero(gr[:, 512:]) == 0
    pick = torch.Generator().manual_seed(1006)
    for _ in range(2):
        b = int(torch.randint(0, 4, (1,), generator=pick))
        h = int(torch.randint(0, 32, (1,), generator=pick))
        sl = lambda t: t[b:b + 1, :512, h:h + 1].contiguous().cpu()
        ref = oracle_mod.recurrent_grad(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), sl(do))
        for name, a, e in zip(("dq", "dk", "dv", "dg", "dbeta"), grads[:5], ref[:5]):
            err = rel_err(a[b:b + 1, :512, h:h + 1], e)
            print(f"backward B=4 T=4096 H=32, sample ({b}, {h}) {name}: {err:.3e}")
            assert err <= 1e-4, (name, b, h, err)
        assert rel_err(grads[5][b:b + 1, h:h + 1], ref[5]) <= 1e-4  # that chain's dh0
