"""GPU parity of the backward (kda_bwd) against the float64 autograd oracle:
every gradient (dq, dk, dv, dg, dbeta, dh0) element by element, on fixed and
packed batches whose lengths fall on and around the 16-token sub-chunks, both
head sizes and both input dtypes, with and without a start state and a
final-state cotangent."""
import numpy as np
import pytest
import torch

import kda_inputs
from _util import rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-4  # the backward computes in float32 whatever the input dtype
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _cotangents(x, seed, dhT=True):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    do = torch.randn(x.v.shape, generator=gen, device=DEV)
    n = x.h0.shape[0] if x.h0 is not None else (x.q.shape[0] if x.cu_seqlens is None
                                                 else x.cu_seqlens.numel() - 1)
    H, dk, dv = x.q.shape[2], x.q.shape[3], x.v.shape[3]
    dh = 0.1 * torch.randn(n, H, dk, dv, generator=gen, device=DEV) if dhT else None
    return do, dh


def _check(kda, oracle_mod, x, do, dh, tol=TOL):
    got = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, cu_seqlens=x.cu_seqlens, h0=x.h0, dhT=dh)
    torch.cuda.synchronize()
    ref = oracle_mod.recurrent_grad(x.q, x.k, x.v, x.g, x.beta, do, cu_seqlens=x.cu_seqlens,
                                    h0=x.h0, dhT=dh)
    for name, a, b in zip(NAMES, got, ref):
        if b.size == 0:
            continue
        e = rel_err(a, b)
        assert e <= tol, f"{name}: {e:.3e} > {tol}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 100])
def test_fixed_length(kda, oracle_mod, dtype, d, T):
    x = kda_inputs.fixed(2, T, 2, d, dtype=dtype, device=DEV, seed=700 + T + d, h0_std=0.1)
    do, dh = _cotangents(x, 701 + T)
    _check(kda, oracle_mod, x, do, dh)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_packed_varlen(kda, oracle_mod, dtype, d):
    x = kda_inputs.packed([1, 16, 0, 33, 70, 2], 2, d, dtype=dtype, device=DEV, seed=710 + d,
                          h0_std=0.1)
    do, dh = _cotangents(x, 711)
    _check(kda, oracle_mod, x, do, dh)


def test_no_start_state_no_state_cotangent(kda, oracle_mod):
    x = kda_inputs.fixed(1, 50, 3, 128, dtype=torch.bfloat16, device=DEV, seed=720)
    do, _ = _cotangents(x, 721, dhT=False)
    _check(kda, oracle_mod, x, do, None)


def test_longer_sequence_and_nondefault_scale(kda, oracle_mod):
    """Many sub-chunks (the state cotangent travels through 19 of them) and a
    read-out scale other than dk^-1/2."""
    x = kda_inputs.fixed(1, 300, 2, 128, dtype=torch.bfloat16, device=DEV, seed=730,
                         h0_std=0.1)
    do, dh = _cotangents(x, 731)
    got = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, h0=x.h0, dhT=dh, scale=0.3)
    torch.cuda.synchronize()
    ref = oracle_mod.recurrent_grad(x.q, x.k, x.v, x.g, x.beta, do, h0=x.h0, dhT=dh, scale=0.3)
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(a, b) <= TOL, name


def test_state_cotangent_alone(kda, oracle_mod):
    """dout = 0: every gradient comes through the final state.  (Over a few hundred
    tokens of this gate distribution dh0 falls below float32's range, so 40 tokens.)"""
    x = kda_inputs.fixed(1, 40, 2, 128, dtype=torch.bfloat16, device=DEV, seed=732,
                         h0_std=0.1)
    do, dh = _cotangents(x, 733)
    zero = torch.zeros_like(do)
    got = kda.bwd(x.q, x.k, x.v, x.g, x.beta, zero, h0=x.h0, dhT=dh)
    torch.cuda.synchronize()
    ref = oracle_mod.recurrent_grad(x.q, x.k, x.v, x.g, x.beta, zero, h0=x.h0, dhT=dh)
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(a, b) <= TOL, name


def test_strong_gates(kda, oracle_mod):
    """Gates of -30 on some channels and tokens.  Tokens 20-22 of head 1 stay within
    the range where the pairwise factors are split; tokens 33-38 of head 0 (-180
    nats in one sub-chunk) take the explicit exponentials of differences."""
    x = kda_inputs.fixed(1, 50, 2, 64, dtype=torch.float32, device=DEV, seed=740, h0_std=0.1)
    x.g[0, 5, 0, :10] = -30.0
    x.g[0, 20:23, 1, 3] = -30.0
    x.g[0, 33:39, 0, :4] = -30.0
    do, dh = _cotangents(x, 741)
    _check(kda, oracle_mod, x, do, dh)


def test_empty_batch_passes_the_state_cotangent(kda):
    x = kda_inputs.packed([0, 0], 2, 128, dtype=torch.bfloat16, device=DEV, seed=750,
                          h0_std=0.1)
    do, dh = _cotangents(x, 751)
    got = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, cu_seqlens=x.cu_seqlens, h0=x.h0, dhT=dh)
    torch.cuda.synchronize()
    assert torch.equal(got[5], dh)


def test_bad_cu_seqlens_is_reported(kda):
    x = kda_inputs.packed([10, 20], 1, 64, dtype=torch.float32, device=DEV, seed=760)
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device=DEV)
    do = torch.zeros_like(x.v, dtype=torch.float32)
    shape = kda.make_shape(x.q, x.v, packed_seqs=2)
    ws = torch.empty(kda.bwd_workspace_size(shape), dtype=torch.uint8, device=DEV)
    kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, cu_seqlens=bad, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_ERR_BAD_SEQLENS


@pytest.mark.parametrize("d", [64, 128])
def test_repeatable_bit_for_bit(kda, d):
    """Two calls on the same inputs give the same gradients bit for bit: every
    cross-warp sum (dbeta's row sums among them) is taken in a fixed order."""
    x = kda_inputs.fixed(2, 300, 4, d, dtype=torch.bfloat16, device=DEV, seed=760 + d,
                         h0_std=0.1)
    do, dh = _cotangents(x, 761)
    a = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, h0=x.h0, dhT=dh)
    b = kda.bwd(x.q, x.k, x.v, x.g, x.beta, do, h0=x.h0, dhT=dh)
    torch.cuda.synchronize()
    for name, u, v in zip(NAMES, a, b):
        assert torch.equal(u, v), name
