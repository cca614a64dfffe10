"""GPU parity of the fused input preprocessing (q/k L2 normalisation, decay
log(alpha) = -softplus(g), beta = sigmoid(beta)) in prefill and decode: the
CUDA path on raw inputs against the float64 oracle run on the oracle's own
preprocessing of the same inputs."""
import itertools

import pytest
import torch

import kda_inputs
from _util import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.float32: TOL_F32, torch.bfloat16: TOL_BF16}
STEPS = ("qk_l2norm", "gate_softplus", "beta_sigmoid")


def _raw_fixed(B, T, H, d, dtype, seed):
    return kda_inputs.draw_raw((B, T), H, d, d, dtype=dtype, device=DEV, seed=seed,
                               num_states=B, h0_std=0.1)


def _raw_packed(lengths, H, d, dtype, seed):
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    x = kda_inputs.draw_raw((1, int(cu[-1])), H, d, d, dtype=dtype, device=DEV, seed=seed,
                            num_states=len(lengths), h0_std=0.1)
    x.cu_seqlens = cu.to(torch.int32).to(DEV)
    return x


def _split(oracle_mod, x, on):
    """Kernel inputs that leave exactly the steps in ``on`` to the kernel (the
    others applied beforehand by the oracle, the results cast to the input dtype
    as a caller would store them) and the oracle's fully preprocessed inputs from
    those same values."""
    off = {s: s not in on for s in STEPS}
    pre = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, **off)
    kq, kk, kg, kb = (t.to(x.q.dtype).contiguous() for t in pre)
    full = oracle_mod.preprocess(kq, kk, kg, kb, **{s: s in on for s in STEPS})
    dev = lambda t: t.to(DEV).contiguous()
    return (dev(kq), dev(kk), dev(kg), dev(kb)), full


def _check_prefill(kda, oracle_mod, x, dtype, on=STEPS):
    (q, k, g, b), (fq, fk, fg, fb) = _split(oracle_mod, x, on)
    flags = {s: s in on for s in STEPS}
    o, hT = kda.fwd_preproc(q, k, x.v, g, b, cu_seqlens=x.cu_seqlens, h0=x.h0, **flags)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, cu_seqlens=x.cu_seqlens, h0=x.h0)
    tol = TOL[dtype]
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    assert eo <= tol, f"o: {eo:.3e} > {tol}"
    assert eh <= tol, f"hT: {eh:.3e} > {tol}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_prefill_all_steps(kda, oracle_mod, dtype, d, T):
    x = _raw_fixed(2, T, 3, d, dtype, seed=500 + T + d)
    _check_prefill(kda, oracle_mod, x, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_packed(kda, oracle_mod, dtype):
    x = _raw_packed([1, 64, 0, 130, 77], 2, 128, dtype, seed=510)
    _check_prefill(kda, oracle_mod, x, dtype)


@pytest.mark.parametrize("on", [c for r in (1, 2) for c in itertools.combinations(STEPS, r)],
                         ids=lambda c: "+".join(s.split("_")[0] for s in c))
def test_prefill_each_step_alone_and_in_pairs(kda, oracle_mod, on):
    x = _raw_fixed(1, 150, 2, 128, torch.bfloat16, seed=520)
    _check_prefill(kda, oracle_mod, x, torch.bfloat16, on=on)


def test_prefill_no_steps_equals_plain_forward(kda):
    """With every flag off the fused entry point is the plain prefill, bit for bit."""
    x = kda_inputs.fixed(2, 130, 2, 128, dtype=torch.bfloat16, device=DEV, seed=530,
                         h0_std=0.1)
    o1, h1 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    o2, h2 = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, qk_l2norm=False,
                             gate_softplus=False, beta_sigmoid=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_zero_vectors_and_large_gates(kda, oracle_mod, dtype):
    """A zero q or k row stays zero (the norm floor); gate inputs far above the
    softplus threshold and very negative ones are handled as in the oracle."""
    x = _raw_fixed(1, 100, 2, 128, dtype, seed=540)
    x.q[0, 3, 0] = 0
    x.k[0, 70, 1] = 0
    x.g[0, 10, 0, :8] = 30.0
    x.g[0, 11, 1, :8] = -30.0
    x.beta[0, 12, :] = torch.tensor([40.0, -40.0], dtype=dtype)
    _check_prefill(kda, oracle_mod, x, dtype)


def test_prefill_long_chain_split(kda, oracle_mod):
    """The segment split of a very long chain applies the same preprocessing in
    every launch of the plan."""
    x = _raw_fixed(1, 64 * 257 + 37, 1, 128, torch.bfloat16, seed=550)
    shape = kda.make_shape(x.q, x.v)
    assert kda.workspace_size(shape) > 256
    _check_prefill(kda, oracle_mod, x, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T_step", [1, 3, 8])
def test_decode_all_steps(kda, oracle_mod, dtype, d, T_step):
    x = kda_inputs.draw_raw((5, T_step), 3, d, d, dtype=dtype, device=DEV, seed=560 + T_step,
                            num_states=5, h0_std=0.1)
    x.k[1, 0, 2] = 0
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta)
    state = x.h0.clone()
    o = kda.decode_preproc(x.q, x.k, x.v, x.g, x.beta, state)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(state, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("on", [(s,) for s in STEPS], ids=lambda c: c[0].split("_")[0])
def test_decode_each_step_alone(kda, oracle_mod, on):
    x = kda_inputs.draw_raw((4, 8), 2, 128, 128, dtype=torch.bfloat16, device=DEV, seed=570,
                            num_states=4, h0_std=0.1)
    (q, k, g, b), (fq, fk, fg, fb) = _split(oracle_mod, x, on)
    state = x.h0.clone()
    o = kda.decode_preproc(q, k, x.v, g, b, state, **{s: s in on for s in STEPS})
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(state, h_ref) <= TOL_BF16


def test_decode_preproc_continues_prefill_preproc(kda, oracle_mod):
    """Prefill of a prompt then decode steps, both on raw inputs, match one oracle
    run over the whole sequence."""
    x = _raw_fixed(2, 140, 2, 128, torch.bfloat16, seed=580)
    P = 128
    pre = lambda t: t[:, :P].contiguous()
    post = lambda t: t[:, P:].contiguous()
    _, hT = kda.fwd_preproc(pre(x.q), pre(x.k), pre(x.v), pre(x.g), pre(x.beta), h0=x.h0)
    outs = []
    for s in range(0, 12, 4):
        sl = lambda t: post(t)[:, s:s + 4].contiguous()
        outs.append(kda.decode_preproc(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), hT))
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(torch.cat(outs, 1), o_ref[:, P:]) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_gate_activation_precision(kda):
    """float32 decode from h0 = I with k = 0: the state after one token is
    diag(alpha), alpha = exp(-softplus(g)), so its diagonal shows the kernel's
    gate activation.  Over g in [-40, 40] the relative error of alpha (= the
    absolute error of log(alpha)) stays within the activation's 4e-7 plus the
    float32 roundings of log(alpha) and of exp."""
    n, H, d = 48, 4, 128
    gen = torch.Generator().manual_seed(590)
    graw = torch.linspace(-40.0, 40.0, n * H * d, dtype=torch.float64)
    graw = graw[torch.randperm(graw.numel(), generator=gen)].reshape(n, 1, H, d)
    g32 = graw.float()
    q = torch.randn(n, 1, H, d, generator=gen)
    v = torch.randn(n, 1, H, d, generator=gen)
    b = torch.randn(n, 1, H, generator=gen)
    k = torch.zeros(n, 1, H, d)
    state = torch.eye(d).expand(n, H, d, d).contiguous().to(DEV)
    kda.decode_preproc(q.to(DEV), k.to(DEV), v.to(DEV), g32.to(DEV), b.to(DEV), state)
    torch.cuda.synchronize()
    st = state.double().cpu()
    alpha = st.diagonal(dim1=-2, dim2=-1)
    off = st - torch.diag_embed(alpha)
    assert torch.count_nonzero(off) == 0
    logalpha = -torch.logaddexp(torch.zeros_like(graw), g32.double())[:, 0]
    ref = torch.exp(logalpha)
    rel = (alpha - ref).abs() / ref
    bound = 7e-7 + 1.2e-7 * logalpha.abs()
    assert torch.all(rel <= bound), float((rel / bound).max())


def _gate_scale(H, seed):
    gen = torch.Generator().manual_seed(seed)
    return (torch.rand(H, generator=gen) * 1.5 + 0.25).to(DEV)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 128),
                                     (torch.float32, 64), (torch.bfloat16, 64)],
                         ids=["bf16-128", "f32-128", "f32-64", "bf16-64"])
@pytest.mark.parametrize("per_head", [False, True], ids=["per-channel", "per-head"])
def test_prefill_gate_scale_and_scalar_gate(kda, oracle_mod, dtype, d, per_head):
    """log(alpha) = -a_h softplus(g) with a per-head scale a_h, per channel and in the
    scalar-gate variant (g [B, T, H] shared by the key channels), packed."""
    x = _raw_packed([1, 64, 0, 130, 77], 3, d, dtype, seed=600 + d)
    if per_head:
        x.g = x.g[..., 0].contiguous()
    a = _gate_scale(3, 601)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                            gate_per_head=per_head, gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=per_head,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, cu_seqlens=x.cu_seqlens, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 128),
                                     (torch.float32, 64)], ids=["bf16-128", "f32-128", "f32-64"])
@pytest.mark.parametrize("per_head", [False, True], ids=["per-channel", "per-head"])
def test_prefill_gate_scale_8(kda, oracle_mod, dtype, d, per_head):
    """A per-head decay-rate scale of 8: log(alpha) = -8 softplus(g), about 6.5 nats
    per token on average, so most chunks exceed the span one factorisation holds and
    the bf16 path runs them token by token.  Packed, with an empty sequence."""
    x = _raw_packed([1, 64, 0, 130, 77, 200], 2, d, dtype, seed=640 + d)
    if per_head:
        x.g = x.g[..., 0].contiguous()
    a = torch.full((2,), 8.0, device=DEV)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                            gate_per_head=per_head, gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=per_head,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, cu_seqlens=x.cu_seqlens, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("per_head", [False, True], ids=["per-channel", "per-head"])
def test_prefill_more_chains_than_sms(kda, oracle_mod, per_head):
    """320 (sequence, head) chains of mixed lengths: the persistent CTAs each take
    several chains in turn, with the gate activation and the norms fused."""
    gen = torch.Generator().manual_seed(660)
    lens = torch.randint(1, 200, (40,), generator=gen).tolist()
    x = _raw_packed(lens, 8, 128, torch.bfloat16, seed=661)
    if per_head:
        x.g = x.g[..., 0].contiguous()
    a = _gate_scale(8, 662)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                            gate_per_head=per_head, gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=per_head,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, cu_seqlens=x.cu_seqlens, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_prefill_fixed_length_more_chains_than_sms(kda, oracle_mod):
    """B=5, H=40 (200 chains) on raw inputs with every step fused."""
    x = _raw_fixed(5, 90, 40, 128, torch.bfloat16, seed=670)
    _check_prefill(kda, oracle_mod, x, torch.bfloat16)


def test_decode_gate_scale_8(kda, oracle_mod):
    x = kda_inputs.draw_raw((5, 8), 3, 128, 128, dtype=torch.bfloat16, device=DEV, seed=650,
                            num_states=5, h0_std=0.1)
    a = torch.full((3,), 8.0, device=DEV)
    state = x.h0.clone()
    o = kda.decode_preproc(x.q, x.k, x.v, x.g, x.beta, state, gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(state, h_ref) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_scalar_log_decay_without_softplus(kda, oracle_mod, dtype):
    """A per-head gate given directly as log(alpha) (no activation) is broadcast over
    the key channels: the scalar-gate (GDN) recurrence, several chunks."""
    x = _raw_fixed(2, 200, 2, 128, dtype, seed=610)
    graw = x.g[..., 0].contiguous()
    lg = oracle_mod.preprocess(x.q, x.k, graw, x.beta, qk_l2norm=False, beta_sigmoid=False,
                               gate_per_head=True)[2][..., 0].contiguous().to(DEV)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, lg, x.beta, h0=x.h0, gate_softplus=False,
                            gate_per_head=True)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, lg, x.beta, gate_softplus=False,
                                           gate_per_head=True)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(hT, h_ref) <= TOL[dtype]


def test_prefill_scalar_gate_long_chain_split(kda, oracle_mod):
    x = _raw_fixed(1, 64 * 257 + 37, 1, 128, torch.bfloat16, seed=620)
    x.g = x.g[..., 0].contiguous()
    a = _gate_scale(1, 621)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, gate_per_head=True,
                            gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=True,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("per_head", [False, True], ids=["per-channel", "per-head"])
def test_decode_gate_scale_and_scalar_gate(kda, oracle_mod, dtype, per_head):
    x = kda_inputs.draw_raw((5, 8), 3, 128, 128, dtype=dtype, device=DEV, seed=630,
                            num_states=5, h0_std=0.1)
    if per_head:
        x.g = x.g[..., 0].contiguous()
    a = _gate_scale(3, 631)
    state = x.h0.clone()
    o = kda.decode_preproc(x.q, x.k, x.v, x.g, x.beta, state, gate_per_head=per_head,
                           gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=per_head,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(state, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("per_head", [False, True], ids=["per-channel", "per-head"])
def test_decode_preproc_many_chains(kda, oracle_mod, per_head):
    """The fused preprocessing on a pool of 96 x 5 = 480 chains, more than the
    device holds CTAs at once: every chain's scalars (beta, a per-head gate, its
    head's gate scale) and normalised q, k must follow their chain."""
    x = kda_inputs.draw_raw((96, 8), 5, 128, 128, dtype=torch.bfloat16, device=DEV, seed=640,
                            num_states=96, h0_std=0.1)
    if per_head:
        x.g = x.g[..., 0].contiguous()
    a = _gate_scale(5, 641)
    state = x.h0.clone()
    o = kda.decode_preproc(x.q, x.k, x.v, x.g, x.beta, state, qk_l2norm=True,
                           gate_softplus=True, beta_sigmoid=True, gate_per_head=per_head,
                           gate_scale=a)
    torch.cuda.synchronize()
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta, gate_per_head=per_head,
                                           gate_scale=a)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(state, h_ref) <= TOL_BF16
