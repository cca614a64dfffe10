"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than itself: a
hand-derived worked example, a closed form, a special case that reduces to a
textbook result, an independent dense (Kronecker) formulation, or an
algebraic property of the recurrence.  Together they catch a dropped term, a
wrong sign or index, a transposed state, a decay applied on the wrong side,
and a read-out taken before the write.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, L, H, dk, dv, *, decay=(0.0, 1.0)):
    """float64 inputs with unit-norm q, k and gates alpha = exp(g) in a range."""
    q = rng.standard_normal((L, H, dk))
    k = rng.standard_normal((L, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((L, H, dv))
    lo, hi = decay
    alpha = rng.uniform(max(lo, 1e-3), hi, (L, H, dk))
    g = np.log(alpha)
    beta = rng.uniform(0.0, 1.0, (L, H))
    return q, k, v, g, beta


def _run(oracle, q, k, v, g, beta, h0=None, scale=None, cu=None):
    L, H = beta.shape
    if cu is None:
        cu = np.array([0, L])
    return oracle.recurrent(q, k, v, g, beta, cu_seqlens=cu, h0=h0, scale=scale)


# 1. hand-derived worked examples ------------------------------------------------

def test_scalar_two_token_golden(oracle_mod):
    d = json.load(open(os.path.join(GOLDEN, "scalar_two_token.json")))
    L = len(d["beta"])
    sh = lambda x, w: np.array(x, dtype=np.float64).reshape(L, 1, w)
    o, hT = _run(oracle_mod, sh(d["q"], 1), sh(d["k"], 1), sh(d["v"], 1),
                 np.log(sh(d["alpha"], 1)), np.array(d["beta"]).reshape(L, 1),
                 h0=np.array(d["h0"]).reshape(1, 1, 1, 1), scale=d["scale"])
    np.testing.assert_allclose(o.reshape(L, 1), d["o"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(hT.reshape(1, 1), d["hT"], rtol=0, atol=1e-15)


def test_matrix_two_token_golden(oracle_mod):
    d = json.load(open(os.path.join(GOLDEN, "matrix_two_token.json")))
    S = np.array(d["h0"], dtype=np.float64).reshape(1, 1, 2, 2)
    for t in range(2):
        row = lambda key: np.array(d[key][t], dtype=np.float64).reshape(1, 1, -1)
        o, S = _run(oracle_mod, row("q"), row("k"), row("v"), np.log(row("alpha")),
                    np.array([[d["beta"][t]]]), h0=S, scale=d["scale"][t])
        np.testing.assert_allclose(o.reshape(2), d["o"][t], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S.reshape(2, 2), d["hT"], rtol=0, atol=1e-14)


# 2. closed forms and special cases ------------------------------------------------

def test_beta_zero_is_pure_channel_decay(oracle_mod):
    """beta = 0: no writes, so hT = diag(exp(sum g)) h0 and
    o_t = scale * h0^T (exp(Gamma_t) * q_t) with Gamma_t the inclusive log-decay sum."""
    rng = np.random.default_rng(1)
    L, H, dk, dv = 37, 2, 6, 5
    q, k, v, g, beta = _rand_inputs(rng, L, H, dk, dv, decay=(0.5, 1.0))
    beta[:] = 0.0
    h0 = rng.standard_normal((1, H, dk, dv))
    o, hT = _run(oracle_mod, q, k, v, g, beta, h0=h0, scale=0.3)
    Gam = np.cumsum(g, axis=0)  # [L, H, dk]
    for h in range(H):
        np.testing.assert_allclose(hT[0, h], np.exp(Gam[-1, h])[:, None] * h0[0, h],
                                   rtol=1e-13, atol=1e-14)
        o_ref = 0.3 * (np.exp(Gam[:, h]) * q[:, h]) @ h0[0, h]
        np.testing.assert_allclose(o[:, h], o_ref, rtol=1e-12, atol=1e-13)


def test_ungated_orthonormal_keys_are_exact_memory(oracle_mod):
    """alpha = 1, beta = 1, h0 = 0, orthonormal keys: S = sum_i k_i v_i^T and
    S^T k_j = v_j exactly (the delta rule as an associative memory)."""
    rng = np.random.default_rng(2)
    dk, dv, n = 8, 3, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :n].T                       # n orthonormal rows
    vals = rng.standard_normal((n, dv))
    k = keys[:, None, :]
    q = keys[:, None, :]                     # read each key back right after writing it
    v = vals[:, None, :]
    g = np.zeros((n, 1, dk))
    beta = np.ones((n, 1))
    o, hT = _run(oracle_mod, q, k, v, g, beta, scale=1.0)
    np.testing.assert_allclose(hT[0, 0], keys.T @ vals, rtol=0, atol=1e-13)
    np.testing.assert_allclose(hT[0, 0].T @ keys.T, vals.T, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[:, 0], vals, rtol=0, atol=1e-13)


def test_beta_one_overwrites_same_key(oracle_mod):
    """alpha = 1, beta = 1: writing the same unit key twice leaves S^T k equal to
    the latest value (the second write replaces, not adds)."""
    dk, dv = 4, 2
    kvec = np.array([0.5, 0.5, 0.5, 0.5])
    k = np.stack([kvec, kvec])[:, None, :]
    v = np.array([[1.0, -2.0], [3.0, 4.0]])[:, None, :]
    g = np.zeros((2, 1, dk))
    beta = np.ones((2, 1))
    o, hT = _run(oracle_mod, k, k, v, g, beta, scale=1.0)
    np.testing.assert_allclose(hT[0, 0].T @ kvec, [3.0, 4.0], atol=1e-15)
    np.testing.assert_allclose(o[1, 0], [3.0, 4.0], atol=1e-15)


def test_single_token_from_zero(oracle_mod):
    """From S = 0 one token gives S = beta k v^T and o = scale beta (q.k) v."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta = _rand_inputs(rng, 1, 1, 5, 7)
    o, hT = _run(oracle_mod, q, k, v, g, beta, scale=0.7)
    np.testing.assert_allclose(hT[0, 0], beta[0, 0] * np.outer(k[0, 0], v[0, 0]), atol=1e-15)
    np.testing.assert_allclose(o[0, 0], 0.7 * beta[0, 0] * (q[0, 0] @ k[0, 0]) * v[0, 0],
                               atol=1e-15)


def test_scalar_gate_reduces_to_ungated_rule(oracle_mod):
    """Gated DeltaNet special case (one gate value shared by all channels).

    With A_t = prod_{m<=t} a_m, the scaled state S_t / A_t follows the ungated
    delta rule on values v_t / A_t.  So running the oracle with g = 0 on v / A
    and rescaling by A must reproduce the gated run: this pins where the decay
    enters (before the write, on the state only)."""
    rng = np.random.default_rng(4)
    L, dk, dv = 40, 6, 4
    q, k, v, _, beta = _rand_inputs(rng, L, 1, dk, dv)
    a = rng.uniform(0.9, 1.0, L)
    g = np.repeat(np.log(a)[:, None, None], dk, axis=2)
    h0 = rng.standard_normal((1, 1, dk, dv))
    o, hT = _run(oracle_mod, q, k, v, g, beta, h0=h0, scale=0.5)
    A = np.cumprod(a)
    o2, hT2 = _run(oracle_mod, q, k, v / A[:, None, None], np.zeros_like(g), beta, h0=h0,
                   scale=0.5)
    np.testing.assert_allclose(o, o2 * A[:, None, None], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, hT2 * A[-1], rtol=1e-11, atol=1e-12)


# 3. brute force through a different formulation -------------------------------------

@pytest.mark.parametrize("L,dk,dv", [(1, 3, 2), (2, 2, 3), (3, 4, 4), (4, 3, 5)])
def test_kronecker_vec_form(oracle_mod, L, dk, dv):
    """Column-stacked vec(S) evolves as vec(S_t) = (I_dv kron M_t) vec(S_{t-1}) +
    beta_t (v_t kron k_t) with the diagonal-plus-low-rank transition
    M_t = (I - beta_t k_t k_t^T) diag(alpha_t), and o_t = scale (I_dv kron q_t^T) vec(S_t)."""
    rng = np.random.default_rng(10 + L)
    q, k, v, g, beta = _rand_inputs(rng, L, 1, dk, dv)
    h0 = rng.standard_normal((1, 1, dk, dv))
    o, hT = _run(oracle_mod, q, k, v, g, beta, h0=h0, scale=0.9)
    vecS = h0[0, 0].reshape(-1, order="F")
    for t in range(L):
        kt, qt, vt, bt = k[t, 0], q[t, 0], v[t, 0], beta[t, 0]
        Mt = (np.eye(dk) - bt * np.outer(kt, kt)) @ np.diag(np.exp(g[t, 0]))
        vecS = np.kron(np.eye(dv), Mt) @ vecS + bt * np.kron(vt, kt)
        ot = 0.9 * np.kron(np.eye(dv), qt[None, :]) @ vecS
        np.testing.assert_allclose(o[t, 0], ot, rtol=0, atol=1e-13)
    np.testing.assert_allclose(hT[0, 0], vecS.reshape(dk, dv, order="F"), rtol=0, atol=1e-13)


def test_per_token_write_invariant(oracle_mod):
    """After token t: S_t^T k_t = (1 - beta_t |k_t|^2) (D_t S_{t-1})^T k_t + beta_t |k_t|^2 v_t,
    and o_t = scale S_t^T q_t, using prefix runs for S_{t-1} and S_t."""
    rng = np.random.default_rng(5)
    L, dk, dv = 9, 5, 3
    q, k, v, g, beta = _rand_inputs(rng, L, 1, dk, dv)
    k[:, 0] *= rng.uniform(0.5, 1.5, (L, 1))    # the identity holds for any key norm
    h0 = rng.standard_normal((1, 1, dk, dv))
    o, _ = _run(oracle_mod, q, k, v, g, beta, h0=h0, scale=0.25)
    prev = h0[0, 0]
    for t in range(L):
        sl = slice(0, t + 1)
        _, St = _run(oracle_mod, q[sl], k[sl], v[sl], g[sl], beta[sl], h0=h0, scale=0.25)
        St = St[0, 0]
        kt, bt = k[t, 0], beta[t, 0]
        DS = np.exp(g[t, 0])[:, None] * prev
        kk = kt @ kt
        np.testing.assert_allclose(St.T @ kt, (1 - bt * kk) * (DS.T @ kt) + bt * kk * v[t, 0],
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o[t, 0], 0.25 * St.T @ q[t, 0], rtol=1e-12, atol=1e-13)
        prev = St


# 4. algebraic properties -------------------------------------------------------------

def test_linear_in_values_and_start_state(oracle_mod):
    rng = np.random.default_rng(6)
    L, H, dk, dv = 50, 2, 8, 6
    q, k, v1, g, beta = _rand_inputs(rng, L, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    h1 = rng.standard_normal((1, H, dk, dv))
    h2 = rng.standard_normal((1, H, dk, dv))
    a, b = 0.7, -1.3
    o1, s1 = _run(oracle_mod, q, k, v1, g, beta, h0=h1)
    o2, s2 = _run(oracle_mod, q, k, v2, g, beta, h0=h2)
    o3, s3 = _run(oracle_mod, q, k, a * v1 + b * v2, g, beta, h0=a * h1 + b * h2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(s3, a * s1 + b * s2, rtol=1e-11, atol=1e-12)


def test_packed_equals_independent_runs(oracle_mod):
    """State resets at every packed boundary: no crosstalk between sequences."""
    rng = np.random.default_rng(7)
    lens = [5, 0, 17, 1, 33]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, dk, dv = 3, 4, 5
    q, k, v, g, beta = _rand_inputs(rng, int(cu[-1]), H, dk, dv)
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    o, hT = oracle_mod.recurrent(q, k, v, g, beta, cu_seqlens=cu, h0=h0)
    for n, (a, z) in enumerate(zip(cu[:-1], cu[1:])):
        o1, h1 = _run(oracle_mod, q[a:z], k[a:z], v[a:z], g[a:z], beta[a:z], h0=h0[n:n + 1])
        np.testing.assert_allclose(o[a:z], o1, rtol=0, atol=0)
        np.testing.assert_allclose(hT[n], h1[0], rtol=0, atol=0)
    # a zero-length sequence hands its start state straight through
    np.testing.assert_array_equal(hT[1], h0[1])


def test_stepwise_decode_equals_one_run(oracle_mod):
    """Eight T=1 steps chained through the state equal one 8-token run."""
    rng = np.random.default_rng(8)
    H, dk, dv = 2, 6, 6
    q, k, v, g, beta = _rand_inputs(rng, 8, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    o, hT = _run(oracle_mod, q, k, v, g, beta, h0=h0)
    S = h0
    for t in range(8):
        sl = slice(t, t + 1)
        ot, S = _run(oracle_mod, q[sl], k[sl], v[sl], g[sl], beta[sl], h0=S)
        np.testing.assert_allclose(ot, o[sl], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S, hT, rtol=1e-13, atol=1e-14)


def test_float32_and_float64_inputs_agree(oracle_mod):
    rng = np.random.default_rng(9)
    q, k, v, g, beta = (x.astype(np.float32).astype(np.float64)
                        for x in _rand_inputs(rng, 20, 2, 4, 4))
    o64, h64 = _run(oracle_mod, q, k, v, g, beta)
    o32, h32 = _run(oracle_mod, *(x.astype(np.float32) for x in (q, k, v, g, beta)))
    np.testing.assert_array_equal(o64, o32)
    np.testing.assert_array_equal(h64, h32)


# 5. the chunkwise form and the segment decomposition --------------------------------

@pytest.mark.parametrize("C,sub", [(1, 1), (2, 2), (4, 2), (16, 16), (16, 4), (64, 16),
                                   (64, 64)])
def test_chunked_equals_recurrent(oracle_mod, C, sub):
    """The chunkwise-parallel rearrangement (with the sub-chunk decay split) is exact."""
    rng = np.random.default_rng(20 + C)
    lens = [150, 64, 3, 0, 129]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, dk, dv = 2, 8, 6
    q, k, v, g, beta = _rand_inputs(rng, int(cu[-1]), H, dk, dv, decay=(0.3, 1.0))
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    o_r, h_r = oracle_mod.recurrent(q, k, v, g, beta, cu_seqlens=cu, h0=h0, scale=0.6)
    o_c, h_c = oracle_mod.chunked(q, k, v, g, beta, cu_seqlens=cu, h0=h0, scale=0.6,
                                  C=C, sub=sub)
    ref = np.sqrt(np.mean(o_r ** 2))
    assert np.max(np.abs(o_c - o_r)) <= 1e-12 * ref
    assert np.max(np.abs(h_c - h_r)) <= 1e-12 * np.sqrt(np.mean(h_r ** 2))


def test_chunked_on_the_workload_gate_distribution(oracle_mod):
    """Same check at d = 64 with the workloads' strong gates, g = -softplus(N(0,1)),
    where a 64-token chunk decays by about e^-52 per channel."""
    rng = np.random.default_rng(30)
    L, H, d = 200, 1, 64
    q, k, v, _, beta = _rand_inputs(rng, L, H, d, d)
    g = -np.logaddexp(0.0, rng.standard_normal((L, H, d)))
    o_r, h_r = _run(oracle_mod, q, k, v, g, beta)
    o_c, h_c = oracle_mod.chunked(q, k, v, g, beta, cu_seqlens=np.array([0, L]), C=64,
                                  sub=16)
    assert np.max(np.abs(o_c - o_r)) <= 1e-12 * np.sqrt(np.mean(o_r ** 2))
    assert np.max(np.abs(h_c - h_r)) <= 1e-12 * np.sqrt(np.mean(h_r ** 2))


def test_segment_composition_reproduces_full_run(oracle_mod):
    """S_end = M S_start + b per segment; folding the segments' affine maps in
    order reproduces the full-sequence final state (the context-parallel scan)."""
    rng = np.random.default_rng(40)
    L, dk, dv = 120, 6, 5
    q, k, v, g, beta = _rand_inputs(rng, L, 1, dk, dv, decay=(0.8, 1.0))
    h0 = rng.standard_normal((1, 1, dk, dv))
    _, hT = _run(oracle_mod, q, k, v, g, beta, h0=h0)
    cuts = [0, 13, 50, 51, 97, 120]
    segs = [oracle_mod.segment_transition(k[a:z, 0], v[a:z, 0], g[a:z, 0], beta[a:z, 0])
            for a, z in zip(cuts[:-1], cuts[1:])]
    total = segs[0]
    for s in segs[1:]:
        total = oracle_mod.compose(total, s)
    np.testing.assert_allclose(oracle_mod.apply_transition(total, h0[0, 0]), hT[0, 0],
                               rtol=1e-11, atol=1e-12)
    # associativity of the fold
    x, y, z = segs[0], segs[1], segs[3]
    l = oracle_mod.compose(oracle_mod.compose(x, y), z)
    r = oracle_mod.compose(x, oracle_mod.compose(y, z))
    np.testing.assert_allclose(l[0], r[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l[1], r[1], rtol=1e-12, atol=1e-13)
    # the transition of a segment is not the identity-free sum of zero-start states
    assert not np.allclose(hT[0, 0], sum(s[1] for s in segs))


# 6. input preprocessing ------------------------------------------------------------
def test_preprocess_closed_forms(oracle_mod):
    """sigmoid(0) = 1/2, softplus(0) = ln 2, softplus(x) - softplus(-x) = x,
    exp(-softplus(x)) = sigmoid(-x), and softplus(x) -> x for large x."""
    import torch
    x = torch.tensor([0.0, -3.0, -0.5, 0.25, 2.0, 19.5, 20.5, 60.0], dtype=torch.float64)
    q = torch.ones(x.numel(), 1, 4, dtype=torch.float64)
    _, _, g, b = oracle_mod.preprocess(q, q, x.view(-1, 1, 1).expand(-1, 1, 4), x.view(-1, 1),
                                       qk_l2norm=False)
    _, _, gm, bm = oracle_mod.preprocess(q, q, (-x).view(-1, 1, 1).expand(-1, 1, 4),
                                         (-x).view(-1, 1), qk_l2norm=False)
    sp, spm = -g[:, 0, 0].numpy(), -gm[:, 0, 0].numpy()
    sig, sigm = b[:, 0].numpy(), bm[:, 0].numpy()
    xs = x.numpy()
    assert sig[0] == 0.5
    assert abs(sp[0] - np.log(2.0)) < 1e-15
    exact = np.abs(xs) <= 20.0
    np.testing.assert_allclose((sp - spm)[exact], xs[exact], rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.exp(-sp)[exact], sigm[exact], rtol=1e-12, atol=0)
    # above 20 softplus is taken as x: the error is log1p(e^-x) < e^-20
    np.testing.assert_allclose((sp - spm)[~exact], xs[~exact], rtol=0, atol=np.exp(-20.0))
    np.testing.assert_allclose(sig + sigm, 1.0, rtol=0, atol=1e-15)
    assert sp[-1] == 60.0 and sp[-2] == 20.5
    # a decay from the gate is in (0, 1]: -softplus(x) < 0
    assert np.all(g.numpy() < 0)


def test_preprocess_l2_norm(oracle_mod):
    """Normalised q, k have unit norm and the same direction; a zero vector stays
    zero (the 1e-12 floor); the steps are independent of one another."""
    import torch
    rng = np.random.default_rng(61)
    q = torch.from_numpy(rng.standard_normal((5, 2, 7)) * 3.0)
    k = torch.from_numpy(rng.standard_normal((5, 2, 7)) * 0.01)
    k[2, 1] = 0.0
    g = torch.from_numpy(rng.standard_normal((5, 2, 7)))
    b = torch.from_numpy(rng.standard_normal((5, 2)))
    qn, kn, gn, bn = oracle_mod.preprocess(q, k, g, b, gate_softplus=False, beta_sigmoid=False)
    nq = torch.linalg.vector_norm(qn, dim=-1)
    nk = torch.linalg.vector_norm(kn, dim=-1)
    np.testing.assert_allclose(nq.numpy(), 1.0, rtol=0, atol=1e-14)
    mask = torch.ones(5, 2, dtype=torch.bool)
    mask[2, 1] = False
    np.testing.assert_allclose(nk[mask].numpy(), 1.0, rtol=0, atol=1e-14)
    assert torch.all(kn[2, 1] == 0)
    # same direction: x = ||x|| * x_hat
    np.testing.assert_allclose((qn * torch.linalg.vector_norm(q, dim=-1, keepdim=True)).numpy(),
                               q.numpy(), rtol=1e-13, atol=1e-15)
    assert torch.equal(gn, g) and torch.equal(bn, b)
    # all steps off: identity
    out = oracle_mod.preprocess(q, k, g, b, qk_l2norm=False, gate_softplus=False,
                                beta_sigmoid=False)
    for a, e in zip(out, (q, k, g, b)):
        assert torch.equal(a, e)


def test_preprocess_rounds_gate_and_beta_to_input_dtype(oracle_mod):
    """bf16 inputs: the gate and beta come back as bf16, each value the rounding of
    the float64 result; normalised q and k come back unrounded (float64), and with
    the norm step off q and k keep their dtype."""
    import torch
    x = torch.tensor([[[0.3, -1.7, 2.2, 0.0]]], dtype=torch.bfloat16)
    b = torch.tensor([[0.7]], dtype=torch.bfloat16)
    qn, kn, gn, bn = oracle_mod.preprocess(x, x, x, b)
    assert gn.dtype == torch.bfloat16 and bn.dtype == torch.bfloat16
    assert qn.dtype == torch.float64 and kn.dtype == torch.float64
    xd = x.double().numpy()[0, 0]
    want_q = xd / np.sqrt(np.sum(xd * xd))
    want_g = -np.log1p(np.exp(xd))
    want_b = 1.0 / (1.0 + np.exp(-0.69921875))   # bf16(0.7)
    np.testing.assert_allclose(qn[0, 0].numpy(), want_q, rtol=1e-15, atol=0)
    assert torch.equal(gn[0, 0], torch.from_numpy(want_g).to(torch.bfloat16))
    assert bn.item() == torch.tensor(want_b).to(torch.bfloat16).item()
    q2, k2, _, _ = oracle_mod.preprocess(x, x, x, b, qk_l2norm=False)
    assert q2.dtype == torch.bfloat16 and torch.equal(q2, x)


def test_preprocess_gate_scale_and_per_head(oracle_mod):
    """A per-head scale multiplies -softplus (scale 1 is the unscaled gate, scale 2
    doubles it); a per-head gate equals the per-channel gate with that value on
    every channel, and it turns KDA into the scalar-gate (GDN) recurrence: the
    decay of every key channel is the same."""
    import torch
    rng = np.random.default_rng(62)
    L, H, d = 7, 3, 5
    q = torch.from_numpy(rng.standard_normal((L, H, d)))
    k = torch.from_numpy(rng.standard_normal((L, H, d)))
    g1 = torch.from_numpy(rng.standard_normal((L, H)))
    b = torch.from_numpy(rng.standard_normal((L, H)))
    ones = np.ones(H)
    base = oracle_mod.preprocess(q, k, g1[..., None].expand(L, H, d).contiguous(), b)
    per_head = oracle_mod.preprocess(q, k, g1, b, gate_per_head=True)
    for x, y in zip(base, per_head):
        assert torch.equal(x, y)
    scaled1 = oracle_mod.preprocess(q, k, g1, b, gate_per_head=True, gate_scale=ones)
    assert torch.equal(scaled1[2], per_head[2])
    sc = np.array([2.0, 0.5, 0.0])
    scaled = oracle_mod.preprocess(q, k, g1, b, gate_per_head=True, gate_scale=sc)[2]
    np.testing.assert_allclose(scaled.numpy(), per_head[2].numpy() * sc[None, :, None],
                               rtol=1e-15, atol=0)
    assert torch.all(scaled[:, 2] == 0)  # scale 0: no decay
    # every channel of a head decays alike: the state's column norms keep their ratios
    # when beta = 0 (pure decay), as in the scalar-gate recurrence
    qn, kn, gn, _ = per_head
    v = rng.standard_normal((L, H, d))
    h0 = rng.standard_normal((1, H, d, d))
    _, hT = oracle_mod.recurrent(qn.numpy(), kn.numpy(), v, gn.numpy(), np.zeros((L, H)),
                                 cu_seqlens=np.array([0, L]), h0=h0)
    decay = np.exp(gn.numpy().sum(axis=0))          # [H, d], equal over d
    np.testing.assert_allclose(decay, decay[:, :1].repeat(d, axis=1), rtol=1e-15)
    np.testing.assert_allclose(hT[0], decay[:, :, None] * h0[0], rtol=1e-12, atol=1e-14)


# 7. gradients ----------------------------------------------------------------------
def _loss(oracle_mod, q, k, v, g, beta, h0, do, dhT, cu):
    o, hT = oracle_mod.recurrent(q, k, v, g, beta, cu_seqlens=cu, h0=h0)
    return float(np.sum(o * do) + np.sum(hT * dhT))


def test_grad_matches_central_differences(oracle_mod):
    """Every gradient of the autograd oracle equals the central difference of the
    C oracle's loss (a separate implementation of the forward) on a tiny packed
    batch with a start state and a final-state cotangent."""
    rng = np.random.default_rng(70)
    cu = np.array([0, 3, 3, 5])
    L, H, dk, dv = 5, 2, 3, 2
    q, k, v, g, beta = _rand_inputs(rng, L, H, dk, dv, decay=(0.4, 0.95))
    h0 = rng.standard_normal((3, H, dk, dv))
    do = rng.standard_normal((L, H, dv))
    dhT = rng.standard_normal((3, H, dk, dv))
    grads = oracle_mod.recurrent_grad(q, k, v, g, beta, do, cu_seqlens=cu, h0=h0, dhT=dhT)
    args = [q, k, v, g, beta, h0]
    eps = 1e-6
    for i, (x, gr) in enumerate(zip(args, grads)):
        assert gr.shape == x.shape
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = list(args), list(args)
            ap[i], am[i] = xp, xm
            fd[idx] = (_loss(oracle_mod, *ap, do, dhT, cu) - _loss(oracle_mod, *am, do, dhT, cu)) \
                / (2 * eps)
        np.testing.assert_allclose(gr, fd, rtol=1e-6, atol=1e-8)


def test_grad_single_token_closed_form(oracle_mod):
    """One token from a zero state: o = scale beta (k.q) v, so dv = scale beta (k.q) do,
    dq = scale beta (v.do) k, dk = scale beta (v.do) q, dbeta = scale (k.q)(v.do), and
    the gate has no effect (dg = 0)."""
    rng = np.random.default_rng(71)
    q, k, v, g, beta = _rand_inputs(rng, 1, 1, 4, 3)
    do = rng.standard_normal((1, 1, 3))
    s = 0.7
    dq, dk, dv, dg, db, dh0 = oracle_mod.recurrent_grad(q, k, v, g, beta, do,
                                                        cu_seqlens=np.array([0, 1]), scale=s)
    kq = float(k[0, 0] @ q[0, 0])
    vd = float(v[0, 0] @ do[0, 0])
    b = beta[0, 0]
    np.testing.assert_allclose(dv[0, 0], s * b * kq * do[0, 0], rtol=1e-13)
    np.testing.assert_allclose(dq[0, 0], s * b * vd * k[0, 0], rtol=1e-13)
    np.testing.assert_allclose(dk[0, 0], s * b * vd * q[0, 0], rtol=1e-13)
    np.testing.assert_allclose(db[0, 0], s * kq * vd, rtol=1e-13)
    assert np.all(dg == 0)
    # the start state's gradient: dh0 = diag(alpha) (I - beta k k^T) (scale q do^T)
    alpha = np.exp(g[0, 0])
    kk = k[0, 0]
    want = alpha[:, None] * ((np.eye(4) - b * np.outer(kk, kk)) @ (s * np.outer(q[0, 0], do[0, 0])))
    np.testing.assert_allclose(dh0[0, 0], want, rtol=1e-12, atol=1e-14)


def test_grad_is_linear_in_the_cotangents(oracle_mod):
    rng = np.random.default_rng(72)
    q, k, v, g, beta = _rand_inputs(rng, 6, 1, 3, 3, decay=(0.5, 1.0))
    h0 = rng.standard_normal((1, 1, 3, 3))
    do1, do2 = rng.standard_normal((2, 6, 1, 3))
    dh1, dh2 = rng.standard_normal((2, 1, 1, 3, 3))
    cu = np.array([0, 6])
    g1 = oracle_mod.recurrent_grad(q, k, v, g, beta, do1, cu_seqlens=cu, h0=h0, dhT=dh1)
    g2 = oracle_mod.recurrent_grad(q, k, v, g, beta, do2, cu_seqlens=cu, h0=h0, dhT=dh2)
    g12 = oracle_mod.recurrent_grad(q, k, v, g, beta, 2 * do1 - do2, cu_seqlens=cu, h0=h0,
                                    dhT=2 * dh1 - dh2)
    for a, b, c in zip(g1, g2, g12):
        np.testing.assert_allclose(c, 2 * a - b, rtol=1e-11, atol=1e-12)
