"""GPU parity on small shapes: the CUDA path through the C ABI against the
float64 oracle, element by element.  Shapes span several chunks and a ragged
tail, packed batches with empty and one-token sequences, both head sizes and
both input dtypes."""
import numpy as np
import pytest
import torch

import kda_inputs
from _util import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.float32: TOL_F32, torch.bfloat16: TOL_BF16}


def _check_fwd(kda, oracle_mod, x, dtype, out_dtype=torch.float32):
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                    out_dtype=out_dtype)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    tol = TOL[dtype]
    if out_dtype == torch.bfloat16:  # the output rounding itself: half a bf16 ulp of |o|
        d = np.abs(o.float().cpu().numpy() - o_ref)
        bound = tol * np.sqrt(np.mean(o_ref ** 2)) + np.abs(o_ref) * 2.0 ** -8
        assert np.all(d <= bound)
    else:
        assert eo <= tol, f"o: {eo:.3e} > {tol}"
    assert eh <= tol, f"hT: {eh:.3e} > {tol}"
    return eo, eh


def test_tiny_fp32_workload(kda, oracle_mod):
    """B=1, T=256, H=2, d=64, float32 in and out, h0 = 0."""
    x = kda_inputs.workload(0, device=DEV)
    _check_fwd(kda, oracle_mod, x, torch.float32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_fixed_length(kda, oracle_mod, dtype, d, T):
    x = kda_inputs.fixed(2, T, 3, d, dtype=dtype, device=DEV, seed=T * 7 + d, h0_std=0.1)
    _check_fwd(kda, oracle_mod, x, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_packed_varlen(kda, oracle_mod, dtype, d):
    x = kda_inputs.packed([1, 2, 64, 0, 65, 130, 200], 2, d, dtype=dtype, device=DEV,
                          seed=11 + d, h0_std=0.1)
    _check_fwd(kda, oracle_mod, x, dtype)


def test_zero_start_state_and_no_final_state(kda, oracle_mod):
    x = kda_inputs.fixed(1, 100, 2, 128, dtype=torch.bfloat16, device=DEV, seed=5)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, output_final_state=False)
    assert hT is None
    o_ref, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta)
    assert rel_err(o, o_ref) <= TOL_BF16


def test_bf16_output(kda, oracle_mod):
    x = kda_inputs.fixed(1, 130, 2, 128, dtype=torch.bfloat16, device=DEV, seed=6, h0_std=0.1)
    _check_fwd(kda, oracle_mod, x, torch.bfloat16, out_dtype=torch.bfloat16)


def test_empty_batch_writes_start_state(kda, oracle_mod):
    x = kda_inputs.packed([0, 0, 0], 2, 128, dtype=torch.bfloat16, device=DEV, seed=3,
                          h0_std=0.1)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(hT, x.h0)


def test_repeatable_bit_for_bit(kda):
    x = kda_inputs.packed([90, 300, 17], 4, 128, dtype=torch.bfloat16, device=DEV, seed=21,
                          h0_std=0.1)
    o1, h1 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    o2, h2 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_bad_cu_seqlens_is_reported_not_executed(kda):
    x = kda_inputs.packed([50, 50], 2, 128, dtype=torch.bfloat16, device=DEV, seed=4)
    bad = torch.tensor([0, 60, 40], dtype=torch.int32, device=DEV)  # decreasing
    ws = kda.new_workspace(kda.make_shape(x.q, x.v, packed_seqs=2), DEV)
    o = torch.full((1, 100, 2, 128), 7.0, device=DEV)
    kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=bad, out=o, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_ERR_BAD_SEQLENS
    assert torch.all(o == 7.0)  # nothing was written
    assert kda.read_device_status(ws) == kda.KDA_OK  # reading clears the latch
    short = torch.tensor([0, 50, 90], dtype=torch.int32, device=DEV)  # does not end at T
    kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=short, out=o, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_ERR_BAD_SEQLENS


# prefix-cache checkpoints ------------------------------------------------------------

def _ckpt_refs(oracle_mod, x, seqs, interval):
    """Oracle states after each `interval` tokens of each sequence, built one
    interval at a time.  seqs: (batch index, first token, length, h0 index or None)."""
    refs = []
    for b, t0, ln, hi in seqs:
        state = None if hi is None else x.h0[hi:hi + 1].contiguous()
        for j in range(ln // interval):
            sl = lambda t: t[b:b + 1, t0 + j * interval:t0 + (j + 1) * interval].contiguous()
            _, h = oracle_mod.recurrent(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), h0=state)
            refs.append(h[0])
            state = torch.from_numpy(h).float()
    return refs


def _check_ckpts(ck, refs, tol):
    assert ck.shape[0] == len(refs)
    for r, ref in enumerate(refs):
        assert rel_err(ck[r], ref) <= tol, f"checkpoint row {r}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_checkpoints_fixed_length(kda, oracle_mod, dtype, d):
    """B=2, T=1100: states after 512 and 1024 tokens of each sequence, with o and hT
    unchanged from kda_fwd."""
    x = kda_inputs.fixed(2, 1100, 2, d, dtype=dtype, device=DEV, seed=31 + d, h0_std=0.1)
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, interval=512)
    o2, h2 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    assert off.tolist() == [0, 2, 4]
    assert torch.equal(o, o2) and torch.equal(hT, h2)
    _check_ckpts(ck, _ckpt_refs(oracle_mod, x, [(0, 0, 1100, 0), (1, 0, 1100, 1)], 512),
                 TOL[dtype])


@pytest.mark.parametrize("dtype,d,interval", [(torch.bfloat16, 128, 512), (torch.bfloat16, 128, 64),
                                              (torch.float32, 64, 64), (torch.float32, 128, 128)],
                         ids=["bf16-512", "bf16-64", "f32-d64-64", "f32-d128-128"])
def test_checkpoints_packed(kda, oracle_mod, dtype, d, interval):
    """Packed lengths with empty, short and exact-multiple sequences: each sequence
    checkpoints from its own start; row offsets follow the lengths."""
    lens = [600, 1024, 100, 0, 1537, 64]
    x = kda_inputs.packed(lens, 2, d, dtype=dtype, device=DEV, seed=37, h0_std=0.1)
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                         h0=x.h0, interval=interval)
    torch.cuda.synchronize()
    starts = [sum(lens[:i]) for i in range(len(lens))]
    assert off.tolist() == [sum(l // interval for l in lens[:i]) for i in range(len(lens) + 1)]
    refs = _ckpt_refs(oracle_mod, x, [(0, starts[i], lens[i], i) for i in range(len(lens))],
                      interval)
    _check_ckpts(ck, refs, TOL[dtype])


def test_checkpoints_long_chain_split(kda, oracle_mod):
    """The segment split computes the outputs of each segment from its scanned start
    state; checkpoints are taken there too, at positions relative to the sequence."""
    x = kda_inputs.fixed(1, 64 * 257 + 37, 2, 128, dtype=torch.bfloat16, device=DEV, seed=41,
                         h0_std=0.1)
    assert kda.workspace_size(kda.make_shape(x.q, x.v)) > 256  # the split plan is active
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, interval=512)
    torch.cuda.synchronize()
    _check_ckpts(ck, _ckpt_refs(oracle_mod, x, [(0, 0, x.q.shape[1], 0)], 512), TOL_BF16)


def test_checkpoints_bad_offsets_are_reported(kda):
    """Offsets that disagree with the lengths are latched; that sequence writes no
    checkpoint, the others do, and o is unaffected."""
    import ctypes
    lens = [600, 1024]
    x = kda_inputs.packed(lens, 2, 128, dtype=torch.bfloat16, device=DEV, seed=43)
    shape = kda.make_shape(x.q, x.v, packed_seqs=2)
    ws = kda.new_workspace(shape, DEV)
    o = torch.empty(1, sum(lens), 2, 128, device=DEV)
    ck = torch.full((4, 2, 128, 128), float("nan"), device=DEV)
    offs = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)  # sequence 0 has 1, not 2
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = kda.load().kda_fwd_checkpoints(
        ctypes.byref(shape), vp(x.q), vp(x.k), vp(x.v), vp(x.g), vp(x.beta), vp(x.cu_seqlens),
        None, vp(o), None, 512, vp(ck), vp(offs), 4, vp(ws), ws.numel(), None)
    assert rc == kda.KDA_OK
    assert kda.read_device_status(ws) == kda.KDA_ERR_INVALID_ARG
    o_ref, _ = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.isnan(ck[:2]).all()     # sequence 0: refused, its rows untouched
    assert torch.isfinite(ck[2:]).all()  # sequence 1: rows 2 and 3 written


# decode ---------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T_step", [1, 3, 8])
def test_decode(kda, oracle_mod, dtype, d, T_step):
    x = kda_inputs.decode_pool(num_seqs=5, H=3, d=d, T_step=T_step, dtype=dtype, device=DEV,
                               seed=100 + T_step)
    state = x.h0.clone()
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    tol = TOL[dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(state, h_ref) <= tol


@pytest.mark.parametrize("T_step", [2, 4, 5, 6, 7])
def test_decode_every_step_count(kda, oracle_mod, T_step):
    """d=128 steps of every other token count (the staging of a step's inputs
    covers 1 to 4 rounds of the block): each matches the oracle at the float32
    bound, and the same step taken one token at a time agrees to 1e-5."""
    x = kda_inputs.decode_pool(num_seqs=6, H=4, d=128, T_step=T_step, dtype=torch.float32,
                               device=DEV, seed=400 + T_step)
    state = x.h0.clone()
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    s1 = x.h0.clone()
    o1 = torch.cat([kda.decode(x.q[:, t:t + 1].contiguous(), x.k[:, t:t + 1].contiguous(),
                               x.v[:, t:t + 1].contiguous(), x.g[:, t:t + 1].contiguous(),
                               x.beta[:, t:t + 1].contiguous(), s1) for t in range(T_step)],
                   dim=1)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_F32
    assert rel_err(state, h_ref) <= TOL_F32
    assert rel_err(o, o1.double().cpu().numpy()) <= 1e-5
    assert rel_err(state, s1.double().cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("d", [64, 128])
def test_decode_extreme_gates(kda, oracle_mod, d):
    """Gates strong enough that the product of alpha over the step underflows
    float32 (head 0: g = -25 on a few channels; head 1: alpha = 0 on one channel)
    take the explicit per-token decay; head 2 keeps ordinary gates.  All match
    the oracle."""
    x = kda_inputs.decode_pool(num_seqs=4, H=3, d=d, T_step=8, dtype=torch.float32, device=DEV,
                               seed=321)
    g = x.g.clone()
    g[:, :, 0, :5] = -25.0
    g[:, :, 1, 7] = float("-inf")
    state = x.h0.clone()
    o = kda.decode(x.q, x.k, x.v, g, x.beta, state)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_F32
    assert rel_err(state, h_ref) <= TOL_F32


# decode with commit counts (speculative-decode verification and replay) ---------------

def _commit_refs(oracle_mod, x, counts):
    """Oracle state after each sequence's first counts[n] tokens (h0 when 0)."""
    refs = []
    for n, c in enumerate(counts):
        if c == 0:
            refs.append(x.h0[n].double().cpu().numpy())
            continue
        sl = lambda t: t[n:n + 1, :c].contiguous()
        _, h = oracle_mod.recurrent(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta),
                                    h0=x.h0[n:n + 1].contiguous())
        refs.append(h[0])
    return refs


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_commit_counts(kda, oracle_mod, dtype, d):
    """Every token produces its output; the state kept is the one after the
    accepted prefix (0 = verification only, T_step = plain decode)."""
    x = kda_inputs.decode_pool(num_seqs=6, H=3, d=d, T_step=8, dtype=dtype, device=DEV, seed=91)
    counts = [0, 1, 3, 5, 8, 8]
    state = x.h0.clone()
    o = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                          torch.tensor(counts, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    o_ref, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    tol = TOL[dtype]
    assert rel_err(o, o_ref) <= tol
    for n, ref in enumerate(_commit_refs(oracle_mod, x, counts)):
        if counts[n] == 0:
            assert torch.equal(state[n], x.h0[n])  # untouched
        else:
            assert rel_err(state[n], ref) <= tol


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.bfloat16, 128)],
                         ids=["f32-d64", "bf16-d128"])
def test_decode_commit_many_chains(kda, oracle_mod, dtype, d):
    """640 (sequence, head) chains, more than the device holds CTAs at once (two
    per SM), so CTAs of later waves reuse the SMs.  The commit counts cycle
    through 0..8, so neighbouring chains keep states after different prefixes."""
    num_seqs, H = 160, 4
    x = kda_inputs.decode_pool(num_seqs=num_seqs, H=H, d=d, T_step=8, dtype=dtype, device=DEV,
                               seed=93)
    counts = [n % 9 for n in range(num_seqs)]
    state = x.h0.clone()
    o = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                          torch.tensor(counts, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    o_ref, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    tol = TOL[dtype]
    assert rel_err(o, o_ref) <= tol
    for n, ref in enumerate(_commit_refs(oracle_mod, x, counts)):
        if counts[n] == 0:
            assert torch.equal(state[n], x.h0[n])
        else:
            assert rel_err(state[n], ref) <= tol


@pytest.mark.parametrize("T_step", [2, 5, 8])
def test_decode_commit_every_count(kda, oracle_mod, T_step):
    """Commit counts 0..T_step on one batch (bf16 inputs, bf16 outputs): outputs of
    all tokens, and each sequence's kept state after its accepted prefix."""
    counts = list(range(T_step + 1))
    x = kda_inputs.decode_pool(num_seqs=len(counts), H=2, d=128, T_step=T_step,
                               dtype=torch.bfloat16, device=DEV, seed=500 + T_step)
    state = x.h0.clone()
    o = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                          torch.tensor(counts, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    o_ref, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    for n, ref in enumerate(_commit_refs(oracle_mod, x, counts)):
        if counts[n] == 0:
            assert torch.equal(state[n], x.h0[n])
        else:
            assert rel_err(state[n], ref) <= TOL_BF16


def test_decode_commit_verify_then_replay(kda):
    """The two-call flow: verify T_step drafts without committing, then replay the
    same cached inputs committing the accepted prefix.  The kept state equals
    kda_decode over that prefix; the verification outputs equal kda_decode's."""
    x = kda_inputs.decode_pool(num_seqs=4, H=2, d=128, T_step=6, dtype=torch.bfloat16,
                               device=DEV, seed=92)
    accepted = 4
    state = x.h0.clone()
    zeros = torch.zeros(4, dtype=torch.int32, device=DEV)
    o_verify = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state, zeros)
    assert torch.equal(state, x.h0)
    none = kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                             torch.full((4,), accepted, dtype=torch.int32, device=DEV),
                             want_out=False)
    assert none is None
    ref_state = x.h0.clone()
    pre = lambda t: t[:, :accepted].contiguous()
    kda.decode(pre(x.q), pre(x.k), pre(x.v), pre(x.g), pre(x.beta), ref_state)
    full_state = x.h0.clone()
    o_full = kda.decode(x.q, x.k, x.v, x.g, x.beta, full_state)
    torch.cuda.synchronize()
    assert rel_err(state, ref_state.double().cpu().numpy()) <= 1e-5
    assert rel_err(o_verify, o_full.double().cpu().numpy()) <= 1e-6


def test_decode_commit_bad_count_is_reported(kda):
    """A count outside 0..T_step is latched; that sequence keeps its state and the
    others commit normally."""
    x = kda_inputs.decode_pool(num_seqs=3, H=2, d=64, T_step=4, dtype=torch.float32,
                               device=DEV, seed=93)
    state = x.h0.clone()
    ref = x.h0.clone()
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    kda.decode_commit(x.q, x.k, x.v, x.g, x.beta, state,
                      torch.tensor([4, 5, -1], dtype=torch.int32, device=DEV), workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_ERR_INVALID_ARG
    kda.decode(x.q[:1].contiguous(), x.k[:1].contiguous(), x.v[:1].contiguous(),
               x.g[:1].contiguous(), x.beta[:1].contiguous(), ref[:1])
    torch.cuda.synchronize()
    assert rel_err(state[0], ref[0].double().cpu().numpy()) <= 1e-6
    assert torch.equal(state[1:], x.h0[1:])


def test_decode_replay_equals_single_steps_and_prefill(kda):
    """One 8-token replay step == eight 1-token steps == prefill from the same state."""
    x = kda_inputs.decode_pool(num_seqs=3, H=2, d=128, T_step=8, dtype=torch.float32,
                               device=DEV, seed=55)
    s8 = x.h0.clone()
    o8 = kda.decode(x.q, x.k, x.v, x.g, x.beta, s8)
    s1 = x.h0.clone()
    o1 = torch.cat([kda.decode(x.q[:, t:t + 1].contiguous(), x.k[:, t:t + 1].contiguous(),
                               x.v[:, t:t + 1].contiguous(), x.g[:, t:t + 1].contiguous(),
                               x.beta[:, t:t + 1].contiguous(), s1) for t in range(8)], dim=1)
    op, hp = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    ref = o8.double().cpu().numpy()
    assert rel_err(o1, ref) <= 1e-5 and rel_err(s1, s8.double().cpu().numpy()) <= 1e-5
    assert rel_err(op, ref) <= 1e-4 and rel_err(hp, s8.double().cpu().numpy()) <= 1e-4


def test_long_chain_split_matches_oracle_and_unsplit_run(kda, oracle_mod):
    """Two very long chains: the segment split (4 segments joined by their state
    maps) is used with the full workspace and skipped with the minimum one; both
    match the oracle."""
    x = kda_inputs.fixed(1, 64 * 257 + 37, 2, 128, dtype=torch.bfloat16, device=DEV, seed=77,
                         h0_std=0.1)
    shape = kda.make_shape(x.q, x.v)
    assert kda.workspace_size(shape) > 256  # the split plan is active for this shape
    o_s, h_s = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    small = torch.empty(256, dtype=torch.uint8, device=DEV)
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, workspace=small)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    for o, h in ((o_s, h_s), (o_u, h_u)):
        assert rel_err(o, o_ref) <= TOL_BF16
        assert rel_err(h, h_ref) <= TOL_BF16


def test_long_chain_split_many_segments(kda, oracle_mod):
    """One chain of 2561 chunks (ragged last chunk): the plan cuts it into 40
    segments (the first of 65 chunks, the others of 64), composed by 39 steps of the
    segment scan; split and unsplit runs both match the oracle."""
    x = kda_inputs.fixed(1, 64 * 64 * 40 + 17, 1, 128, dtype=torch.bfloat16, device=DEV,
                         seed=78, h0_std=0.1)
    shape = kda.make_shape(x.q, x.v)
    assert kda.workspace_size(shape) == 256 + (3 * 40 - 2) * 128 * 128 * 4
    o_s, h_s = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    small = torch.empty(256, dtype=torch.uint8, device=DEV)
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, workspace=small)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    for o, h in ((o_s, h_s), (o_u, h_u)):
        assert rel_err(o, o_ref) <= TOL_BF16
        assert rel_err(h, h_ref) <= TOL_BF16


def test_long_chain_split_longer_first_segment(kda, oracle_mod):
    """32 chains of 384 chunks with start states: the plan makes segment 0 twice as
    long as the other four (128 and 64 chunks), since it runs once, in the first
    launch, beside the 192 transition items of the others.  Three sampled heads
    match the oracle; every head matches the unsplit run."""
    x = kda_inputs.fixed(1, 64 * 384, 32, 128, dtype=torch.bfloat16, device=DEV, seed=79,
                         h0_std=0.1)
    shape = kda.make_shape(x.q, x.v)
    assert kda.workspace_size(shape) == 256 + 32 * (3 * 5 - 2) * 128 * 128 * 4
    o_s, h_s = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    small = torch.empty(256, dtype=torch.uint8, device=DEV)
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, workspace=small)
    torch.cuda.synchronize()
    assert rel_err(o_s, o_u.double().cpu().numpy()) <= 1e-3
    assert rel_err(h_s, h_u.double().cpu().numpy()) <= 1e-3
    heads = [0, 17, 31]
    sub = lambda t: t[:, :, heads].contiguous().cpu()
    o_ref, h_ref = oracle_mod.recurrent(*(sub(t) for t in (x.q, x.k, x.v, x.g, x.beta)),
                                        h0=x.h0[:, heads].contiguous().cpu())
    assert rel_err(o_s[:, :, heads], o_ref) <= TOL_BF16
    assert rel_err(h_s[:, heads], h_ref) <= TOL_BF16


def test_checkpoints_longer_first_segment(kda, oracle_mod):
    """The split of 32 chains of 384 chunks (segment 0 of 128 chunks, four of 64) with
    a checkpoint every 2048 tokens: those inside and at the end of segment 0 come from
    the first launch, the others from the second, at positions counted from the
    sequence's start.  Three sampled heads match the oracle's prefix states, and o
    and hT equal kda_fwd's."""
    x = kda_inputs.fixed(1, 64 * 384, 32, 128, dtype=torch.bfloat16, device=DEV, seed=81,
                         h0_std=0.1)
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, interval=2048)
    o2, h2 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    assert off.tolist() == [0, 12]
    assert torch.equal(o, o2) and torch.equal(hT, h2)
    heads = [0, 17, 31]
    q, k, v, g, b = (t[:, :, heads].contiguous().cpu() for t in (x.q, x.k, x.v, x.g, x.beta))
    state = x.h0[:, heads].contiguous().cpu()
    for r in range(12):
        sl = lambda t: t[:, r * 2048:(r + 1) * 2048].contiguous()
        _, h = oracle_mod.recurrent(sl(q), sl(k), sl(v), sl(g), sl(b), h0=state)
        assert rel_err(ck[r][heads], h[0]) <= TOL_BF16, f"checkpoint {r}"
        state = torch.from_numpy(h).float()


def test_bounded_wait_runs_out_and_is_reported(kda, oracle_mod):
    """A device wait that can never complete gives up after its budget, latches
    KDA_ERR_DEVICE_TIMEOUT, and leaves the context usable for the next call."""
    import ctypes
    L = kda.load()
    L.kda_selftest_bounded_wait.restype = ctypes.c_int
    L.kda_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    rc = L.kda_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == kda.KDA_OK
    assert kda.read_device_status(ws) == kda.KDA_ERR_DEVICE_TIMEOUT
    x = kda_inputs.fixed(1, 70, 2, 128, dtype=torch.bfloat16, device=DEV, seed=8)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta)
    torch.cuda.synchronize()
    o_ref, _ = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta)
    assert rel_err(o, o_ref) <= TOL_BF16


# strong gates: decay beyond the range one chunk's factorisation holds -----------------
# The gate is per channel in (0, 1) ("Kimi K3 NPU Training", section 模型结构), so any
# log(alpha) <= 0 is valid, alpha = 0 (g = -inf) included.  The bf16 tensor-core path
# runs a chunk whose in-chunk decay span leaves its factor range token by token; the
# float32 path takes exponentials of differences.  Both must match the oracle.

def _strong_gates(g, pattern):
    """g (token axis 1) with a few channels pushed far past the workload's range."""
    g = g.clone()
    if pattern == "g-3":        # e^-3 per token on four channels: 192 nats per chunk
        g[..., 5:9] = -3.0
    elif pattern == "g-25":     # e^-25 per token on two channels
        g[..., 40:42] = -25.0
    elif pattern == "alpha0":   # alpha = 0 at two tokens of one channel (chunks 1 and 2)
        g[:, 70, :, 3] = float("-inf")
        g[:, 150, :, 3] = float("-inf")
    elif pattern == "burst":    # every channel at -30 for four tokens (chunk 0 only)
        g[:, 40:44] = -30.0
    return g


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 128),
                                     (torch.float32, 64), (torch.bfloat16, 64)],
                         ids=["bf16-128", "f32-128", "f32-64", "bf16-64"])
@pytest.mark.parametrize("pattern", ["g-3", "g-25", "alpha0", "burst"])
def test_strong_gates_match_oracle(kda, oracle_mod, dtype, d, pattern):
    x = kda_inputs.fixed(2, 200, 2, d, dtype=dtype, device=DEV, seed=900 + d, h0_std=0.1)
    x.g = _strong_gates(x.g, pattern)
    ws = kda.new_workspace(kda.make_shape(x.q, x.v), DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_OK
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["o32", "o16"])
def test_strong_gates_packed(kda, oracle_mod, dtype, out_dtype):
    """Packed sequences (an empty and a one-token one included) with alpha = 0, -25 and
    -4 runs crossing sequence boundaries, beside chunks of ordinary gates."""
    x = kda_inputs.packed([1, 64, 0, 130, 77, 200], 2, 128, dtype=dtype, device=DEV, seed=910,
                          h0_std=0.1)
    g = x.g.clone()
    g[:, 60:70, :, 7] = float("-inf")
    g[:, 100:110, :, :4] = -25.0
    g[:, 300:330, :, 50:60] = -4.0
    x.g = g
    _check_fwd(kda, oracle_mod, x, dtype, out_dtype=out_dtype)


def test_strong_gates_long_chain_split(kda, oracle_mod):
    """A chain long enough for the segment split, with strong decay inside some
    segments: the transition passes (identity start, v = 0) and the output pass run
    those chunks token by token too."""
    T = 64 * 257 + 37
    x = kda_inputs.fixed(1, T, 2, 128, dtype=torch.bfloat16, device=DEV, seed=920, h0_std=0.1)
    g = x.g.clone()
    g[:, 5000:9000, :, 5:9] = -3.0
    g[:, 12000, :, 3] = float("-inf")
    g[:, 15000:15004] = -30.0
    x.g = g
    shape = kda.make_shape(x.q, x.v)
    assert kda.workspace_size(shape) > 256  # the split is planned
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_strong_gates_checkpoints(kda, oracle_mod, dtype):
    """Checkpoints written by chunks that ran token by token."""
    x = kda_inputs.fixed(2, 200, 2, 128, dtype=dtype, device=DEV, seed=930, h0_std=0.1)
    g = _strong_gates(x.g, "alpha0")
    g[:, :64, :, 40:42] = -25.0
    x.g = g
    o, hT, ck, _ = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, interval=64, h0=x.h0)
    torch.cuda.synchronize()
    refs = _ckpt_refs(oracle_mod, x, [(b, 0, 200, b) for b in range(2)], 64)
    _check_ckpts(ck, refs, TOL[dtype])
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("T", [200, 64 * 257 + 37], ids=["chain", "segment-split"])
def test_final_state_may_alias_start_state(kda, oracle_mod, T):
    """hT written into the h0 buffer (in place) gives the same result as separate buffers,
    both for whole chains and for long chains cut into segments."""
    x = kda_inputs.fixed(1, T, 2, 128, dtype=torch.bfloat16, device=DEV, seed=31, h0_std=0.1)
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    state = x.h0.clone()
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=state, hT=state)
    torch.cuda.synchronize()
    assert hT.data_ptr() == state.data_ptr()
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(state, h_ref) <= TOL_BF16


def test_nondefault_scale_single_head_bf16_output_packed(kda, oracle_mod):
    x = kda_inputs.packed([300, 1, 77], 1, 128, dtype=torch.bfloat16, device=DEV, seed=41,
                          h0_std=0.1)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0, scale=0.37,
                    out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0, scale=0.37)
    d = np.abs(o.float().cpu().numpy() - o_ref)
    assert np.all(d <= TOL_BF16 * np.sqrt(np.mean(o_ref ** 2)) + np.abs(o_ref) * 2.0 ** -8)
    assert rel_err(hT, h_ref) <= TOL_BF16


# one batch partitioned across ranks, the shards run one after another on one GPU ------

@pytest.mark.parametrize("by", ["sequence", "head"])
def test_sharded_batch_equals_unsharded(kda, by):
    """Every chain is independent, so a batch computed shard by shard (the sequence
    partition of 3 ranks, longest first, or the head partition) and put back in place
    equals the whole batch's result bit for bit."""
    from kda_delta_rule_fwd_gb300 import shard
    lens = [700, 0, 65, 1, 300, 64, 1030, 9]
    x = kda_inputs.packed(lens, 5, 128, dtype=torch.bfloat16, device=DEV, seed=950,
                          h0_std=0.1)
    o_ref, h_ref = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
    if by == "sequence":
        shards = [shard.take_sequences(x, idx) for idx in shard.lpt_by_sequence(lens, 3)]
    else:
        shards = [shard.take_heads(x, h0, h1) for h0, h1 in shard.heads_by_rank(5, 3)]
    outs, states = [], []
    for s in shards:
        o, h = kda.fwd(s.q, s.k, s.v, s.g, s.beta, cu_seqlens=s.cu_seqlens, h0=s.h0)
        outs.append(o)
        states.append(h)
    torch.cuda.synchronize()
    if by == "sequence":
        o, h = shard.place_sequences(x.q.shape[1], x.cu_seqlens.tolist(), shards, outs, states)
    else:
        o, h = torch.cat(outs, dim=2), torch.cat(states, dim=1)
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)


# long sequences inside packed batches: the device-planned segment split ------------

def _packed_plan(ws, N):
    """The plan the device wrote into the workspace after the order list:
    (transition items, split sequences, output items, segment length in chunks)."""
    at = 256 + (N + 63) // 64 * 256
    return ws[at:at + 16].view(torch.int32).tolist()


def test_packed_long_chain_split(kda, oracle_mod):
    """[2^18, 300, 1, 5000] tokens, H=2: the planner cuts the 4096-chunk sequence
    into 63 segments, segment 0 of 128 chunks (run from the start state with its
    outputs in the transition pass) and the others of 64, and leaves the others
    whole: 62 transition entries, 62 + 3 output items.  The split run and a run
    without the split (minimum workspace) both match the oracle."""
    lens = [1 << 18, 300, 1, 5000]
    x = kda_inputs.packed(lens, 2, 128, dtype=torch.bfloat16, device=DEV, seed=960, h0_std=0.1)
    shape = kda.make_shape(x.q, x.v, packed_seqs=4)
    ws = kda.new_workspace(shape, DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_OK
    assert _packed_plan(ws, 4) == [62, 1, 62 + 3, 64]
    small = torch.empty(512, dtype=torch.uint8, device=DEV)
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                       workspace=small)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    for oo, hh in ((o, hT), (o_u, h_u)):
        assert rel_err(oo, o_ref) <= TOL_BF16
        assert rel_err(hh, h_ref) <= TOL_BF16


def test_packed_split_longer_first_segments(kda, oracle_mod):
    """[65536, 40000, 9000] tokens, H=4, start states: the planner (S = 64 chunks,
    segment 0 twice as long) cuts the first two sequences into 15 segments of 64
    chunks after a segment 0 of 128, and 8 of 70 after one of 135 (their segment-0
    items run first, the longer first), while the third, too short for that, gets 2
    equal segments of 71: 14 + 7 + 1 transition entries and as many output items.
    Every head matches the oracle, and the run without the split."""
    lens = [65536, 40000, 9000]
    x = kda_inputs.packed(lens, 4, 128, dtype=torch.bfloat16, device=DEV, seed=965, h0_std=0.1)
    shape = kda.make_shape(x.q, x.v, packed_seqs=3)
    ws = kda.new_workspace(shape, DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_OK
    assert _packed_plan(ws, 3) == [22, 3, 22, 64]
    small = torch.empty(512, dtype=torch.uint8, device=DEV)
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                       workspace=small)
    torch.cuda.synchronize()
    assert rel_err(o, o_u.double().cpu().numpy()) <= 1e-3
    assert rel_err(hT, h_u.double().cpu().numpy()) <= 1e-3
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_packed_split_many_sequences(kda, oracle_mod):
    """600 packed sequences, one of 20000 tokens and 599 of 1 to 50: past 512
    sequences the planner costs its candidates one by one with block reductions
    (below, a thread costs each candidate over every sequence); it splits the long
    sequence and leaves the others whole.  Every element matches the oracle."""
    lens = [20000] + [1 + (i * 37) % 50 for i in range(599)]
    x = kda_inputs.packed(lens, 2, 128, dtype=torch.bfloat16, device=DEV, seed=975, h0_std=0.1)
    shape = kda.make_shape(x.q, x.v, packed_seqs=len(lens))
    ws = kda.new_workspace(shape, DEV)
    o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0, workspace=ws)
    assert kda.read_device_status(ws) == kda.KDA_OK
    n_trans, n_split, n_out, S = _packed_plan(ws, len(lens))
    assert n_split == 1 and S >= 64 and n_out == n_trans + 599
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_packed_split_mixed_with_checkpoints(kda, oracle_mod):
    """Two split sequences of different segment lengths, an empty and short ones,
    strong gates inside a split sequence (token path in the transition passes),
    checkpoints every 512 tokens at positions relative to each sequence."""
    lens = [20000, 0, 9000, 64, 129]
    x = kda_inputs.packed(lens, 2, 128, dtype=torch.bfloat16, device=DEV, seed=970, h0_std=0.1)
    g = x.g.clone()
    g[:, 7000:7100, :, 5:9] = -25.0
    g[:, 12345, :, 3] = float("-inf")
    x.g = g
    shape = kda.make_shape(x.q, x.v, packed_seqs=5)
    ws = kda.new_workspace(shape, DEV)
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, interval=512,
                                         cu_seqlens=x.cu_seqlens, h0=x.h0, workspace=ws)
    torch.cuda.synchronize()
    n_trans, n_split, n_out, S = _packed_plan(ws, 5)
    assert n_split == 2 and S >= 64
    starts = [sum(lens[:i]) for i in range(len(lens))]
    refs = _ckpt_refs(oracle_mod, x, [(0, starts[i], lens[i], i) for i in range(len(lens))], 512)
    _check_ckpts(ck, refs, TOL_BF16)
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens,
                                        h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_packed_split_fused_preprocessing(kda, oracle_mod):
    """The packed split under the fused preprocessing (raw q, k, gate and beta)."""
    lens = [40000, 300]
    cu = torch.tensor([0, 40000, 40300], dtype=torch.int32)
    x = kda_inputs.draw_raw((1, 40300), 2, 128, 128, device=DEV, seed=980, num_states=2,
                            h0_std=0.1)
    x.cu_seqlens = cu.to(DEV)
    shape = kda.make_shape(x.q, x.v, packed_seqs=2)
    ws = kda.new_workspace(shape, DEV)
    o, hT = kda.fwd_preproc(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0,
                            workspace=ws)
    torch.cuda.synchronize()
    assert _packed_plan(ws, 2)[1] == 1
    fq, fk, fg, fb = oracle_mod.preprocess(x.q, x.k, x.g, x.beta)
    o_ref, h_ref = oracle_mod.recurrent(fq, fk, x.v, fg, fb, cu_seqlens=x.cu_seqlens, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


# more (sequence, head) chains than SMs: persistent CTAs take several items each -------

def test_fixed_length_more_chains_than_sms(kda, oracle_mod):
    """B=6, H=32: 192 chains on at most 152 CTAs, each taking items in turn from the
    launch's counter; plain, then with checkpoints every 64 tokens."""
    x = kda_inputs.fixed(6, 130, 32, 128, dtype=torch.bfloat16, device=DEV, seed=990,
                         h0_std=0.1)
    _check_fwd(kda, oracle_mod, x, torch.bfloat16)
    o, hT, ck, off = kda.fwd_checkpoints(x.q, x.k, x.v, x.g, x.beta, interval=64, h0=x.h0)
    o2, h2 = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(hT, h2)
    refs = _ckpt_refs(oracle_mod, x, [(b, 0, 130, b) for b in range(6)], 64)
    _check_ckpts(ck, refs, TOL_BF16)
