"""kda_fwd_noalloc: the prefill entry point for callers that cannot allocate
device memory (their memory is planned in full by a host framework, or their
bindings cannot reach a device allocator).  It keeps its scratch in a fixed
array inside the library instead of a caller workspace.  Checked through the
C ABI against kda_fwd, bit for bit, on two calls in a row, since every call
reuses the same array."""
import ctypes

import pytest
import torch

import kda_inputs
from _util import TOL_BF16, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _entry(kda):
    f = kda.load().kda_fwd_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    # shape, q, k, v, g, beta, cu_seqlens, h0, out, hT, status_out, stream
    f.argtypes = [ctypes.POINTER(kda.Shape)] + [vp] * 11
    return f


def _call(kda, f, x, status):
    N = x.cu_seqlens.numel() - 1 if x.cu_seqlens is not None else x.q.shape[0]
    shape = kda.make_shape(x.q, x.v, packed_seqs=None if x.cu_seqlens is None else N)
    B, T, H, d = x.q.shape
    o = torch.full((B, T, H, d), float("nan"), device=DEV)
    hT = torch.full((N, H, d, d), float("nan"), device=DEV)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = f(ctypes.byref(shape), p(x.q), p(x.k), p(x.v), p(x.g), p(x.beta), p(x.cu_seqlens),
           p(x.h0), p(o), p(hT), p(status),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, hT


@pytest.mark.parametrize("packed", [True, False], ids=["packed", "fixed"])
def test_noalloc_matches_kda_fwd_on_two_calls(kda, packed):
    """Two calls in a row: each equals kda_fwd bit for bit (the same kernels run;
    only the scratch's home differs), although the second finds the first's
    contents in the shared array."""
    f = _entry(kda)
    status = torch.full((1,), 12345, dtype=torch.int32, device=DEV)
    for call in range(2):
        if packed:
            x = kda_inputs.packed([70, 0, 130, 5 + call, 64], 4, 128, dtype=torch.bfloat16,
                                  device=DEV, seed=40 + call, h0_std=0.1)
        else:
            x = kda_inputs.fixed(2, 150 + call, 3, 128, dtype=torch.bfloat16, device=DEV,
                                 seed=50 + call, h0_std=0.1)
        ref_o, ref_h = kda.fwd(x.q, x.k, x.v, x.g, x.beta, cu_seqlens=x.cu_seqlens, h0=x.h0)
        status.fill_(12345)
        rc, o, hT = _call(kda, f, x, status)
        torch.cuda.synchronize()
        assert rc == kda.KDA_OK, kda.status_string(rc)
        assert int(status.item()) == kda.KDA_OK
        assert torch.equal(o, ref_o)
        assert torch.equal(hT, ref_h)


def test_noalloc_fixed_length_ignores_num_seqs(kda):
    """num_seqs only describes packed batches: a fixed-length call carrying a stale
    value beyond the array's sequence limit still runs."""
    f = _entry(kda)
    x = kda_inputs.fixed(2, 100, 2, 128, dtype=torch.bfloat16, device=DEV, seed=55)
    shape = kda.make_shape(x.q, x.v)
    shape.num_seqs = 100000
    o = torch.empty_like(x.v, dtype=torch.float32)
    hT = torch.empty(2, 2, 128, 128, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = f(ctypes.byref(shape), p(x.q), p(x.k), p(x.v), p(x.g), p(x.beta), None, None, p(o),
           p(hT), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK, kda.status_string(rc)
    ref_o, ref_h = kda.fwd(x.q, x.k, x.v, x.g, x.beta)
    assert torch.equal(o, ref_o) and torch.equal(hT, ref_h)


def test_noalloc_long_chain_runs_unsplit(kda, oracle_mod):
    """A chain kda_fwd cuts into segments (that needs its workspace) runs whole
    through the fixed array, with the same results within the tolerance."""
    f = _entry(kda)
    x = kda_inputs.fixed(1, 64 * 257 + 37, 2, 128, dtype=torch.bfloat16, device=DEV, seed=57,
                         h0_std=0.1)
    assert kda.workspace_size(kda.make_shape(x.q, x.v)) > 256  # kda_fwd would split it
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc, o, hT = _call(kda, f, x, status)
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK and int(status.item()) == kda.KDA_OK
    small = torch.empty(256, dtype=torch.uint8, device=DEV)  # kda_fwd without the split
    o_u, h_u = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0, workspace=small)
    assert torch.equal(o, o_u) and torch.equal(hT, h_u)
    o_ref, h_ref = oracle_mod.recurrent(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    assert rel_err(o, o_ref) <= TOL_BF16
    assert rel_err(hT, h_ref) <= TOL_BF16


def test_noalloc_reports_device_errors_and_limits(kda):
    f = _entry(kda)
    x = kda_inputs.packed([50, 50], 2, 128, dtype=torch.bfloat16, device=DEV, seed=4)
    x.cu_seqlens = torch.tensor([0, 60, 40], dtype=torch.int32, device=DEV)  # decreasing
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc, _, _ = _call(kda, f, x, status)
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK
    assert int(status.item()) == kda.KDA_ERR_BAD_SEQLENS
    # more sequences than the fixed array holds: rejected before any launch
    shape = kda.make_shape(x.q, x.v, packed_seqs=16385)
    vp = ctypes.c_void_p
    rc = f(ctypes.byref(shape), *([vp(x.q.data_ptr())] * 5), vp(x.cu_seqlens.data_ptr()), None,
           vp(x.q.data_ptr()), None, None, None)
    assert rc == kda.KDA_ERR_UNSUPPORTED
