"""Python binding of the GB300 KDA forward library (``libkda.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/kda.h``.  torch supplies
device memory and the current CUDA stream.  If the shared library has not
been built, :func:`load` raises; there is no other code path.

    o, hT = kda_delta_rule_fwd_gb300.fwd(q, k, v, g, beta, cu_seqlens=..., h0=...)
    o = kda_delta_rule_fwd_gb300.decode(q, k, v, g, beta, state)   # state updated in place
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_BAD_SEQLENS = 5
KDA_ERR_DEVICE_TIMEOUT = 6
KDA_ERR_DECAY_RANGE = 7

KDA_F32 = 0
KDA_BF16 = 1

_DT = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}


class Shape(ctypes.Structure):
    """Mirror of ``kda_shape``."""
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("scale", ctypes.c_float)]


class Preproc(ctypes.Structure):
    """Mirror of ``kda_preproc`` (fused input preprocessing flags)."""
    _fields_ = [("qk_l2norm", ctypes.c_int32), ("gate_softplus", ctypes.c_int32),
                ("beta_sigmoid", ctypes.c_int32), ("gate_per_head", ctypes.c_int32),
                ("gate_scale", ctypes.c_void_p)]


def _preproc(q, g, qk_l2norm, gate_softplus, beta_sigmoid, gate_per_head, gate_scale):
    if gate_per_head and tuple(g.shape) != tuple(q.shape[:-1]):
        raise ValueError("a per-head gate has the shape of q without its last dimension")
    if not gate_per_head and g.shape != q.shape:
        raise ValueError("g must have the shape of q")
    if gate_scale is not None and (not gate_scale.is_cuda or gate_scale.dtype != torch.float32
                                   or gate_scale.numel() != q.shape[2]):
        raise ValueError("gate_scale must be a CUDA float32 tensor with one value per head")
    return Preproc(int(qk_l2norm), int(gate_softplus), int(beta_sigmoid), int(gate_per_head),
                   _ptr(gate_scale))


class KDAError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Open ``libkda.so`` (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"KDA CUDA library not built: {p} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(p)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        sp = ctypes.POINTER(Shape)
        lib.kda_workspace_size.restype = sz
        lib.kda_workspace_size.argtypes = [sp]
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_fwd_checkpoints.restype = ctypes.c_int
        lib.kda_fwd_checkpoints.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_int32, vp, vp, ctypes.c_int64, vp, sz, vp]
        pp = ctypes.POINTER(Preproc)
        lib.kda_fwd_preproc.restype = ctypes.c_int
        lib.kda_fwd_preproc.argtypes = [sp, pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_decode_preproc.restype = ctypes.c_int
        lib.kda_decode_preproc.argtypes = [sp, pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_decode.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_decode_commit.restype = ctypes.c_int
        lib.kda_decode_commit.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_bwd_workspace_size.restype = sz
        lib.kda_bwd_workspace_size.argtypes = [sp]
        lib.kda_bwd.restype = ctypes.c_int
        lib.kda_bwd.argtypes = [sp] + [vp] * 16 + [sz, vp]
        lib.kda_read_device_status.restype = ctypes.c_int
        lib.kda_read_device_status.argtypes = [vp, vp]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_version.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def version() -> str:
    return load().kda_version().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(q, v, *, packed_seqs=None, scale=None, out_dtype=torch.float32) -> Shape:
    """kda_shape for activations ``q [B,T,H,dk]`` and ``v [B,T,H,dv]``."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in _DT or out_dtype not in _DT:
        raise TypeError("q/k/v/g/beta and the output must be float32 or bfloat16")
    return Shape(B, T, H, dk, dv, 0 if packed_seqs is None else packed_seqs, _DT[q.dtype],
                 _DT[out_dtype], float(dk ** -0.5 if scale is None else scale))


def workspace_size(shape: Shape) -> int:
    return int(load().kda_workspace_size(ctypes.byref(shape)))


def new_workspace(shape: Shape, device) -> torch.Tensor:
    """A device buffer of ``kda_workspace_size`` bytes (torch allocations are 256-byte aligned)."""
    return torch.empty(workspace_size(shape), dtype=torch.uint8, device=device)


def _check_inputs(q, k, v, g, beta):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, g and beta must share one dtype")


def fwd(q, k, v, g, beta, *, cu_seqlens=None, h0=None, scale=None, out_dtype=torch.float32,
        out=None, hT=None, output_final_state=True, workspace=None, stream=None):
    """KDA chunkwise prefill.  Shapes as in ``kda_fwd``: ``q,k,g [B,T,H,dk]``,
    ``v [B,T,H,dv]``, ``beta [B,T,H]``; packed batches are ``[1,T,H,d]`` with int32
    ``cu_seqlens``.  Returns ``(o, hT)`` (``hT`` is None unless requested)."""
    _check_inputs(q, k, v, g, beta)
    N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    shape = make_shape(q, v, packed_seqs=None if cu_seqlens is None else N, scale=scale,
                       out_dtype=out_dtype)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=out_dtype, device=q.device)
    if hT is None and output_final_state:
        hT = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    rc = load().kda_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        _ptr(cu_seqlens), _ptr(h0), _ptr(out), _ptr(hT), _ptr(workspace),
                        workspace.numel(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_fwd")
    return out, hT


def fwd_checkpoints(q, k, v, g, beta, *, interval=512, cu_seqlens=None, h0=None, scale=None,
                    out_dtype=torch.float32, out=None, hT=None, output_final_state=True,
                    ckpt=None, offsets=None, workspace=None, stream=None):
    """``fwd`` plus prefix-cache checkpoints: the state after every ``interval``
    tokens (a multiple of 64) of each sequence.  Returns ``(o, hT, ckpt, offsets)``
    with ``ckpt [rows, H, dk, dv]`` float32; sequence n's checkpoints are rows
    ``offsets[n] .. offsets[n+1]-1`` (``offsets`` is a device int32 ``[N+1]``).  For
    packed batches the offsets come from ``cu_seqlens`` on the device, and sizing
    ``ckpt`` reads their total on the host (one synchronisation).  A caller that
    passes ``ckpt`` (and, for packed batches, ``offsets``) gets no device work from
    this function besides the kernels; ``offsets`` is then returned as given."""
    _check_inputs(q, k, v, g, beta)
    N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    shape = make_shape(q, v, packed_seqs=None if cu_seqlens is None else N, scale=scale,
                       out_dtype=out_dtype)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if ckpt is not None:
        if cu_seqlens is not None and offsets is None:
            raise ValueError("a packed batch with a given ckpt buffer needs its offsets")
        rows = ckpt.shape[0]
    elif cu_seqlens is None:
        per = T // interval
        offsets = torch.arange(N + 1, dtype=torch.int32, device=q.device) * per
        rows = N * per
    else:
        counts = (cu_seqlens[1:] - cu_seqlens[:-1]) // interval
        offsets = torch.zeros(N + 1, dtype=torch.int32, device=q.device)
        offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
        rows = int(offsets[-1].item())
    if ckpt is None:
        ckpt = torch.empty(rows, H, dk, dv, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=out_dtype, device=q.device)
    if hT is None and output_final_state:
        hT = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    # an empty checkpoint buffer still needs a valid pointer
    ck = ckpt if rows > 0 else torch.empty(4, dtype=torch.float32, device=q.device)
    rc = load().kda_fwd_checkpoints(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
        _ptr(h0), _ptr(out), _ptr(hT), int(interval), _ptr(ck),
        _ptr(offsets) if cu_seqlens is not None else None, rows, _ptr(workspace),
        workspace.numel(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_fwd_checkpoints")
    return out, hT, ckpt, offsets


def fwd_preproc(q, k, v, g, beta, *, qk_l2norm=True, gate_softplus=True, beta_sigmoid=True,
                gate_per_head=False, gate_scale=None, cu_seqlens=None, h0=None, scale=None,
                out_dtype=torch.float32, out=None, hT=None, output_final_state=True,
                workspace=None, stream=None):
    """``fwd`` on raw inputs with the preprocessing fused into the kernels: q, k
    L2-normalised per (token, head), log(alpha) = -gate_scale[h] softplus(g), beta =
    sigmoid(beta), each computed in float32 and rounded to the input dtype (selected
    by the flags).  ``gate_per_head``: g is ``[B,T,H]``, one gate per token and head
    shared by the key channels (the scalar-gate variant)."""
    _check_inputs(q, k, v, g, beta)
    N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    shape = make_shape(q, v, packed_seqs=None if cu_seqlens is None else N, scale=scale,
                       out_dtype=out_dtype)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=out_dtype, device=q.device)
    if hT is None and output_final_state:
        hT = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    pre = _preproc(q, g, qk_l2norm, gate_softplus, beta_sigmoid, gate_per_head, gate_scale)
    rc = load().kda_fwd_preproc(ctypes.byref(shape), ctypes.byref(pre), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), _ptr(h0),
                                _ptr(out), _ptr(hT), _ptr(workspace), workspace.numel(),
                                _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_fwd_preproc")
    return out, hT


def bwd_workspace_size(shape: Shape) -> int:
    return int(load().kda_bwd_workspace_size(ctypes.byref(shape)))


def bwd(q, k, v, g, beta, dout, *, cu_seqlens=None, h0=None, dhT=None, scale=None,
        want_dh0=True, workspace=None, stream=None):
    """Gradients of ``sum(o * dout) + sum(hT * dhT)`` for ``fwd``'s inputs.  Returns
    ``(dq, dk, dv, dg, dbeta, dh0)``, float32 (``dh0`` None unless ``want_dh0``)."""
    _check_inputs(q, k, v, g, beta)
    if dout.dtype != torch.float32 or not dout.is_contiguous() or dout.shape != v.shape:
        raise ValueError("dout must be a contiguous float32 tensor shaped like v")
    N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    shape = make_shape(q, v, packed_seqs=None if cu_seqlens is None else N, scale=scale)
    B, T, H, dk = q.shape
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk_, dg = (torch.empty(B, T, H, dk, **f32) for _ in range(3))
    dv = torch.empty(B, T, H, v.shape[-1], **f32)
    dbeta = torch.empty(B, T, H, **f32)
    dh0 = torch.empty(N, H, dk, v.shape[-1], **f32) if want_dh0 else None
    if workspace is None:
        workspace = torch.empty(bwd_workspace_size(shape), dtype=torch.uint8, device=q.device)
    rc = load().kda_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        _ptr(cu_seqlens), _ptr(h0), _ptr(dout), _ptr(dhT), _ptr(dq), _ptr(dk_),
                        _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(workspace),
                        workspace.numel(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_bwd")
    return dq, dk_, dv, dg, dbeta, dh0


def decode_preproc(q, k, v, g, beta, state, *, qk_l2norm=True, gate_softplus=True,
                   beta_sigmoid=True, gate_per_head=False, gate_scale=None, scale=None,
                   out_dtype=torch.float32, out=None, workspace=None, stream=None):
    """``decode`` on raw inputs with the preprocessing of ``fwd_preproc`` fused in."""
    _check_inputs(q, k, v, g, beta)
    shape = make_shape(q, v, scale=scale, out_dtype=out_dtype)
    B, T, H, dk = q.shape
    if out is None:
        out = torch.empty(B, T, H, v.shape[-1], dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    pre = _preproc(q, g, qk_l2norm, gate_softplus, beta_sigmoid, gate_per_head, gate_scale)
    rc = load().kda_decode_preproc(ctypes.byref(shape), ctypes.byref(pre), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                                   _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_decode_preproc")
    return out


def decode(q, k, v, g, beta, state, *, scale=None, out_dtype=torch.float32, out=None,
           workspace=None, stream=None):
    """KDA decode step over ``q [B,T_step,H,dk]`` (T_step 1..8); ``state [B,H,dk,dv]``
    float32 is updated in place.  Returns ``o [B,T_step,H,dv]``."""
    _check_inputs(q, k, v, g, beta)
    shape = make_shape(q, v, scale=scale, out_dtype=out_dtype)
    B, T, H, dk = q.shape
    if out is None:
        out = torch.empty(B, T, H, v.shape[-1], dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    rc = load().kda_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(state), _ptr(out), _ptr(workspace), workspace.numel(),
                           _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_decode")
    return out


def decode_commit(q, k, v, g, beta, state, num_commit, *, scale=None, out_dtype=torch.float32,
                  out=None, want_out=True, workspace=None, stream=None):
    """Decode step that keeps, per sequence n, the state after its first
    ``num_commit[n]`` tokens (device int32 ``[B]``, each in 0..T_step) while every
    token still produces its output (speculative-decode verification and replay).
    Returns ``o [B,T_step,H,dv]``, or None when ``want_out`` is False."""
    _check_inputs(q, k, v, g, beta)
    if num_commit.dtype != torch.int32 or num_commit.numel() != q.shape[0]:
        raise ValueError("num_commit must be int32 with one count per sequence")
    shape = make_shape(q, v, scale=scale, out_dtype=out_dtype)
    B, T, H, dk = q.shape
    if out is None and want_out:
        out = torch.empty(B, T, H, v.shape[-1], dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = new_workspace(shape, q.device)
    rc = load().kda_decode_commit(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta), _ptr(num_commit), _ptr(state),
                                  _ptr(out) if out is not None else None, _ptr(workspace),
                                  workspace.numel(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_decode_commit")
    return out


def read_device_status(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the status latched on the device."""
    return int(load().kda_read_device_status(_ptr(workspace), _stream_ptr(stream)))
