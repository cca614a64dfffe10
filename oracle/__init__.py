"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct CPU evaluations of the Kimi Delta Attention
(KDA) forward, in float64.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library and never imports it.

Three forms are provided, each citing the passage it follows:

* :func:`recurrent` -- the definition, token by token (C, ``kda_oracle.c``).
  "Kimi K3 技术报告摘要", section 1 预训练 Recipe, 训练策略 table, KDA row:
  a delta-rule recurrence with a channel-wise forget gate.  Per token
  ``S <- diag(alpha_t) S``, ``S <- S + beta_t k_t (v_t - S^T k_t)^T``,
  ``o_t = scale * S^T q_t``; the state resets at every packed-sequence
  boundary ("Kimi K3 NPU Training", section 定长与 TND).
* :func:`chunked` -- the chunkwise-parallel form of the same recurrence
  (parallel inside a chunk, recurrent across chunks; same KDA row) written
  out with numpy, including the sub-chunk decay factorisation.
* :func:`segment_transition` / :func:`compose` -- the associative affine
  decomposition that KDA context parallelism rests on ("Kimi K3 模型结构（7）：
  结构决定系统", section 上下文并行: each segment contributes a local transition
  matrix and a zero-start state; a prefix scan combines them).
* :func:`recurrent_grad` -- the gradients of the forward's outputs (o and the
  final state) with respect to q, k, v, g, beta and h0: reverse-mode automatic
  differentiation (torch autograd, float64, CPU) of the token recurrence written
  out step by step.  The backward is one of the KDA training operators on "Kimi
  K3 NPU Training" (section 结论, item 1; section NPU 算子支持度, row KDA 反向:
  dq, dk, dv, dbeta, dgate and dstate).
* :func:`preprocess` -- the input preprocessing that the fused entry points
  apply ("Kimi K3 NPU Training", section 模型结构, steps 1 and 3: q/k L2
  normalisation, channel-wise decay and beta from the gate inputs), evaluated
  in float64; the gate and beta are rounded to the input dtype, the normalised
  q and k are not.

Parity status: every function here is pinned by ``tests/test_oracle.py``
against closed forms, special cases and a brute-force Kronecker formulation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``_build/libkda_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path):
    """Open a compiled oracle library (the default one, or a test's mutant copy)."""
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.kda_oracle_recurrent.restype = ctypes.c_int
    lib.kda_oracle_recurrent.argtypes = [
        i64, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp,
        ctypes.c_int, ctypes.c_double, vp, vp, ctypes.c_int]
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    lib.kda_oracle_max_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def max_threads() -> int:
    """Threads the oracle uses by default (OpenMP's view of the host)."""
    return int(_load().kda_oracle_max_threads())


def _as_host(x, f64):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: an exact float32 (or float64) copy
        x = x.detach().to("cpu")
        x = (x.double() if f64 else x.float()).numpy()
    return np.ascontiguousarray(x, dtype=np.float64 if f64 else np.float32)


def _is_f64(x):
    return x is not None and str(getattr(x, "dtype", "")) in ("float64", "torch.float64")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrent(q, k, v, g, beta, *, cu_seqlens=None, h0=None, scale=None, n_threads=None,
              lib=None):
    """Token-by-token KDA forward in float64 (the definition).

    Shapes: fixed batch ``q,k,g [B,T,H,dk]``, ``v [B,T,H,dv]``, ``beta [B,T,H]``;
    or packed ``[T,H,d]`` / ``[T,H]`` with ``cu_seqlens`` (N+1 offsets).
    ``g`` is log(alpha).  ``h0`` is ``[N,H,dk,dv]`` or None (zeros).
    ``scale`` defaults to dk**-0.5.  Inputs may be numpy arrays or torch
    tensors; they are copied to host float32 (exact for bf16 and fp32 data), or
    to float64 when any activation is float64.
    ``lib`` overrides the compiled library (used by the mutation tests).
    Returns ``(o, hT)`` as float64 arrays with ``o`` shaped like ``v``.
    """
    # float64 buffers when any activation is float64 (exact for the others too)
    f64 = any(_is_f64(x) for x in (q, k, v, g, beta))
    q, k, v, g, beta = (_as_host(x, f64) for x in (q, k, v, g, beta))
    h0 = _as_host(h0, f64)
    out_shape = v.shape
    if cu_seqlens is None:
        if q.ndim != 4:
            raise ValueError("fixed-length inputs must be [B,T,H,d]")
        B, T, H, dk = q.shape
        cu = np.arange(B + 1, dtype=np.int64) * T
        q, k, v, g = (x.reshape(B * T, H, -1) for x in (q, k, v, g))
        beta = beta.reshape(B * T, H)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        if q.ndim == 4:  # [1, T, H, d]
            q, k, v, g = (x.reshape(x.shape[1], x.shape[2], x.shape[3]) for x in (q, k, v, g))
            beta = beta.reshape(beta.shape[1], beta.shape[2])
        H, dk = q.shape[1], q.shape[2]
    dv = v.shape[-1]
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != q.shape[0]:
        raise ValueError("cu_seqlens must start at 0 and end at the token count")
    if scale is None:
        scale = dk ** -0.5
    if h0 is not None and h0.shape != (N, H, dk, dv):
        raise ValueError("h0 must be [N,H,dk,dv]")
    o = np.empty(v.shape, dtype=np.float64)
    hT = np.empty((N, H, dk, dv), dtype=np.float64)
    nt = max_threads() if n_threads is None else int(n_threads)
    rc = (lib or _load()).kda_oracle_recurrent(N, _ptr(cu), H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(g), _ptr(beta), _ptr(h0), int(f64), float(scale),
                                      _ptr(o), _ptr(hT), nt)
    if rc != 0:
        raise RuntimeError("oracle: bad arguments or out of memory")
    return o.reshape(out_shape), hT


# ---------------------------------------------------------------------------
# gradients (torch autograd, float64)
# ---------------------------------------------------------------------------

def recurrent_grad(q, k, v, g, beta, do, *, cu_seqlens=None, h0=None, dhT=None, scale=None):
    """Gradients of L = sum(o * do) + sum(hT * dhT) (dhT None: no state term).

    Shapes as in :func:`recurrent`; ``do`` is shaped like ``v``.  The forward
    is the recurrence itself, one token at a time, vectorised over heads only:
      S <- diag(e^g_t) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;
      o_t = scale S^T q_t
    and the gradients are torch autograd's, in float64.  Returns numpy float64
    ``(dq, dk, dv, dg, dbeta, dh0)`` shaped like the inputs (dh0 [N,H,dk,dv],
    also when h0 is None, i.e. zero).
    """
    import torch

    def t64(x):
        if x is None:
            return None
        if hasattr(x, "detach"):
            x = x.detach().double().cpu().numpy()
        return torch.from_numpy(np.array(x, dtype=np.float64))

    Q, K, V, G, Bt, dO = (t64(x) for x in (q, k, v, g, beta, do))
    shapes = [x.shape for x in (Q, K, V, G, Bt)]
    if cu_seqlens is None:
        B, T = Q.shape[0], Q.shape[1]
        cu = [b * T for b in range(B + 1)]
    else:
        cu = [int(c) for c in (cu_seqlens.detach().cpu().numpy()
                               if hasattr(cu_seqlens, "detach") else cu_seqlens)]
    H, dk = Q.shape[-2], Q.shape[-1]
    dv = V.shape[-1]
    N = len(cu) - 1
    if scale is None:
        scale = dk ** -0.5
    H0 = t64(h0) if h0 is not None else torch.zeros(N, H, dk, dv, dtype=torch.float64)
    leaves = [Q, K, V, G, Bt, H0]
    for x in leaves:
        x.requires_grad_(True)
    Qf, Kf, Gf = (x.reshape(-1, H, dk) for x in (Q, K, G))
    Vf = V.reshape(-1, H, dv)
    Bf = Bt.reshape(-1, H)
    outs, finals = [], []
    for n in range(N):
        S = H0[n]
        for t in range(cu[n], cu[n + 1]):
            S = S * torch.exp(Gf[t])[:, :, None]
            pred = torch.einsum("hkv,hk->hv", S, Kf[t])
            u = Bf[t][:, None] * (Vf[t] - pred)
            S = S + Kf[t][:, :, None] * u[:, None, :]
            outs.append(scale * torch.einsum("hkv,hk->hv", S, Qf[t]))
        finals.append(S)
    loss = (torch.stack(outs) * dO.reshape(-1, H, dv)).sum() if outs else Q.sum() * 0.0
    if dhT is not None:
        loss = loss + (torch.stack(finals) * t64(dhT)).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    res = []
    for x, gr, shp in zip(leaves, grads, shapes + [H0.shape]):
        res.append(np.zeros(tuple(shp)) if gr is None else gr.numpy().reshape(shp))
    return tuple(res)


# ---------------------------------------------------------------------------
# input preprocessing (numpy, float64)
# ---------------------------------------------------------------------------

def preprocess(q, k, g, beta, *, qk_l2norm=True, gate_softplus=True, beta_sigmoid=True,
               gate_scale=None, gate_per_head=False):
    """Preprocessed (q, k, g, beta) as torch tensors.

    Each enabled step follows its definition in float64 on the given values.  The
    gate and beta are then rounded to the input dtype (the kernels round them
    there too); normalised q and k stay float64 (the kernels carry them in
    float32, unrounded):
      q, k:  x / max(||x||_2, 1e-12) over the head dimension
      g:     -a_h softplus(g), softplus(x) = log(1 + e^x) (= x above 20), a_h the
             per-head scale (1 when gate_scale is None)
      beta:  1 / (1 + e^-beta)
    With gate_per_head, g holds one value per (token, head) (the scalar-gate
    variant); the result is that value repeated over the dk key channels.
    """
    import torch
    dt = q.dtype
    f = lambda t: t.detach().double().cpu().numpy()
    back = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dt)
    Q, K, G, Bt = f(q), f(k), f(g), f(beta)
    if qk_l2norm:
        Q = Q / np.maximum(np.sqrt(np.sum(Q * Q, axis=-1, keepdims=True)), 1e-12)
        K = K / np.maximum(np.sqrt(np.sum(K * K, axis=-1, keepdims=True)), 1e-12)
    if gate_per_head:
        G = G[..., None]
    if gate_softplus:
        G = -np.where(G > 20.0, G, np.log1p(np.exp(np.minimum(G, 20.0))))
        if gate_scale is not None:
            a = np.asarray(gate_scale.detach().double().cpu().numpy()
                           if hasattr(gate_scale, "detach") else gate_scale, dtype=np.float64)
            G = G * a[:, None]
    if beta_sigmoid:
        Bt = 1.0 / (1.0 + np.exp(-Bt))
    Gr = back(G)
    if gate_per_head:
        Gr = Gr.expand(*G.shape[:-1], Q.shape[-1]).contiguous()
    exact = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    qk = exact if qk_l2norm else back
    return qk(Q), qk(K), Gr, back(Bt)


# ---------------------------------------------------------------------------
# chunkwise-parallel form (numpy, float64)
# ---------------------------------------------------------------------------

def _tri_inv_unit_lower(A):
    """(I + A)^-1 for strictly lower-triangular A, by forward substitution."""
    n = A.shape[0]
    T = np.eye(n)
    for i in range(1, n):
        # row i of (I + A) T = I  =>  T[i] = e_i - sum_{j<i} A[i, j] T[j]
        T[i, :i] -= A[i, :i] @ T[:i, :i]
    return T


def chunk_chain(Q, K, V, G, b, S, scale, C=64, sub=16):
    """One (sequence, head) chain in chunks of C tokens.

    Inside a chunk with inclusive log-decay prefix sums Gam (per channel):
      A   = strict_lower(diag(b) (K*e^Gam)(K*e^-Gam)^T)    decayed key products
      Aqk = lower_incl_diag((Q*e^Gam)(K*e^-Gam)^T)          decayed query-key products
      T   = (I + A)^-1,  W = T diag(b) (K*e^Gam),  Ut = T diag(b) V
      U   = Ut - W S
      O   = scale ((Q*e^Gam) S + Aqk U)
      S  <- diag(e^Gam_last) S + (K*e^(Gam_last - Gam))^T U
    The decayed products are evaluated per column block of ``sub`` tokens,
    with the decay split about the log-decay value just before the block
    (row factor <= 1, column factor bounded by the block's own decay).
    Returns (O [L,dv], S_end [dk,dv]).
    """
    L, dk = K.shape
    O = np.empty((L, V.shape[1]))
    S = np.array(S, dtype=np.float64, copy=True)
    for s in range(0, L, C):
        e = min(L, s + C)
        n = e - s
        q, k, v, g, bb = Q[s:e], K[s:e], V[s:e], G[s:e], b[s:e]
        Gam = np.cumsum(g, axis=0)
        Akk = np.zeros((n, n))
        Aqk = np.zeros((n, n))
        for J in range(0, n, sub):
            je = min(n, J + sub)
            rho = Gam[J - 1] if J > 0 else np.zeros(dk)
            row = np.exp(Gam[J:] - rho)          # tokens at or after block J
            col = k[J:je] * np.exp(rho - Gam[J:je])
            Akk[J:, J:je] = (k[J:] * row) @ col.T
            Aqk[J:, J:je] = (q[J:] * row) @ col.T
        A = np.tril(Akk, -1) * bb[:, None]
        Aqk = np.tril(Aqk, 0)
        T = _tri_inv_unit_lower(A)
        gam = np.exp(Gam)
        W = T @ (bb[:, None] * k * gam)
        Ut = T @ (bb[:, None] * v)
        U = Ut - W @ S
        O[s:e] = scale * ((q * gam) @ S + Aqk @ U)
        S = np.exp(Gam[-1])[:, None] * S + (k * np.exp(Gam[-1] - Gam)).T @ U
    return O, S


def chunked(q, k, v, g, beta, *, cu_seqlens=None, h0=None, scale=None, C=64, sub=16):
    """Chunkwise form over all chains; same argument conventions as :func:`recurrent`."""
    f64 = lambda x: None if x is None else np.asarray(
        x.detach().cpu().float().numpy() if hasattr(x, "detach") else x, dtype=np.float64)
    q, k, v, g, beta, h0 = (f64(x) for x in (q, k, v, g, beta, h0))
    out_shape = v.shape
    if cu_seqlens is None:
        B, T, H, dk = q.shape
        cu = np.arange(B + 1) * T
        q, k, v, g = (x.reshape(B * T, H, -1) for x in (q, k, v, g))
        beta = beta.reshape(B * T, H)
    else:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
        if q.ndim == 4:
            q, k, v, g = (x[0] for x in (q, k, v, g))
            beta = beta[0]
        H, dk = q.shape[1], q.shape[2]
    dv = v.shape[-1]
    N = len(cu) - 1
    if scale is None:
        scale = dk ** -0.5
    o = np.empty(v.shape)
    hT = np.empty((N, H, dk, dv))
    for n in range(N):
        a, z = cu[n], cu[n + 1]
        for h in range(H):
            S0 = h0[n, h] if h0 is not None else np.zeros((dk, dv))
            O, S = chunk_chain(q[a:z, h], k[a:z, h], v[a:z, h], g[a:z, h], beta[a:z, h],
                               S0, scale, C=C, sub=sub)
            o[a:z, h] = O
            hT[n, h] = S
    return o.reshape(out_shape), hT


# ---------------------------------------------------------------------------
# segment transitions (the affine decomposition behind KDA context parallelism)
# ---------------------------------------------------------------------------

def segment_transition(k, v, g, beta):
    """(M, b) of one segment of one head such that S_end = M @ S_start + b.

    ``k, g`` are [L, dk], ``v`` [L, dv], ``beta`` [L] (float64 numpy).  Every
    token acts on the state affinely, so the segment does too: ``b`` is the
    end state from a zero start, and ``M`` is the end state of the same
    tokens applied to the identity with the values set to zero (each column
    of a dk x dk state evolves independently).
    """
    L, dk = k.shape
    zeros_h = lambda d: np.zeros((1, 1, dk, d))
    kk, gg = k[:, None, :], g[:, None, :]
    bb = beta[:, None]
    cu = np.array([0, L])
    _, b = recurrent(kk, kk, v[:, None, :], gg, bb, cu_seqlens=cu, h0=zeros_h(v.shape[1]),
                     scale=1.0)
    _, M = recurrent(kk, kk, np.zeros((L, 1, dk)), gg, bb, cu_seqlens=cu,
                     h0=np.eye(dk)[None, None], scale=1.0)
    return M[0, 0], b[0, 0]


def compose(first, second):
    """Transition of ``first`` followed by ``second``: S -> M2 (M1 S + b1) + b2."""
    M1, b1 = first
    M2, b2 = second
    return M2 @ M1, M2 @ b1 + b2


def apply_transition(tr, S):
    M, b = tr
    return M @ S + b
