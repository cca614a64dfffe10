"""Seeded synthetic inputs for the KDA forward.

This module only draws random tensors and applies the input conventions the
operator expects; it holds none of the recurrence's arithmetic, so both the
CUDA path's tests and the float64 oracle can take their inputs from it.

Conventions (the operator's preconditions):

* q, k ~ N(0, 1), then L2-normalised over the head dimension (norm floored at
  1e-12) -- "Kimi K3 NPU Training", section 模型结构, step 3: q/k are L2
  normalised before the recurrence.
* v ~ N(0, 1).
* g = log(alpha) = -softplus(x), x ~ N(0, 1): a per-channel forget gate in (0, 1).
* beta = sigmoid(x), x ~ N(0, 1).
* Everything is drawn in float32 and then cast to the requested dtype; the
  oracle consumes the cast values.

Sequence lengths for packed batches are drawn uniformly from [lo, hi].
"""
from __future__ import annotations

import dataclasses

import torch
import torch.nn.functional as F


@dataclasses.dataclass
class KDAInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor | None
    h0: torch.Tensor | None
    scale: float

    @property
    def num_tokens(self) -> int:
        return self.q.shape[0] * self.q.shape[1]


def _gen(device, seed):
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def draw(shape_tok, H, dk, dv, *, dtype=torch.bfloat16, device="cpu", seed=0,
         cu_seqlens=None, num_states=None, h0_std=None):
    """Draw q, k, v, g, beta of leading shape ``shape_tok`` (e.g. (B, T) or (1, T)).

    ``h0_std`` draws a float32 start state ``[num_states, H, dk, dv]`` from
    N(0, h0_std^2); None leaves h0 unset (zero start state).
    """
    gen = _gen(device, seed)
    f32 = dict(device=device, dtype=torch.float32, generator=gen)
    q = torch.randn(*shape_tok, H, dk, **f32)
    k = torch.randn(*shape_tok, H, dk, **f32)
    v = torch.randn(*shape_tok, H, dv, **f32)
    graw = torch.randn(*shape_tok, H, dk, **f32)
    braw = torch.randn(*shape_tok, H, **f32)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    g = -F.softplus(graw)
    beta = torch.sigmoid(braw)
    h0 = None
    if h0_std is not None:
        h0 = torch.randn(num_states, H, dk, dv, **f32) * float(h0_std)
    cast = lambda x: x.to(dtype).contiguous()
    return KDAInputs(cast(q), cast(k), cast(v), cast(g), cast(beta), cu_seqlens, h0,
                     dk ** -0.5)


def draw_raw(shape_tok, H, dk, dv, *, dtype=torch.bfloat16, device="cpu", seed=0,
             cu_seqlens=None, num_states=None, h0_std=None):
    """Like ``draw`` but without the input conventions: q, k ~ N(0, 1) as drawn
    (not normalised), g and beta the raw N(0, 1) gate inputs (no softplus or
    sigmoid), all cast to ``dtype``; the inputs of the fused-preprocessing
    entry points."""
    gen = _gen(device, seed)
    f32 = dict(device=device, dtype=torch.float32, generator=gen)
    q = torch.randn(*shape_tok, H, dk, **f32)
    k = torch.randn(*shape_tok, H, dk, **f32)
    v = torch.randn(*shape_tok, H, dv, **f32)
    graw = torch.randn(*shape_tok, H, dk, **f32)
    braw = torch.randn(*shape_tok, H, **f32)
    h0 = None
    if h0_std is not None:
        h0 = torch.randn(num_states, H, dk, dv, **f32) * float(h0_std)
    cast = lambda x: x.to(dtype).contiguous()
    return KDAInputs(cast(q), cast(k), cast(v), cast(graw), cast(braw), cu_seqlens, h0,
                     dk ** -0.5)


def fixed(B, T, H, d, *, dtype=torch.bfloat16, device="cpu", seed=0, h0_std=None):
    """Fixed-length batch [B, T, H, d]."""
    return draw((B, T), H, d, d, dtype=dtype, device=device, seed=seed,
                num_states=B, h0_std=h0_std)


def seq_lengths(n, lo, hi, seed):
    """n sequence lengths uniform in [lo, hi] (CPU generator, so identical everywhere)."""
    gen = _gen("cpu", seed)
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


def packed(lengths, H, d, *, dtype=torch.bfloat16, device="cpu", seed=0, h0_std=None):
    """Packed variable-length batch [1, sum(lengths), H, d] with int32 cu_seqlens."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    total = int(cu[-1])
    x = draw((1, total), H, d, d, dtype=dtype, device=device, seed=seed,
             num_states=len(lengths), h0_std=h0_std)
    x.cu_seqlens = cu.to(torch.int32).to(device)
    return x


# The five workloads the operator is exercised on (seed 1000 + index).
def workload(index, *, device="cpu", dtype=None):
    """Inputs of workload ``index``:

    0  tiny fp32: B=1, T=256, H=2, d=64
    1  fixed-length prefill: B=4, T=4096, H=32, d=128 (bf16)
    2  packed prefill: 16 sequences, lengths uniform in [128, 8192], H=32,
       d=128, bf16, h0 ~ N(0, 0.1^2)
    3  long context: B=1, T=1,048,576, H=32, d=128, bf16
    4  decode pool: 1024 sequences, H=32, d=128; see :func:`decode_pool`
    """
    seed = 1000 + index
    if index == 0:
        return fixed(1, 256, 2, 64, dtype=dtype or torch.float32, device=device, seed=seed)
    if index == 1:
        return fixed(4, 4096, 32, 128, dtype=dtype or torch.bfloat16, device=device, seed=seed)
    if index == 2:
        lens = seq_lengths(16, 128, 8192, seed)
        return packed(lens, 32, 128, dtype=dtype or torch.bfloat16, device=device, seed=seed,
                      h0_std=0.1)
    if index == 3:
        return fixed(1, 1 << 20, 32, 128, dtype=dtype or torch.bfloat16, device=device,
                     seed=seed)
    raise ValueError(f"no prefill workload {index}")


def decode_pool(num_seqs=1024, H=32, d=128, T_step=1, *, dtype=torch.bfloat16, device="cpu",
                seed=1004, state_std=0.1):
    """Decode step inputs [num_seqs, T_step, H, d] plus a float32 state pool
    [num_seqs, H, d, d] ~ N(0, state_std^2)."""
    x = draw((num_seqs, T_step), H, d, d, dtype=dtype, device=device, seed=seed,
             num_states=num_seqs, h0_std=state_std)
    return x
