"""Small runnable cases of the entry points, for profiling a single kernel.

``python -m kda_delta_rule_fwd_gb300.cases bwd`` runs the backward twice (a
warm-up launch, then the one to capture) on B=1, T=512, H=4, d=128, bf16
inputs with a start state; ``prefill`` does the same for the forward on
B=1, T=4096, H=8; ``decode1`` and ``decode8`` the 1- and 8-token decode on 256
sequences x 32 heads.
Inputs are seeded and synthetic.
"""
from __future__ import annotations

import sys

import torch

import kda_inputs
import kda_delta_rule_fwd_gb300 as kda


def bwd_case(device="cuda:0"):
    x = kda_inputs.fixed(1, 512, 4, 128, dtype=torch.bfloat16, device=device, seed=5,
                         h0_std=0.1)
    gen = torch.Generator(device=device)
    gen.manual_seed(6)
    dout = torch.randn(x.v.shape, generator=gen, device=device)
    for _ in range(2):
        grads = kda.bwd(x.q, x.k, x.v, x.g, x.beta, dout, h0=x.h0)
    torch.cuda.synchronize()
    return grads


def prefill_case(device="cuda:0"):
    x = kda_inputs.fixed(1, 4096, 8, 128, dtype=torch.bfloat16, device=device, seed=7,
                         h0_std=0.1)
    for _ in range(2):
        o, hT = kda.fwd(x.q, x.k, x.v, x.g, x.beta, h0=x.h0)
    torch.cuda.synchronize()
    return o, hT


def decode_case(T_step, device="cuda:0"):
    """T_step-token decode on a pool of 256 sequences x 32 heads (512 MB of state)."""
    x = kda_inputs.decode_pool(num_seqs=256, H=32, d=128, T_step=T_step, device=device,
                               seed=15)
    state = x.h0.clone()
    for _ in range(2):
        o = kda.decode(x.q, x.k, x.v, x.g, x.beta, state)
    torch.cuda.synchronize()
    return o, state


if __name__ == "__main__":
    which = sys.argv[1] if len(sys.argv) > 1 else "bwd"
    out = {"bwd": bwd_case, "prefill": prefill_case, "decode1": lambda: decode_case(1),
           "decode8": lambda: decode_case(8)}[which]()
    print(which, "ok", float(out[0].abs().sum()))
