"""Seeded synthetic inputs shaped like the KDA layer of the pages' model.

This module draws inputs only; it contains none of the operator's arithmetic.
It serves both the CUDA path and the fp64 oracle in the tests and the
benchmark, which is the only thing the two share.

Recipe (all workloads): q, k ~ N(0, 1) then L2-normalised over the head
dimension per (token, head) -- the caller-side L2Norm of the pages' layer;
v ~ N(0, 1); g = max(-5, log sigmoid(x)) with x ~ N(mu, 1) per channel (the
log-decay bounded below by g_min = -5); beta = sigmoid(N(0, 1)) per
(token, head).  bf16 tensors are rounded once (round-to-nearest-even) from
the fp32 draws.  Draw order per workload: q, k, v, x, beta-logits, then the
initial state.  Sizes: 96 heads of dimension 128 ("Inside Kimi K3", section
"Sequence mixing"), contexts up to 256K tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple            # tokens per sequence
    heads: int
    d: int
    dtype: torch.dtype        # q, k, v (and out)
    mu: float                 # mean of the decay logit x
    init_std: float           # std of the initial state (0 = zero state)
    seed: int
    steps: int = 0            # decode workloads: steps per sequence
    notes: str = field(default="", compare=False)

    @property
    def num_seqs(self):
        return len(self.lengths)

    @property
    def total_tokens(self):
        return int(sum(self.lengths))


def _varlen_lengths():
    return tuple(int(x) for x in np.random.default_rng(2).integers(1024, 32769, 8))


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", (256,), 2, 64, torch.float32, 2.0, 0.0, 0,
                          notes="B=1, T=256, H=2, d=64, fp32"),
    "prefill_8k": Workload("prefill_8k", (8192,), 96, 128, torch.bfloat16, 2.0, 0.0, 1,
                           notes="B=1, T=8192, H=96, d=128, bf16 q/k/v/o"),
    "varlen_8seq": Workload("varlen_8seq", _varlen_lengths(), 96, 128, torch.bfloat16, 2.0,
                            0.02, 2, notes="8 packed sequences of 1024..32768 tokens"),
    "prefill_256k": Workload("prefill_256k", (262144,), 96, 128, torch.bfloat16, 4.0, 0.0, 3,
                             notes="B=1, T=262144, retention-skewed gates (x ~ N(4,1))"),
    "decode_256x64": Workload("decode_256x64", (1,) * 256, 96, 128, torch.bfloat16, 2.0, 0.02,
                              4, steps=64, notes="256 sequences x 64 decode steps"),
}


def _gen(seed, device):
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def draw_tokens(T, H, dk, dv, dtype, mu, gen, device):
    """q, k, v, g, beta for T tokens (draw order q, k, v, x, beta-logit)."""
    q = torch.randn((T, H, dk), generator=gen, device=device, dtype=torch.float32)
    q = (q / q.norm(dim=-1, keepdim=True)).to(dtype)
    k = torch.randn((T, H, dk), generator=gen, device=device, dtype=torch.float32)
    k = (k / k.norm(dim=-1, keepdim=True)).to(dtype)
    v = torch.randn((T, H, dv), generator=gen, device=device, dtype=torch.float32).to(dtype)
    x = torch.randn((T, H, dk), generator=gen, device=device, dtype=torch.float32) + mu
    g = torch.nn.functional.logsigmoid(x).clamp_(min=-5.0)
    del x
    beta = torch.sigmoid(torch.randn((T, H), generator=gen, device=device, dtype=torch.float32))
    return q, k, v, g, beta


def prefill_inputs(w: Workload | str, device="cuda", heads=None, lengths=None):
    """Inputs of a prefill workload.  ``heads``/``lengths`` override the
    workload's sizes (smaller cases of the same recipe)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    H = w.heads if heads is None else int(heads)
    lens = tuple(w.lengths if lengths is None else lengths)
    T = int(sum(lens))
    gen = _gen(w.seed, device)
    q, k, v, g, beta = draw_tokens(T, H, w.d, w.d, w.dtype, w.mu, gen, device)
    N = len(lens)
    init = None
    if w.init_std > 0:
        init = torch.randn((N, H, w.d, w.d), generator=gen, device=device,
                           dtype=torch.float32) * w.init_std
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init, cu_seqlens=cu,
                num_seqs=N, lengths=lens)


def decode_inputs(w: Workload | str = "decode_256x64", device="cuda", num_seqs=None,
                  heads=None, steps=None):
    """Initial states [N, H, d, d] and per-step inputs stacked over steps:
    q, k, v, g [S, N, H, d]; beta [S, N, H]."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    N = w.num_seqs if num_seqs is None else int(num_seqs)
    H = w.heads if heads is None else int(heads)
    S = w.steps if steps is None else int(steps)
    gen = _gen(w.seed, device)
    state = torch.randn((N, H, w.d, w.d), generator=gen, device=device,
                        dtype=torch.float32) * w.init_std
    q, k, v, g, beta = draw_tokens(S * N, H, w.d, w.d, w.dtype, w.mu, gen, device)
    shp = (S, N, H, w.d)
    return dict(state=state, q=q.view(shp), k=k.view(shp), v=v.view(shp), g=g.view(shp),
                beta=beta.view(S, N, H))


def random_inputs(T, H, d, dtype=torch.float32, mu=2.0, seed=0, device="cpu",
                  num_seqs=1, init_std=0.0):
    """Same recipe at an arbitrary size (tests of tails and edge cases)."""
    gen = _gen(seed, device)
    q, k, v, g, beta = draw_tokens(T, H, d, d, dtype, mu, gen, device)
    init = None
    if init_std > 0:
        init = torch.randn((num_seqs, H, d, d), generator=gen, device=device,
                           dtype=torch.float32) * init_std
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init)


# Gate logits for the fused gate prologue (kda_prefill_gated).  Recipe:
# z ~ N(-3.6, 1) per (token, head, channel), rounded once to `dtype`; A_h ~
# 0.1 N(0, 1) per head; beta logits ~ N(0, 1) per (token, head).  With
# g = -5 Sigmoid(e^{A_h} z) this gives a mean retention e^g of about 0.87,
# close to the 0.88 of the g recipe above.  Draw order: z, A, beta logits.
GATE_Z_MEAN = -3.6


def gate_logits(T, H, d, dtype=torch.float32, seed=0, device="cpu"):
    gen = _gen(seed, device)
    z = (torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32)
         + GATE_Z_MEAN).to(dtype)
    a_log = 0.1 * torch.randn((H,), generator=gen, device=device, dtype=torch.float32)
    beta_logit = torch.randn((T, H), generator=gen, device=device, dtype=torch.float32)
    return dict(z=z, a_log=a_log, beta_logit=beta_logit)



def output_gate_inputs(T, H, dv, dtype=torch.float32, seed=0, device="cpu"):
    """Inputs of the output gate: gate logits W_g x_t ~ N(0, 1) per (token, head,
    value channel), in the activation dtype, and a per-channel norm weight
    ~ U(0.5, 1.5) (fp32)."""
    gen = _gen(seed, device)
    gate = torch.randn((T, H, dv), generator=gen, device=device, dtype=torch.float32).to(dtype)
    w = 0.5 + torch.rand((dv,), generator=gen, device=device, dtype=torch.float32)
    return dict(gate=gate, norm_weight=w)


def scalar_decay(T, H, mu=2.0, seed=0, device="cpu"):
    """One log-decay per (token, head) for the scalar-decay variant (Gated
    DeltaNet): g = max(-5, log Sigmoid(x)), x ~ N(mu, 1), the per-channel
    recipe drawn once per head instead of once per channel (fp32 [T, H])."""
    gen = _gen(seed, device)
    x = torch.randn((T, H), generator=gen, device=device, dtype=torch.float32) + mu
    return torch.clamp(torch.nn.functional.logsigmoid(x), min=-5.0)


def qkv_projections(T, H, d, N=1, dtype=torch.float32, seed=0, device="cpu"):
    """Inputs of the q, k, v prologue: the projections W_{q,k,v} x_t ~ N(0, 1)
    per (token, head, channel) in the activation dtype; conv weights
    ~ U(-1/2, 1/2) (the usual fan-in bound 1/sqrt(width) of a width-4
    depthwise convolution), fp32 [3, H, d, 4]; a carried conv state
    ~ N(0, 1), fp32 [N, 3, 3, H, d], rounded through the activation dtype (it
    holds earlier inputs)."""
    gen = _gen(seed, device)
    xs = [torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32).to(dtype)
          for _ in range(3)]
    w = torch.rand((3, H, d, 4), generator=gen, device=device, dtype=torch.float32) - 0.5
    state = torch.randn((N, 3, 3, H, d), generator=gen, device=device,
                        dtype=torch.float32).to(dtype).float()
    return dict(x_q=xs[0], x_k=xs[1], x_v=xs[2], conv_weight=w, conv_state=state)
