"""Seeded synthetic inputs for the channelwise gated delta rule forward.

This module only draws random tensors: it holds none of the method's
arithmetic, so both the CUDA path's tests and the fp64 oracle consume exactly
the same values.  Every tensor is drawn in float32 on the CPU from one
``torch.Generator`` in a fixed order (q, k, v, g-raw, beta-raw, h0), then:

* q and k are L2-normalised over the key dimension per (b, t, head) in float32
  and cast to the q/k/v dtype;
* v is cast to the q/k/v dtype;
* g = -softplus(N(g_mu, g_sigma)) (a per-key-channel log-decay <= 0, float32);
* beta = sigmoid(N(beta_mu, beta_sigma)) (float32);
* h0 = h0_scale * N(0, 1) (float32) when an initial state is requested.

These are the distributions the uzu review (trymirai/uzu PR #576, review
thread on the synthetic packed-A test) asks for in a real-scale test:
normalised keys, softplus decays and an initial state at ~0.3 scale.

The named workloads below are the shapes the library is tested and measured
on.  ``device="cuda"`` draws directly on the GPU with a CUDA generator
(different values, same distributions) for throughput runs where no oracle
comparison is made.
"""
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    HK: int
    HV: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype
    h0: bool
    g_mu: float = 0.0
    g_sigma: float = 1.0
    beta_mu: float = 0.0
    beta_sigma: float = 1.0
    h0_scale: float = 0.3
    lengths: Optional[Sequence[int]] = field(default=None)  # ragged batch: one T per sequence


WORKLOADS = {
    # small case the oracle finishes instantly; spans several chunks of 16
    "tiny": Workload("tiny", 1, 64, 2, 2, 32, 32, 16, torch.float32, True),
    # one decode step for a batch of 64 sequences, state updated in place
    "decode_b64": Workload("decode_b64", 64, 1, 16, 32, 128, 128, 64, torch.bfloat16, True),
    # eight sequences of different lengths, each its own call
    "ragged_b8": Workload("ragged_b8", 8, 512, 16, 32, 128, 128, 64, torch.float32, True,
                          lengths=(1, 33, 49, 64, 97, 128, 256, 512)),
    # one 4k-token prefill with a zero initial state
    "prefill_t4k": Workload("prefill_t4k", 1, 4096, 16, 32, 128, 128, 64, torch.bfloat16, False),
    # long prefill with beta near 1 and slow decay (||A|| ~ 1 inside chunks)
    "prefill_t16k": Workload("prefill_t16k", 4, 16384, 16, 32, 128, 128, 64, torch.bfloat16, True,
                             g_mu=-3.0, g_sigma=1.0, beta_mu=2.0, beta_sigma=0.5),
}


def draw(B, T, HK, HV, dk, dv, dtype=torch.float32, h0=True, seed=0, g_mu=0.0, g_sigma=1.0,
         beta_mu=0.0, beta_sigma=1.0, h0_scale=0.3, device="cpu", generator=None,
         scalar_gate=False):
    """Draws one problem.  Returns a dict q, k, v, g, beta, h0 (h0 may be None).
    g is [B, T, HV, dk], or [B, T, HV] (one log-decay per token and head) with
    scalar_gate."""
    if generator is None:
        generator = torch.Generator(device=device)
        generator.manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=device, generator=generator)
    q = torch.randn(B, T, HK, dk, **f32)
    k = torch.randn(B, T, HK, dk, **f32)
    v = torch.randn(B, T, HV, dv, **f32)
    g_raw = torch.randn(*((B, T, HV) if scalar_gate else (B, T, HV, dk)), **f32)
    b_raw = torch.randn(B, T, HV, **f32)
    s0 = torch.randn(B, HV, dk, dv, **f32) if h0 else None
    q = torch.nn.functional.normalize(q, dim=-1)
    k = torch.nn.functional.normalize(k, dim=-1)
    g = -torch.nn.functional.softplus(g_raw * g_sigma + g_mu)
    beta = torch.sigmoid(b_raw * beta_sigma + beta_mu)
    out = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), g=g.contiguous(), beta=beta.contiguous(),
               h0=None if s0 is None else (s0 * h0_scale).contiguous())
    return out


def draw_workload(w: Workload, seed=0, device="cpu"):
    """Draws a named workload.  Ragged workloads return a list of per-sequence
    problems (B=1 each, drawn in order from one generator)."""
    kw = dict(dtype=w.dtype, h0=w.h0, g_mu=w.g_mu, g_sigma=w.g_sigma, beta_mu=w.beta_mu,
              beta_sigma=w.beta_sigma, h0_scale=w.h0_scale, device=device)
    if w.lengths is None:
        return draw(w.B, w.T, w.HK, w.HV, w.dk, w.dv, seed=seed, **kw)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return [draw(1, L, w.HK, w.HV, w.dk, w.dv, generator=gen, **kw) for L in w.lengths]


def pack(seqs):
    """Packs per-sequence problems (B=1 each, as draw_workload returns for a
    ragged workload) back to back: q/k/v/g/beta gain a leading dim of 1 over
    all tokens, h0 stacks to [N, HV, dk, dv] (None if the sequences have
    none).  Returns (packed dict, cu_seqlens list of N + 1 ints)."""
    cu = [0]
    for d in seqs:
        cu.append(cu[-1] + d["q"].shape[1])
    packed = {n: torch.cat([d[n] for d in seqs], dim=1).contiguous()
              for n in ("q", "k", "v", "g", "beta")}
    packed["h0"] = (None if seqs[0]["h0"] is None
                    else torch.cat([d["h0"] for d in seqs], dim=0).contiguous())
    return packed, cu


def draw_parents(B, T, kind="random", seed=0, branching=3):
    """Parent arrays [B, T] (int32, parent[b, t] in [-1, t-1], -1 = a root) of
    draft-token trees, parents before children:
      "chain"   parent t-1 (a plain sequence);
      "star"    every token a root (T independent single-token steps);
      "random"  each token's parent uniform over the earlier tokens, or a
                root with probability 1/(t+1);
      "beam"    breadth-first tree, each node with up to `branching` children
                (the usual shape of a speculative-decoding draft tree)."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    par = torch.empty(B, T, dtype=torch.int32)
    for b in range(B):
        for t in range(T):
            if kind == "chain":
                p = t - 1
            elif kind == "star":
                p = -1
            elif kind == "beam":
                p = (t - 1) // branching if t > 0 else -1
            elif kind == "random":
                p = int(torch.randint(-1, t, (1,), generator=gen)) if t > 0 else -1
            else:
                raise ValueError(kind)
            par[b, t] = p
    return par


def to_f64(x):
    """Exact float64 numpy copy of a tensor (bf16 and f32 values are exact in f64)."""
    if x is None:
        return None
    return x.detach().to("cpu", torch.float64).numpy()
