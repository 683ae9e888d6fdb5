"""Seeded synthetic inputs for the KDA prefill and decode workloads.

This module holds the input recipe only (shapes, distributions, seeds); it
contains none of the recurrence's arithmetic.  The tests, the bench and the
smoke check draw from it; both the CUDA path and the float64 oracle consume
what it produces.

Workloads (named by what they are):

  recurrent_tiny_fp32    1 seq, H=1,  T=64,        d=16,  fp32
  prefill_h16_t4096      1 seq, H=16, T=4096,      d=128, bf16
  varlen16_h32           16 seqs, lengths U{512..16384}, H=32, d=128, bf16,
                         per-sequence S0 ~ N(0, 0.02^2)
  prefill_h32_t1m        1 seq, H=32, T=1,048,576, d=128, bf16
  decode_1024x32         1024 seqs x H=32, one token each, d=128, bf16,
                         state S ~ N(0, 0.02^2) fp32

Distributions (the pages describe KDA's inputs; these are the synthetic stand-ins):
  q ~ N(0,1), scaled by 1/sqrt(d_k) for the d=128 workloads;
  k ~ N(0,1), L2-normalised per (token, head) in fp32 before any cast;
  v ~ N(0,1);
  log_alpha = -softplus(z), z ~ N(-3,1)  (d=128 workloads), or
  log_alpha = log(sigmoid(z)), z ~ N(2,1) (tiny fp32 workload);
  beta = sigmoid(z), z ~ N(0,1).
Draw order: lengths, q, k, v, z_alpha, z_beta, S0.  Seed = 20260000 + index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    H: int
    d: int
    dtype: str                 # "bf16" or "fp32": dtype of q, k, v, o
    lengths: tuple = ()        # fixed lengths; empty => drawn (varlen)
    num_seqs: int = 1
    len_range: tuple = ()      # (lo, hi) inclusive, for drawn lengths
    gate: str = "softplus"     # "softplus": -softplus(N(-3,1)); "logsig": log sigmoid(N(2,1))
    q_scale: bool = True       # scale q by 1/sqrt(d)
    s0_std: float = 0.0        # 0 => no initial state (zeros)
    decode: bool = False

    @property
    def seed(self) -> int:
        return 20260000 + self.index


WORKLOADS = {
    1: Workload(1, "recurrent_tiny_fp32", H=1, d=16, dtype="fp32", lengths=(64,),
                gate="logsig", q_scale=False),
    2: Workload(2, "prefill_h16_t4096", H=16, d=128, dtype="bf16", lengths=(4096,)),
    3: Workload(3, "varlen16_h32", H=32, d=128, dtype="bf16", num_seqs=16,
                len_range=(512, 16384), s0_std=0.02),
    4: Workload(4, "prefill_h32_t1m", H=32, d=128, dtype="bf16", lengths=(1 << 20,)),
    5: Workload(5, "decode_1024x32", H=32, d=128, dtype="bf16", num_seqs=1024,
                lengths=(1,) * 1024, s0_std=0.02, decode=True),
}
BY_NAME = {w.name: w for w in WORKLOADS.values()}


def draw_lengths(w: Workload) -> list:
    if w.lengths:
        return list(w.lengths)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    lo, hi = w.len_range
    return torch.randint(lo, hi + 1, (w.num_seqs,), generator=g).tolist()


@dataclass
class Inputs:
    """One batch.  q, k, log_alpha: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H];
    S0: [N, H, d_k, d_v] fp32 or None; cu_seqlens: [N+1] int32;
    lengths: python list."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor
    beta: torch.Tensor
    S0: torch.Tensor | None
    cu_seqlens: torch.Tensor
    lengths: list = field(default_factory=list)

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)
        return Inputs(mv(self.q), mv(self.k), mv(self.v), mv(self.log_alpha),
                      mv(self.beta), mv(self.S0), mv(self.cu_seqlens),
                      list(self.lengths))


def _tdtype(name):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def generate(lengths, H, dk, dv, dtype="bf16", gate="softplus", q_scale=True,
             s0_std=0.0, seed=0, device="cpu", block_tokens=1 << 16,
             gate_shift=None):
    """Draw one batch of packed sequences.

    Tensors are drawn in blocks of ``block_tokens`` tokens from one seeded
    generator on ``device`` (bounded temporaries for very long inputs).
    ``gate_shift`` (optional float) replaces the gate draw by a constant
    log_alpha (stress cases such as the lower bound -5).
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T = int(sum(lengths))
    td = _tdtype(dtype)
    f32 = torch.float32
    q = torch.empty((T, H, dk), dtype=td, device=dev)
    k = torch.empty((T, H, dk), dtype=td, device=dev)
    v = torch.empty((T, H, dv), dtype=td, device=dev)
    g = torch.empty((T, H, dk), dtype=f32, device=dev)
    b = torch.empty((T, H), dtype=f32, device=dev)
    qs = 1.0 / math.sqrt(dk) if q_scale else 1.0
    for s in range(0, T, block_tokens):
        e = min(T, s + block_tokens)
        n = e - s
        q[s:e] = (torch.randn((n, H, dk), generator=gen, device=dev) * qs).to(td)
        kk = torch.randn((n, H, dk), generator=gen, device=dev)
        kk = kk / kk.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        k[s:e] = kk.to(td)
        v[s:e] = torch.randn((n, H, dv), generator=gen, device=dev).to(td)
        za = torch.randn((n, H, dk), generator=gen, device=dev)
        if gate_shift is not None:
            g[s:e] = float(gate_shift)
        elif gate == "softplus":
            g[s:e] = -torch.nn.functional.softplus(za - 3.0)
        elif gate == "logsig":
            g[s:e] = torch.nn.functional.logsigmoid(za + 2.0)
        else:
            raise ValueError(gate)
        b[s:e] = torch.sigmoid(torch.randn((n, H), generator=gen, device=dev))
    S0 = None
    if s0_std > 0:
        S0 = torch.randn((len(lengths), H, dk, dv), generator=gen, device=dev) * s0_std
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    return Inputs(q, k, v, g, b, S0, cu.to(torch.int32).to(dev), list(lengths))


def workload_inputs(w, device="cpu", **kw):
    """Inputs for one named workload (a Workload, its index or its name)."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    elif isinstance(w, str):
        w = BY_NAME[w]
    return generate(draw_lengths(w), w.H, w.d, w.d, dtype=w.dtype, gate=w.gate,
                    q_scale=w.q_scale, s0_std=w.s0_std, seed=w.seed,
                    device=device, **kw)
