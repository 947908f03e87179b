"""Seeded synthetic inputs for the SSD forward scan.

This module only draws random inputs with the shapes and value distributions of the five
workloads (Mamba-2-shaped layers); it holds none of the scan's arithmetic.  It is shared by the
tests, the benchmark and the smoke check; both the CUDA path and the CPU oracle consume the
same arrays.

Distributions (N(mu, s) read as mean mu and VARIANCE s):
  x  ~ N(0, 1)                               [b, L, H, P]
  dt = softplus(eps + bias_h), eps ~ N(0, 0.5) per (b, t, h); bias_h = softplus^-1(u_h) with
       u_h log-uniform on [dt_lo, dt_hi], one draw per head     [b, L, H]
  A_h = -exp(U(ln 1, ln 16))                 [H]  (fp32)
  B, C ~ N(0, 1 / d_state)                   [b, L, G, N]
  D  = 1, or N(1, 0.1) per head              [H]  (fp32)
  initial_state = none, or N(0, 0.1)         [b, H, P, N]  (fp32)
All draws are fp32 from one CPU torch.Generator (seed 1000 + config index unless given), taken
in a fixed order and in fixed token blocks, then cast to the compute dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import torch

_BLOCK_TOKENS = 4096   # draws are taken in blocks of this many tokens (fixes the stream order)


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str                 # "f32" or "bf16"
    dt_lo: float = 1e-3
    dt_hi: float = 1e-1
    d_mode: str = "ones"       # "ones" | "normal"
    h0_mode: str = "none"      # "none" | "normal"
    seed: int = 1000

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def describe(self) -> str:
        return (f"{self.name}: b={self.batch} L={self.seqlen} H={self.nheads} P={self.headdim} "
                f"N={self.dstate} G={self.ngroups} Q={self.chunk} {self.dtype}")

    def replace(self, **kw) -> "Workload":
        d = asdict(self)
        d.update(kw)
        return Workload(**d)


# The five workloads, restated from their definitions.
WORKLOADS = {
    0: Workload("tiny-fp32", 1, 256, 4, 32, 16, 1, 64, "f32", seed=1000),
    1: Workload("mamba2-130m-layer", 8, 2048, 24, 64, 128, 1, 256, "bf16", seed=1001),
    2: Workload("mamba2-2.7b-layer", 4, 4096, 80, 64, 128, 1, 256, "bf16", d_mode="normal",
                seed=1002),
    3: Workload("long-context-128k", 1, 131072, 80, 64, 128, 1, 256, "bf16", seed=1003),
    4: Workload("large-state-grouped", 2, 16384, 64, 128, 256, 8, 128, "bf16", dt_lo=1e-4,
                h0_mode="normal", seed=1004),
}


# Decoding: one token per sequence through the recurrent step (ssd_step_fwd), on the
# 2.7B-shaped layer's heads with a batch of 128 sequences (a float32 state of 335 MB, larger
# than L2), drawn from the same distributions with a random entering state.
DECODE = {
    0: Workload("decode-2.7b-b128", 128, 1, 80, 64, 128, 1, 1, "bf16", d_mode="normal",
                h0_mode="normal", seed=1100),
}


def _randn(gen, shape, std, block_axis=1):
    """fp32 normal draws, taken in fixed token blocks along ``block_axis``."""
    if len(shape) <= block_axis or shape[block_axis] <= _BLOCK_TOKENS:
        return torch.randn(shape, generator=gen, dtype=torch.float32) * std
    out = torch.empty(shape, dtype=torch.float32)
    L = shape[block_axis]
    for s in range(0, L, _BLOCK_TOKENS):
        e = min(L, s + _BLOCK_TOKENS)
        sl = [slice(None)] * len(shape)
        sl[block_axis] = slice(s, e)
        sub = list(shape)
        sub[block_axis] = e - s
        out[tuple(sl)] = torch.randn(sub, generator=gen, dtype=torch.float32) * std
    return out


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Draw one input set for workload ``w`` on the CPU.

    Returns a dict with x, dt, B, C (compute dtype), A, D (fp32 [H]) and h0 (fp32 or None).
    """
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    if H % G != 0:
        raise ValueError("nheads must be a multiple of ngroups")
    T = w.torch_dtype
    # per-head parameters first
    lo, hi = math.log(w.dt_lo), math.log(w.dt_hi)
    u = torch.exp(torch.rand(H, generator=gen, dtype=torch.float32) * (hi - lo) + lo)
    bias = torch.log(torch.expm1(u))                                 # softplus^-1(u)
    A = -torch.exp(torch.rand(H, generator=gen, dtype=torch.float32) * math.log(16.0))
    if w.d_mode == "ones":
        D = torch.ones(H, dtype=torch.float32)
    else:
        D = 1.0 + math.sqrt(0.1) * torch.randn(H, generator=gen, dtype=torch.float32)
    # per-token tensors
    x = _randn(gen, (b, L, H, P), 1.0).to(T)
    eps = _randn(gen, (b, L, H), math.sqrt(0.5))
    dt = torch.nn.functional.softplus(eps + bias).to(T)
    std_bc = 1.0 / math.sqrt(N)
    B = _randn(gen, (b, L, G, N), std_bc).to(T)
    C = _randn(gen, (b, L, G, N), std_bc).to(T)
    h0 = None
    if w.h0_mode == "normal":
        h0 = math.sqrt(0.1) * torch.randn((b, H, P, N), generator=gen, dtype=torch.float32)
    return dict(x=x, dt=dt, A=A.contiguous(), B=B, C=C, D=D.contiguous(), h0=h0)


def make_shape_inputs(batch, seqlen, nheads, headdim, dstate, ngroups=1, dtype="bf16",
                      seed=0, dt_lo=1e-3, dt_hi=1e-1, d_mode="ones", h0_mode="none") -> dict:
    """Inputs of an arbitrary shape with the same distributions (used for small test cases)."""
    w = Workload("custom", batch, seqlen, nheads, headdim, dstate, ngroups, 64, dtype,
                 dt_lo=dt_lo, dt_hi=dt_hi, d_mode=d_mode, h0_mode=h0_mode, seed=seed)
    return make_inputs(w)


# ---- the block steps around the scan ---------------------------------------------------------
# Causal conv1d over the scan's input channels of the 2.7B-shaped layer: x, B and C side by side
# (d_inner + 2 * ngroups * d_state = 5120 + 256 channels), width 4, b = 4, L = 4096.  Weights
# and bias uniform in +-1/sqrt(width) (the usual Conv1d initialisation), x ~ N(0, 1).
CONV = {"batch": 4, "seqlen": 4096, "channels": 5376, "width": 4, "dtype": "bf16", "seed": 1200}
# Gated RMSNorm over the scan's output of the same layer: rows = b * L = 16384 tokens,
# dim = nheads * headdim = 5120, one group; y, z ~ N(0, 1), weight 1 + N(0, 0.1).
NORM = {"rows": 16384, "dim": 5120, "group_size": 5120, "dtype": "bf16", "seed": 1300}


def make_conv_inputs(batch, seqlen, channels, width, dtype="bf16", seed=0, state=False) -> dict:
    gen = torch.Generator().manual_seed(seed)
    T = torch.float32 if dtype == "f32" else torch.bfloat16
    bound = 1.0 / math.sqrt(width)
    w = (torch.rand((channels, width), generator=gen) * 2 - 1) * bound
    bias = (torch.rand(channels, generator=gen) * 2 - 1) * bound
    x = _randn(gen, (batch, seqlen, channels), 1.0).to(T)
    st = None
    if state:
        st = torch.randn((batch, width - 1, channels), generator=gen).to(T)
    return dict(x=x, weight=w.contiguous(), bias=bias.contiguous(), state=st)


def make_norm_inputs(rows, dim, dtype="bf16", seed=0) -> dict:
    gen = torch.Generator().manual_seed(seed)
    T = torch.float32 if dtype == "f32" else torch.bfloat16
    y = torch.randn((rows, dim), generator=gen).to(T)
    z = torch.randn((rows, dim), generator=gen).to(T)
    w = 1.0 + math.sqrt(0.1) * torch.randn(dim, generator=gen)
    return dict(y=y, z=z, weight=w.contiguous())


# Packed variable-length batch on the 2.7B-shaped layer's heads: 24 sequences whose lengths are
# log-uniform in [64, 4096] (one draw from the seed), back to back in one row, each with its
# own initial state N(0, 0.1).
VARLEN = {"nseq": 24, "min_len": 64, "max_len": 4096, "nheads": 80, "headdim": 64,
          "dstate": 128, "ngroups": 1, "chunk": 256, "dtype": "bf16", "seed": 1400}


def varlen_lengths(nseq, min_len, max_len, seed) -> list:
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand(nseq, generator=gen, dtype=torch.float64)
    lo, hi = math.log(min_len), math.log(max_len)
    return [int(round(math.exp(lo + float(v) * (hi - lo)))) for v in u]


def make_varlen_inputs(lengths, nheads, headdim, dstate, ngroups=1, dtype="bf16", seed=0) -> dict:
    """One packed row of the given sequence lengths (inputs drawn like the scan workloads) plus
    cu_seqlens and per-sequence initial states."""
    total = int(sum(lengths))
    inp = make_shape_inputs(1, total, nheads, headdim, dstate, ngroups, dtype, seed=seed,
                            d_mode="normal")
    gen = torch.Generator().manual_seed(seed + 1)
    inp["h0"] = math.sqrt(0.1) * torch.randn((len(lengths), nheads, headdim, dstate),
                                             generator=gen, dtype=torch.float32)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    inp["cu_seqlens"] = cu
    return inp
