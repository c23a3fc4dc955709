"""Seeded synthetic inputs for the KDA workloads.

This module holds no KDA arithmetic: it only draws random tensors in a fixed
order from a seeded CPU ``torch.Generator`` and rounds them to the storage
dtype.  Both the CUDA library's tests/benchmark and the CPU oracle read the
same host arrays produced here.

Recipe (shared by every workload):
  draw order q, k, v, z, beta-logits, A, S0 from ``torch.Generator().manual_seed(seed)``;
  q, k ~ N(0, 1) per element, then scaled to unit L2 norm per (token, head)
  in fp32;  v ~ N(0, 1);  z ~ N(0, 1) per channel;  beta = sigmoid(N(0, 1));
  A ~ N(0, 0.5) per head (0.5 is the standard deviation);  S0 = 0 or
  ~ N(0, 0.02) (standard deviation) when the workload asks for a nonzero
  initial state.  Values are then rounded to the storage dtype (RNE).
Variable-length workloads draw their sequence lengths first, from a separate
generator with the same seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    H: int
    d_k: int
    d_v: int
    dtype: torch.dtype
    seq_lens: tuple            # lengths of the packed sequences
    nonzero_state: bool = False
    final_state: bool = True

    @property
    def N(self) -> int:
        return len(self.seq_lens)

    @property
    def total_T(self) -> int:
        return int(sum(self.seq_lens))


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    d_k: int
    d_v: int
    dtype: torch.dtype
    steps: int


def varlen_lengths(n: int, lo: int, hi: int, seed: int = 0) -> tuple:
    """n integer lengths drawn uniformly from [lo, hi] (inclusive)."""
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


# The five workloads.  Shapes are (tokens, heads, head dim) as stated for each.
TINY_F32 = PrefillWorkload("tiny fp32 B=1 H=2 T=64 d=32", 2, 32, 32, torch.float32, (64,))
PREFILL_4K = PrefillWorkload("prefill bf16 B=1 H=32 T=4096 d=128", 32, 128, 128,
                             torch.bfloat16, (4096,))
PREFILL_64K = PrefillWorkload("long prefill bf16 B=1 H=96 T=65536 d=128", 96, 128, 128,
                              torch.bfloat16, (65536,))
VARLEN_16 = PrefillWorkload("varlen bf16 16 seqs U[512,16384] H=64 d=128", 64, 128, 128,
                            torch.bfloat16, varlen_lengths(16, 512, 16384, 0),
                            nonzero_state=True)
DECODE_256 = DecodeWorkload("decode B=256 H=96 d=128 fp32 state, bf16 inputs", 256, 96,
                            128, 128, torch.bfloat16, 64)

WORKLOADS = {w.name: w for w in (TINY_F32, PREFILL_4K, PREFILL_64K, VARLEN_16)}


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


@dataclass
class PrefillInputs:
    q: torch.Tensor          # [total_T, H, d_k] storage dtype
    k: torch.Tensor
    v: torch.Tensor          # [total_T, H, d_v]
    z: torch.Tensor          # [total_T, H, d_k]
    beta: torch.Tensor       # [total_T, H]
    A: torch.Tensor          # [H] fp32
    initial_state: Optional[torch.Tensor]  # [N, H, d_k, d_v] fp32 or None
    cu_seqlens: torch.Tensor  # [N + 1] int32
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "PrefillInputs":
        mv = lambda t: None if t is None else t.to(device, non_blocking=True)
        return PrefillInputs(mv(self.q), mv(self.k), mv(self.v), mv(self.z), mv(self.beta),
                             mv(self.A), mv(self.initial_state), mv(self.cu_seqlens), self.extra)


def make_prefill_inputs(seq_lens, H: int, d_k: int, d_v: int, dtype: torch.dtype,
                        seed: int = 0, nonzero_state: bool = False) -> PrefillInputs:
    """Draw one packed prefill batch on the host (see the module docstring)."""
    seq_lens = [int(s) for s in seq_lens]
    T = int(sum(seq_lens))
    g = torch.Generator().manual_seed(seed)
    q = _unit_rows(torch.randn(T, H, d_k, generator=g)).to(dtype)
    k = _unit_rows(torch.randn(T, H, d_k, generator=g)).to(dtype)
    v = torch.randn(T, H, d_v, generator=g).to(dtype)
    z = torch.randn(T, H, d_k, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(T, H, generator=g)).to(dtype)
    A = (0.5 * torch.randn(H, generator=g)).float()
    S0 = None
    if nonzero_state:
        S0 = (0.02 * torch.randn(len(seq_lens), H, d_k, d_v, generator=g)).float()
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    if seq_lens:
        cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(q, k, v, z, beta, A, S0, cu)


def make_workload_inputs(w: PrefillWorkload, seed: int = 0) -> PrefillInputs:
    return make_prefill_inputs(w.seq_lens, w.H, w.d_k, w.d_v, w.dtype, seed, w.nonzero_state)


@dataclass
class DecodeStepInputs:
    q: torch.Tensor     # [B, H, d_k]
    k: torch.Tensor
    v: torch.Tensor     # [B, H, d_v]
    z: torch.Tensor
    beta: torch.Tensor  # [B, H]

    def to(self, device) -> "DecodeStepInputs":
        return DecodeStepInputs(*(t.to(device, non_blocking=True)
                                  for t in (self.q, self.k, self.v, self.z, self.beta)))


def make_decode_state(B: int, H: int, d_k: int, d_v: int, seed: int = 0):
    """A [H] ~ N(0, 0.5) and the resident state [B, H, d_k, d_v] ~ N(0, 0.02)."""
    g = torch.Generator().manual_seed(seed)
    A = (0.5 * torch.randn(H, generator=g)).float()
    S = (0.02 * torch.randn(B, H, d_k, d_v, generator=g)).float()
    return A, S


def make_decode_step(B: int, H: int, d_k: int, d_v: int, dtype: torch.dtype,
                     seed: int = 0, step: int = 0) -> DecodeStepInputs:
    """Per-step token inputs, drawn with seed + 1 + step (order q, k, v, z, beta)."""
    g = torch.Generator().manual_seed(seed + 1 + step)
    q = _unit_rows(torch.randn(B, H, d_k, generator=g)).to(dtype)
    k = _unit_rows(torch.randn(B, H, d_k, generator=g)).to(dtype)
    v = torch.randn(B, H, d_v, generator=g).to(dtype)
    z = torch.randn(B, H, d_k, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(B, H, generator=g)).to(dtype)
    return DecodeStepInputs(q, k, v, z, beta)


def make_conv_params(N: int, H: int, d_k: int, d_v: int, W: int, dtype: torch.dtype,
                     seed: int = 0, with_state: bool = True):
    """Short-convolution weights [H, 2 d_k + d_v, W] fp32 ~ N(0, 0.5) and a
    conv state [N, H, W-1, 2 d_k + d_v] in `dtype` (or None): N(0, 1) draws,
    the q and k channels scaled by 1 / sqrt(d_k) to the size of unit-norm
    rows.  Drawn in that order from generator(seed + 7)."""
    g = torch.Generator().manual_seed(seed + 7)
    Cc = 2 * d_k + d_v
    w = (0.5 * torch.randn(H, Cc, W, generator=g)).float()
    state = None
    if with_state:
        state = torch.randn(N, H, W - 1, Cc, generator=g)
        state[..., :2 * d_k] *= d_k ** -0.5
        state = state.to(dtype)
    return w, state


def make_upstream_grads(total_T: int, N: int, H: int, d_k: int, d_v: int, dtype: torch.dtype,
                        seed: int = 0, with_state: bool = True):
    """Upstream gradients for the backward: dO [total_T, H, d_v] ~ N(0, 1) in
    `dtype` and dL/dS_T [N, H, d_k, d_v] ~ N(0, 0.1) fp32 (or None), drawn in
    that order from generator(seed + 13)."""
    g = torch.Generator().manual_seed(seed + 13)
    dO = torch.randn(total_T, H, d_v, generator=g).to(dtype)
    dSf = (0.1 * torch.randn(N, H, d_k, d_v, generator=g)).float() if with_state else None
    return dO, dSf


def list_workloads() -> List[str]:
    return list(WORKLOADS) + [DECODE_256.name]
