"""Seeded synthetic inputs for the KDA forward workloads.

This module holds only random draws and the workload recipe; none of the
method's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle get
their inputs from here, as identical bytes.

Recipe (one ``torch.Generator`` on the CPU, seeded per workload; draws in this
fixed order: [varlen lengths], q, k, v, g, beta, A_log, dt_bias, initial_state):

* q, k ~ N(0, 1) in fp32, L2-normalised per (token, head) vector, then bf16
  (``raw_qk=True`` keeps the raw N(0, 1) draws, for the in-kernel normalisation);
* v, g, beta logits ~ N(0, 1), then bf16;
* A_log ~ U(0, ln 16) fp32 ``[H]``; dt_bias ~ N(0, 0.1^2) fp32 ``[H, 128]``;
* initial_state ~ N(0, 0.02^2) in its stated dtype;
* varlen lengths ~ U{1..8192}; a draw that is a multiple of 16 gets -1, so
  every sequence ends in a ragged chunk.

Shapes follow the tensor contract of "FlashKDA Input Tensor Shapes and DTypes:
Complete Specification for the Forward Pass" (q, k, v, g ``[B, T, H, 128]`` bf16,
beta ``[B, T, H]`` bf16, fp32 gating parameters, states ``[B|N, H, 128, 128]``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    lower_bound: float
    gate_params: bool              # A_log / dt_bias given (else None)
    init_dtype: Optional[str]      # "fp32" | "bf16" | None
    final_dtype: Optional[str]     # "fp32" | "bf16" | None
    seed: int
    varlen_n: int = 0              # N sequences (B == 1) or 0
    varlen_max: int = 8192
    scale: float = 1.0 / math.sqrt(128.0)


WORKLOADS = {
    # small case: one head, four chunks
    "b1_t64_h1": Workload("b1_t64_h1", 1, 64, 1, -5.0, True, None, "fp32", seed=0),
    # state carry case (also run as two 64-token calls)
    "b2_t128_h8": Workload("b2_t128_h8", 2, 128, 8, -2.0, True, "fp32", "fp32", seed=1),
    # the throughput case
    "b8_t4096_h16": Workload("b8_t4096_h16", 8, 4096, 16, -5.0, False, None, "fp32", seed=2),
    # packed variable-length sequences
    "varlen_n16_h32": Workload("varlen_n16_h32", 1, 0, 32, -5.0, True, "bf16", "bf16", seed=3,
                               varlen_n=16),
    # long context: few states, long chain
    "b1_t131072_h32": Workload("b1_t131072_h32", 1, 131072, 32, -5.0, True, "fp32", "fp32", seed=4),
}
ORDER = ["b1_t64_h1", "b2_t128_h8", "b8_t4096_h16", "varlen_n16_h32", "b1_t131072_h32"]

_DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def varlen_lengths(gen: torch.Generator, n: int, max_len: int):
    lens = torch.randint(1, max_len + 1, (n,), generator=gen, dtype=torch.int64)
    lens = torch.where(lens % 16 == 0, lens - 1, lens)
    return lens


def make(w, seed: Optional[int] = None, T: Optional[int] = None, H: Optional[int] = None,
         B: Optional[int] = None, lengths=None, raw_qk: bool = False) -> dict:
    """Build the CPU tensors of a workload (by name or ``Workload``).

    ``T``/``H``/``B``/``lengths`` override the shape for reduced parity cases;
    ``lengths`` (a list) makes a varlen case; ``raw_qk`` skips the L2 normalisation
    of q and k (same random draws). Returns a dict with keys ``q k v g
    beta A_log dt_bias initial_state cu_seqlens scale lower_bound final_dtype``.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B = w.B if B is None else B
    H = w.H if H is None else H
    cu = None
    if lengths is not None or w.varlen_n:
        if lengths is None:
            lens = varlen_lengths(gen, w.varlen_n, w.varlen_max)
        else:
            lens = torch.tensor(list(lengths), dtype=torch.int64)
        cu = torch.zeros(lens.numel() + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        B, T = 1, int(cu[-1])
    else:
        T = w.T if T is None else T
    D = HEAD_DIM
    nrm = (lambda x: x) if raw_qk else _l2n
    q = nrm(torch.randn(B, T, H, D, generator=gen)).to(torch.bfloat16)
    k = nrm(torch.randn(B, T, H, D, generator=gen)).to(torch.bfloat16)
    v = torch.randn(B, T, H, D, generator=gen).to(torch.bfloat16)
    g = torch.randn(B, T, H, D, generator=gen).to(torch.bfloat16)
    beta = torch.randn(B, T, H, generator=gen).to(torch.bfloat16)
    A_log = dt_bias = None
    if w.gate_params:
        A_log = torch.rand(H, generator=gen) * math.log(16.0)
        dt_bias = torch.randn(H, D, generator=gen) * 0.1
    init = None
    nseq = (cu.numel() - 1) if cu is not None else B
    if w.init_dtype:
        init = (torch.randn(nseq, H, D, D, generator=gen) * 0.02).to(_DT[w.init_dtype])
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                initial_state=init, cu_seqlens=cu, scale=w.scale,
                lower_bound=w.lower_bound, final_dtype=w.final_dtype)


def bf16_bits(t: torch.Tensor):
    """The raw 16-bit patterns of a bf16 CPU tensor, as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def state_f64(t: Optional[torch.Tensor]):
    """Exact float64 copy of a bf16/fp32 state tensor (or None)."""
    return None if t is None else t.float().double().numpy()
