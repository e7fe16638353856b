"""Seeded synthetic inputs for the chunked gated delta rule (no method arithmetic here).

Both the CUDA path and the CPU oracle are fed from these generators, so they
see identical bf16 / fp32 bits.  Recipe (drawn on the CPU with a
``torch.Generator`` seeded per workload, in this order):
  q, k  ~ N(0, 1), L2-normalised over the head dimension in fp32, then cast to bf16
  v     ~ N(0, 1) cast to bf16
  beta  = sigmoid(N(0, 1))            fp32   (write strength in (0, 1))
  g     = -softplus(N(0, 1))          fp32   (log-decay, alpha = exp(g) in (0, 1))
  h0    ~ N(0, 0.1^2) fp32 where the workload has an initial state, else absent
  dO    ~ N(0, 1) bf16;  dht ~ N(0, 0.01^2) fp32   (backward workloads)
Packed variable-length workloads draw sequence lengths with
``numpy.random.default_rng(seed)``: while more than ``hi`` tokens remain,
append L uniform in [lo, min(hi, remaining - lo)]; then append the rest.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    state_mode: str = "e4m3"
    w_mode: str = "e4m3"
    h0: bool = False
    varlen_total: int = 0          # > 0: packed sequences, B == 1, T == total
    varlen_lo: int = 97
    varlen_hi: int = 4096
    backward: bool = False
    scale: float = 1.0
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads of the method's validation plan, by what they are.
WORKLOADS = {
    "tiny": Workload("tiny B1 T128 H2 D64 e4m3", B=1, T=128, Hk=2, Hv=2, Dk=64, Dv=64),
    "layer": Workload("single layer B4 T4096 H16 D128 e4m3", B=4, T=4096, Hk=16, Hv=16,
                      Dk=128, Dv=128, h0=True),
    "grouped_int8": Workload("grouped heads B2 T8192 Hk16 Hv32 D128 int8-state", B=2, T=8192,
                             Hk=16, Hv=32, Dk=128, Dv=128, state_mode="int8", h0=True),
    "varlen": Workload("packed varlen 32768 tokens H32 D128 e4m3", B=1, T=32768, Hk=32,
                       Hv=32, Dk=128, Dv=128, varlen_total=32768),
    "fwd_bwd": Workload("fwd+bwd B8 T4096 H16 D128 e4m3", B=8, T=4096, Hk=16, Hv=16,
                        Dk=128, Dv=128, h0=True, backward=True),
    # one sequence of the single layer: the small case the detailed counter
    # captures run on (inputs and gradients still larger than L2)
    "layer_b1": Workload("single layer B1 T4096 H16 D128 e4m3", B=1, T=4096, Hk=16, Hv=16,
                         Dk=128, Dv=128, h0=True, seed=5),
    # decode QAT: one token per sequence for 256 sequences whose carried states
    # (256 x 16 x 128 x 128 fp32 = 256 MiB) exceed L2
    "decode": Workload("decode step B256 T1 H16 D128 e4m3-state", B=256, T=1, Hk=16, Hv=16,
                       Dk=128, Dv=128, h0=True, seed=5),
    # KDA recurrence (per-key-channel decay), state QDQ every 64 tokens
    "kda": Workload("KDA recurrent B4 T4096 H16 D128 e4m3-state", B=4, T=4096, Hk=16, Hv=16,
                    Dk=128, Dv=128, w_mode="none", h0=True, seed=6),
    # two-precision profile: fp32 anchor, E4M3 read copy (state_mode names the
    # read quantizer), 16-token flushes
    "two_precision": Workload("two-precision B4 T4096 H16 D128 e4m3-read flush16", B=4, T=4096,
                              Hk=16, Hv=16, Dk=128, Dv=128, w_mode="none", h0=True, seed=7),
    # the same launch shape on shorter sequences: the small case of the detailed
    # counter captures of the two-precision kernels
    "two_precision_t1k": Workload("two-precision B4 T1024 H16 D128 e4m3-read flush16", B=4,
                                  T=1024, Hk=16, Hv=16, Dk=128, Dv=128, w_mode="none", h0=True,
                                  seed=7),
}


def varlen_lengths(total: int, lo: int = 97, hi: int = 4096, seed: int = 0):
    rng = np.random.default_rng(seed)
    out = []
    rem = total
    while rem > hi:
        L = int(rng.integers(lo, min(hi, rem - lo) + 1))
        out.append(L)
        rem -= L
    out.append(rem)
    return out


def cu_seqlens_of(lengths):
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    return torch.from_numpy(cu)


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(w: Workload, lengths=None, device="cpu"):
    """Return a dict of CPU tensors (moved to ``device`` at the end)."""
    gen = torch.Generator().manual_seed(w.seed)
    B, T = w.B, w.T
    cu = None
    if w.varlen_total or lengths is not None:
        if lengths is None:
            lengths = varlen_lengths(w.varlen_total, w.varlen_lo, w.varlen_hi, w.seed)
        cu = cu_seqlens_of(lengths)
        B, T = 1, int(cu[-1])
    N = B if cu is None else len(lengths)
    rn = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float32)
    q = _l2n(rn(B, T, w.Hk, w.Dk)).to(torch.bfloat16)
    k = _l2n(rn(B, T, w.Hk, w.Dk)).to(torch.bfloat16)
    v = rn(B, T, w.Hv, w.Dv).to(torch.bfloat16)
    beta = torch.sigmoid(rn(B, T, w.Hv))
    g = -torch.nn.functional.softplus(rn(B, T, w.Hv))
    h0 = rn(N, w.Hv, w.Dk, w.Dv) * 0.1 if w.h0 else None
    d = dict(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu, N=N, B=B, T=T)
    if w.backward:
        d["do"] = rn(B, T, w.Hv, w.Dv).to(torch.bfloat16)
        d["dht"] = rn(N, w.Hv, w.Dk, w.Dv) * 0.01
    if device != "cpu":
        for key, val in list(d.items()):
            if isinstance(val, torch.Tensor):
                d[key] = val.to(device)
    return d


def make_kda_inputs(w: Workload, lengths=None, device="cpu"):
    """make_inputs plus the per-key-channel log decay g_k [B, T, Hv, Dk] of the
    KDA recurrence, -softplus(N(0, 1)) per channel (its own seeded stream)."""
    d = make_inputs(w, lengths=lengths)
    gen = torch.Generator().manual_seed(w.seed + 7919)
    B, T = d["B"], d["T"]
    d["g_k"] = -torch.nn.functional.softplus(
        torch.randn(B, T, w.Hv, w.Dk, generator=gen, dtype=torch.float32))
    if device != "cpu":
        for key, val in list(d.items()):
            if isinstance(val, torch.Tensor):
                d[key] = val.to(device)
    return d


def small(name="small", B=1, T=200, Hk=2, Hv=2, Dk=64, Dv=64, **kw) -> Workload:
    """An ad-hoc workload for parity tests."""
    return Workload(name, B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, **kw)
