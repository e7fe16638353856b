"""Small-case fp64 token recurrence in torch, differentiable — TEST INFRASTRUCTURE ONLY.

The same gated delta rule as ``recurrent.c`` (H = S^T orientation):
    H <- exp(g_t) H;  H <- H + beta_t k_t (v_t - H^T k_t)^T;  o_t = scale H^T q_t
with the state fake QDQ (identity STE) applied to the carried state before
every token t of a sequence with t % chunk == 0, or, when ``quantize_before``
is given, before every token t for which it returns True (a decode after a
prefill of P tokens quantizes before t < P with t % 64 == 0 and before every
t >= P: page "[2/4] GDN/KDA decode QAT with INT8 recurrent state", sections
"What does this PR do?" and "Testing", split carry).  Plain Python loops over
tokens: meant for a few hundred tokens at most, to pin the chunked and decode
oracles against an independent formulation.
"""
from __future__ import annotations

import torch

from .chunked import qdq_ste


def recurrent_torch(q, k, v, beta, g, h0=None, scale=1.0, state_mode="none", chunk=64,
                    block_v=64, quantize_before=None):
    """q,k [B,T,Hk,Dk]; v [B,T,Hv,Dv]; beta,g [B,T,Hv]; h0 [B,Hv,Dk,Dv]; fp64."""
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    if h0 is None:
        h0 = torch.zeros(B, Hv, Dk, Dv, dtype=torch.float64)
    outs = []
    hts = []
    for b in range(B):
        ob = []
        hb = []
        for h in range(Hv):
            hk = h // G
            H = h0[b, h]
            oh = []
            for t in range(T):
                qt = quantize_before(t) if quantize_before is not None else t % chunk == 0
                if state_mode != "none" and qt:
                    H = qdq_ste(H[None], state_mode, block_v)[0]
                H = torch.exp(g[b, t, h]) * H
                kt = k[b, t, hk]
                u = v[b, t, h] - H.transpose(0, 1) @ kt
                H = H + beta[b, t, h] * torch.outer(kt, u)
                oh.append(scale * (H.transpose(0, 1) @ q[b, t, hk]))
            ob.append(torch.stack(oh, 0))
            hb.append(H)
        outs.append(torch.stack(ob, 1))
        hts.append(torch.stack(hb, 0))
    return torch.stack(outs, 0), torch.stack(hts, 0)
