"""KDA recurrent oracle: the delta rule with a per-key-channel (diagonal) decay
and the recurrent-state fake QDQ at chunk boundaries — numpy, fp64.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

Page "[1/4] GDN state/W QAT foundation", section "What does this PR do?":
differentiable GDN/KDA references for numerical validation, and "KDA has a
recurrent reference only"; page "[2/4] GDN/KDA decode QAT with INT8 recurrent
state" applies the same state quantizer (E4M3 or signed symmetric INT8,
per-head [Dk, block_v] scales) to KDA.  The pages print no KDA formula; the
reading used here is the published Kimi Delta Attention recurrence, which
differs from the gated delta rule only in the decay: alpha_t is a vector over
the Dk key channels (g_t = log alpha_t, one value per key channel), applied
to the rows of H = S^T:

    for t in the sequence (token index t from the sequence start):
        if t % chunk == 0:  H <- Q(H)              (fp32 QDQ per [Dk, block_v] tile)
        H <- diag(exp(g_t)) H
        H <- H + beta_t k_t (v_t - H^T k_t)^T
        o_t = scale H^T q_t

with the state QDQ at the same chunk boundaries as the GDN token recurrence
(h0 included, the final state returned unquantized).
"""
from __future__ import annotations

import numpy as np

from . import _np, qdq_groups


def kda_recurrent(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, state_mode="none",
                  block_v=64, chunk=64, record=None):
    """q, k [B, T, Hk, Dk]; v [B, T, Hv, Dv]; beta [B, T, Hv]; g [B, T, Hv, Dk] (log decay per
    key channel); h0 [N, Hv, Dk, Dv] or None; cu_seqlens [N + 1] or None (then B rows).

    Returns (o fp64 [B, T, Hv, Dv], ht fp64 [N, Hv, Dk, Dv]).  With a list as
    ``record``, (sequence, token offset, state [Hv, Dk, Dv] before the
    quantizer) is appended at every state QDQ; nothing else changes."""
    f64 = lambda x: np.asarray(_np(x), dtype=np.float32).astype(np.float64)
    q, k, v, beta, g = f64(q), f64(k), f64(v), f64(beta), f64(g)
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    if cu_seqlens is not None:
        cu = np.asarray(_np(cu_seqlens), dtype=np.int64)
        seqs = [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    else:
        seqs = [(b, 0, T) for b in range(B)]
    N = len(seqs)
    h0 = np.zeros((N, Hv, Dk, Dv)) if h0 is None else f64(h0)
    o = np.zeros((B, T, Hv, Dv))
    ht = np.zeros((N, Hv, Dk, Dv))
    for n, (b, t0, t1) in enumerate(seqs):
        H = h0[n].copy()                                            # [Hv, Dk, Dv]
        for t in range(t0, t1):
            if state_mode != "none" and (t - t0) % chunk == 0:
                if record is not None:
                    record.append((n, t - t0, H.copy()))
                H = qdq_groups(H.astype(np.float32), block_v, state_mode)[0].astype(np.float64)
            kt = k[b, t][np.arange(Hv) // G]                         # [Hv, Dk]
            qt = q[b, t][np.arange(Hv) // G]
            H = np.exp(g[b, t])[:, :, None] * H
            u = v[b, t] - np.einsum("hkv,hk->hv", H, kt)
            H = H + beta[b, t][:, None, None] * kt[:, :, None] * u[:, None, :]
            o[b, t] = scale * np.einsum("hkv,hk->hv", H, qt)
        ht[n] = H
    return o, ht
