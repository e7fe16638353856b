"""Decode QAT oracle: one gated delta rule step per token with state QDQ — numpy, fp64.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

Page "[2/4] GDN/KDA decode QAT with INT8 recurrent state", section "What does
this PR do?": an explicit prefix length selects an exact chunked prefill, and
the tokens after it are "token-state writes" — the recurrent state passes
through the state quantizer (E4M3, or signed symmetric INT8 with per-head
[Dk, block_v] scales) at every token instead of every 64-token chunk.  Section
"Testing" asks for both readouts and for the split carry (the prefill's final
state chained into decode).  The page prints no formula; the reading used here
is the chunk-boundary rule of the chunked forward with a chunk of one token
(H = S^T, Dk x Dv, the carried state S arriving unquantized, exactly like the
final state ``ht`` of a prefill):

    S^  = Q(S)                                   (fp32 QDQ per [Dk, block_v] tile)
    H   = exp(g) S^ + beta k (v - exp(g) S^^T k)^T
    o   = scale H^T q          readout "pre"  (as inside a chunk of the forward)
        = scale Q(H)^T q       readout "post" (the state the next token reads)
    S  <- H                    (carried unquantized; the next token quantizes it)

so a call over T tokens equals T calls of one token chained through S, and a
prefill followed by decode equals the token recurrence whose state is
quantized before tokens t % 64 == 0 of the prefix and before every token
after it.
"""
from __future__ import annotations

import numpy as np

from . import _np, qdq_groups


def _q(H, mode, block_v):
    """Fake QDQ of fp64 states [B, Hv, Dk, Dv] after rounding to fp32 (qdq.c)."""
    B, Hv, Dk, Dv = H.shape
    y, sc, cd = qdq_groups(H.astype(np.float32).reshape(B * Hv, Dk, Dv), block_v, mode,
                           with_codes=True)
    return (y.reshape(B, Hv, Dk, Dv).astype(np.float64), sc.reshape(B, Hv, Dv // block_v),
            cd.reshape(B, Hv, Dk, Dv))


def decode(q, k, v, beta, g, state_in, scale=1.0, state_mode="e4m3", block_v=64,
           readout="pre", record=False):
    """q, k [B, T, Hk, Dk]; v [B, T, Hv, Dv]; beta, g [B, T, Hv]; state_in [B, Hv, Dk, Dv].

    Returns (o fp64 [B, T, Hv, Dv], state_out fp64 [B, Hv, Dk, Dv]) and, with
    ``record`` and a quantizing mode, (codes u8 [B, T, Hv, Dk, Dv],
    scales fp32 [B, T, Hv, Dv / block_v]) of the quantized state each token read.
    """
    if readout not in ("pre", "post"):
        raise ValueError("readout must be 'pre' or 'post'")
    q, k, v = (np.asarray(_np(x), dtype=np.float32).astype(np.float64) for x in (q, k, v))
    beta, g = (np.asarray(_np(x), dtype=np.float32).astype(np.float64) for x in (beta, g))
    S = np.asarray(_np(state_in), dtype=np.float32).astype(np.float64)
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    heads = np.arange(Hv) // (Hv // Hk)
    quant = state_mode != "none"
    o = np.zeros((B, T, Hv, Dv))
    codes = np.zeros((B, T, Hv, Dk, Dv), np.uint8) if (record and quant) else None
    scales = np.zeros((B, T, Hv, Dv // block_v), np.float32) if (record and quant) else None
    for t in range(T):
        kt, qt = k[:, t][:, heads], q[:, t][:, heads]             # [B, Hv, Dk]
        if quant:
            Sq, sc, cd = _q(S, state_mode, block_v)
            if codes is not None:
                codes[:, t], scales[:, t] = cd, sc
        else:
            Sq = S
        Sa = np.exp(g[:, t])[:, :, None, None] * Sq
        u = v[:, t] - np.einsum("bhkv,bhk->bhv", Sa, kt)
        H = Sa + beta[:, t][:, :, None, None] * kt[:, :, :, None] * u[:, :, None, :]
        R = _q(H, state_mode, block_v)[0] if (readout == "post" and quant) else H
        o[:, t] = scale * np.einsum("bhkv,bhk->bhv", R, qt)
        S = H
    if record:
        return o, S, codes, scales
    return o, S
