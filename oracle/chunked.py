"""O2: chunked (WY) gated delta rule with state and W fake QDQ — torch CPU, fp64.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

Follows the chunked training form that the GatedDeltaNet QAT pages quantize
("[1/4] GDN state/W QAT foundation", section "What does this PR do?": chunk
size 64, dynamic E4M3 fake QDQ at the state and W sites, identity STE, the
triangular solve stays exact, the quantized W is the one saved for backward;
section Usage: `gdn_state_quantizer` with `axis (0, 1)` and `state.block_v
64`, `gdn_w_quantizer` with `axis (0, 1, 2)`; "[2/4] GDN/KDA decode QAT with
INT8 recurrent state": INT8 variant with per-head [Dk, block_v] scales).

The pages print no equations.  For one sequence and value head, with H the
Dk x Dv state (H = S^T) entering a chunk of L <= 64 tokens, the steps are the
published WY form of the gated delta rule, taken in this order:

  a1  gamma_i = sum_{s <= i} g_s                      (restarts every chunk)
  a2  A_ij    = beta_i exp(gamma_i - gamma_j) k_i.k_j  for i > j, else 0
  a3  T       = (I + A)^-1                         (exact triangular solve)
  a4  W       = T diag(beta * exp(gamma)) K,   U = T diag(beta) V
  a5  W^      = Q_W(W)        one scale over the whole [L, Dk] tile
  a6  H^      = Q_S(H)        one scale per [Dk, block_v] column tile
  a7  Delta   = U - W^ H^
  a8  O       = scale * (diag(exp(gamma)) Q H^ + (Gamma (.) Q K^T, lower incl. diag) Delta)
  a9  H_next  = exp(gamma_L) H^ + (diag(exp(gamma_L - gamma)) K)^T Delta

Q_W / Q_S are the fp32 QDQ of ``oracle/qdq.c`` (the state/W are rounded to
fp32 first).  Gradients come from torch autograd of this graph, with every
QDQ written as x + (Q(x) - x).detach(): the identity straight-through
estimator.  The final state H after the last chunk is returned unquantized.
Value head h reads query/key head h // (Hv / Hk).
"""
from __future__ import annotations

import numpy as np
import torch

from . import qdq_groups


def qdq_ste(x: torch.Tensor, mode: str, group_cols: int, record=None):
    """Fake QDQ with identity STE of x [batch, rows, cols] (fp64).

    One scale per (batch, block of group_cols columns) over all rows.
    """
    if mode == "none":
        return x
    xf = x.detach().to(torch.float32).numpy()
    y, sc, cd = qdq_groups(xf, group_cols, mode, with_codes=True)
    if record is not None:
        record.append((cd, sc))
    y = torch.from_numpy(y).to(torch.float64)
    return x + (y - x).detach()


def neumann_inverse(A, degree):
    """T = sum_{i=0..degree} (-A)^i, the Neumann polynomial for (I + A)^-1 of a
    strictly lower-triangular A ("[7/7] Experimental GDN/KDA approximate-inverse
    QAT", "What does this PR do?": an explicit polynomial degree, the backward
    differentiating the actual polynomial).  Exact once degree >= L - 1."""
    L = A.shape[-1]
    eye = torch.eye(L, dtype=A.dtype).expand(A.shape)
    T, Xp = eye, eye
    for _ in range(degree):
        Xp = Xp @ (-A)
        T = T + Xp
    return T


def _chunk_step(Qc, Kc, Vc, bc, gc, H, scale, state_mode, w_mode, block_v, rec, inter,
                neumann_degree=None):
    """One chunk for a batch of value-head problems. Qc,Kc [S,L,Dk]; Vc [S,L,Dv];
    bc,gc [S,L]; H [S,Dk,Dv].  Returns (O [S,L,Dv], H_next)."""
    S, L, Dk = Kc.shape
    dt = Kc.dtype
    gam = torch.cumsum(gc, dim=-1)                                    # a1
    le = torch.tril(torch.ones(L, L, dtype=torch.bool))
    strict = torch.tril(torch.ones(L, L, dtype=torch.bool), diagonal=-1)
    diff = gam[:, :, None] - gam[:, None, :]
    Gam = torch.where(le, torch.exp(torch.where(le, diff, torch.zeros((), dtype=dt))),
                      torch.zeros((), dtype=dt))
    KK = Kc @ Kc.transpose(-1, -2)
    A = torch.where(strict, bc[:, :, None] * Gam * KK, torch.zeros((), dtype=dt))  # a2
    eye = torch.eye(L, dtype=dt).expand(S, L, L)
    if neumann_degree is None:
        T = torch.linalg.solve_triangular(eye + A, eye, upper=False, unitriangular=True)  # a3
    else:
        T = neumann_inverse(A, neumann_degree)
    W = T @ ((bc * torch.exp(gam))[:, :, None] * Kc)                  # a4
    U = T @ (bc[:, :, None] * Vc)
    Wh = qdq_ste(W, w_mode, Dk, rec["w"] if rec is not None else None)      # a5
    Hh = qdq_ste(H, state_mode, block_v, rec["s"] if rec is not None else None)  # a6
    Delta = U - Wh @ Hh                                               # a7
    P = torch.where(le, Gam * (Qc @ Kc.transpose(-1, -2)), torch.zeros((), dtype=dt))
    O = scale * (torch.exp(gam)[:, :, None] * (Qc @ Hh) + P @ Delta)  # a8
    gL = gam[:, -1]
    Kd = Kc * torch.exp(gL[:, None] - gam)[:, :, None]
    Hn = torch.exp(gL)[:, None, None] * Hh + Kd.transpose(-1, -2) @ Delta  # a9
    if inter is not None:
        inter.append(dict(gamma=gam, A=A, T=T, W=W, U=U, W_hat=Wh, H=H, H_hat=Hh,
                          Delta=Delta))
    return O, Hn


def _run_equal(q, k, v, beta, g, h0, scale, state_mode, w_mode, chunk, block_v, rec, inter,
               neumann_degree=None):
    """Equal-length batch. q,k [S,L,Hk,Dk]; v [S,L,Hv,Dv]; beta,g [S,L,Hv]; h0 [S,Hv,Dk,Dv]."""
    S, L, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    idx = torch.arange(Hv) // G
    # value-head views: [S*Hv, L, D]
    qv = q[:, :, idx, :].permute(0, 2, 1, 3).reshape(S * Hv, L, Dk)
    kv = k[:, :, idx, :].permute(0, 2, 1, 3).reshape(S * Hv, L, Dk)
    vv = v.permute(0, 2, 1, 3).reshape(S * Hv, L, Dv)
    bv = beta.permute(0, 2, 1).reshape(S * Hv, L)
    gv = g.permute(0, 2, 1).reshape(S * Hv, L)
    H = h0.reshape(S * Hv, Dk, Dv)
    outs = []
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        O, H = _chunk_step(qv[:, c0:c1], kv[:, c0:c1], vv[:, c0:c1], bv[:, c0:c1],
                           gv[:, c0:c1], H, scale, state_mode, w_mode, block_v, rec, inter,
                           neumann_degree)
        outs.append(O)
    o = torch.cat(outs, dim=1) if outs else vv.new_zeros(S * Hv, 0, Dv)
    o = o.reshape(S, Hv, L, Dv).permute(0, 2, 1, 3)
    return o, H.reshape(S, Hv, Dk, Dv)


def chunked(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, state_mode="none",
            w_mode="none", chunk=64, block_v=64, record=False, intermediates=False,
            neumann_degree=None):
    """O2.  Tensors are torch CPU; they are used in fp64 (bf16 widens exactly).
    ``neumann_degree`` replaces the exact solve by the Neumann polynomial of that
    degree (see neumann_inverse).

    q, k [B,T,Hk,Dk]; v [B,T,Hv,Dv]; beta, g [B,T,Hv]; h0 [N,Hv,Dk,Dv] or None;
    cu_seqlens [N+1] (B == 1) or None.  Differentiable in every float input.

    Returns (o [B,T,Hv,Dv], ht [N,Hv,Dk,Dv]) and, with ``record``, a dict of
    per-chunk numpy records, chunks numbered densely (sequence after sequence):
      state_codes [nc,Hv,Dk,Dv] u8, state_scales [nc,Hv,Dv/block_v],
      w_codes: list over sequences of [L,Hv,Dk] u8, w_scales [nc,Hv]
    With ``intermediates``, a list (per sequence) of per-chunk dicts of tensors.
    """
    d = lambda t: None if t is None else (t if t.dtype == torch.float64 else t.to(torch.float64))
    q, k, v, beta, g, h0 = d(q), d(k), d(v), d(beta), d(g), d(h0)
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    if cu_seqlens is None:
        N = B
        seqs = [(None, T)]
    else:
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        N = len(cu) - 1
        seqs = [(n, cu[n + 1] - cu[n]) for n in range(N)]
    if h0 is None:
        h0 = torch.zeros(N, Hv, Dk, Dv, dtype=torch.float64)
    recs, inters = [], []
    if cu_seqlens is None:
        rec = {"w": [], "s": []} if record else None
        inter = [] if intermediates else None
        o, ht = _run_equal(q, k, v, beta, g, h0, scale, state_mode, w_mode, chunk, block_v,
                           rec, inter, neumann_degree)
        recs.append((rec, B, T))
        inters.append(inter)
    else:
        os_, hts = [], []
        for n, L in seqs:
            sl = slice(cu[n], cu[n + 1])
            rec = {"w": [], "s": []} if record else None
            inter = [] if intermediates else None
            o_n, h_n = _run_equal(q[:, sl], k[:, sl], v[:, sl], beta[:, sl], g[:, sl],
                                  h0[n:n + 1], scale, state_mode, w_mode, chunk, block_v,
                                  rec, inter, neumann_degree)
            os_.append(o_n)
            hts.append(h_n)
            recs.append((rec, 1, L))
            inters.append(inter)
        o = torch.cat(os_, dim=1)
        ht = torch.cat(hts, dim=0)
    out = (o, ht)
    if record:
        out = out + (_collect(recs, Hv, Dk, Dv, chunk, block_v, state_mode, w_mode),)
    if intermediates:
        out = out + (inters,)
    return out


def _collect(recs, Hv, Dk, Dv, chunk, block_v, state_mode, w_mode):
    """Reorder per-step records (each over [S*Hv] problems) into dense chunk order."""
    sc_codes, sc_scales, w_codes, w_scales = [], [], [], []
    for rec, S, L in recs:
        nchk = -(-L // chunk)
        if nchk == 0:        # an empty sequence has no chunk boundary and no W tile
            continue
        if state_mode != "none":
            # rec["s"][c] = (codes [S*Hv,Dk,Dv], scales [S*Hv, Dv/block_v])
            cds = np.stack([c for c, _ in rec["s"]], 0).reshape(nchk, S, Hv, Dk, Dv)
            scs = np.stack([s for _, s in rec["s"]], 0).reshape(nchk, S, Hv, Dv // block_v)
            sc_codes.append(cds.transpose(1, 0, 2, 3, 4).reshape(S * nchk, Hv, Dk, Dv))
            sc_scales.append(scs.transpose(1, 0, 2, 3).reshape(S * nchk, Hv, Dv // block_v))
        if w_mode != "none":
            # rec["w"][c] = (codes [S*Hv,Lc,Dk], scales [S*Hv,1])
            for s in range(S):
                per = []
                for c in range(nchk):
                    cd, sc = rec["w"][c]
                    cd = cd.reshape(S, Hv, -1, Dk)[s]          # [Hv, Lc, Dk]
                    per.append(cd.transpose(1, 0, 2))          # [Lc, Hv, Dk]
                    w_scales.append(sc.reshape(S, Hv)[s])
                w_codes.append(np.concatenate(per, 0))
    out = {}
    if state_mode != "none" and sc_codes:
        out["state_codes"] = np.concatenate(sc_codes, 0)
        out["state_scales"] = np.concatenate(sc_scales, 0)
    if w_mode != "none" and w_codes:
        out["w_codes"] = w_codes
        out["w_scales"] = np.stack(w_scales, 0)
    return out
