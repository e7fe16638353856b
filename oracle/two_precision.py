"""Two-precision GDN oracle: an fp32 recurrence anchor and a dynamic E4M3 read
copy that only the outputs see — numpy, fp64.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

Page "[5/8] ReplaySSM state QAT and two-precision GDN", section "What does this
PR do?": the profile keeps an FP32 recurrence anchor and a dynamic FP8 E4M3
read copy grouped by the 128 key channels of each value row; every 16-token
flush recomputes the recurrence from the raw inputs and the FP32 anchor, and
read-side quantization errors never overwrite the anchor.  Scope on that page:
GDN, normalized q/k, K = 128, FP8 or disabled read quantization.  The page
prints no formula; the reading used here (H = S^T, Dk x Dv, t counted from the
sequence start, W the flush period):

    anchor A (starts at h0), read state R:
    for t in the sequence:
        if t % W == 0:  R <- Q_read(A)     (fp32 QDQ; one scale per value row of S,
                                            i.e. per column of H over all Dk key rows)
        A <- exp(g_t) A;  A <- A + beta_t k_t (v_t - A^T k_t)^T     (raw inputs only)
        R <- exp(g_t) R;  R <- R + beta_t k_t (v_t - R^T k_t)^T     (the token's forward)
        o_t = scale R^T q_t
    ht = A

so inside a window the outputs follow the ordinary recurrence started from the
quantized snapshot of the anchor, and the anchor itself is the unquantized
recurrence.  With the read quantizer disabled R == A and the profile is the
plain gated delta rule.

``two_precision_torch`` is the same loop in differentiable torch with the read
quantizer as an identity straight-through estimator: its autograd is the
backward ("window-wise adjoint") the kernels are checked against.
"""
from __future__ import annotations

import numpy as np

from . import _np, qdq_groups


def read_copy(A, read_mode):
    """Q_read of fp64 anchors [..., Dk, Dv]: fp32 QDQ (qdq.c) with one group per
    column spanning all Dk rows."""
    if read_mode == "none":
        return A.copy()
    if read_mode != "e4m3":
        raise ValueError("the read quantizer is E4M3 or disabled")
    shp = A.shape
    y, _ = qdq_groups(A.astype(np.float32).reshape(-1, shp[-2], shp[-1]), 1, "e4m3")
    return y.reshape(shp).astype(np.float64)


def two_precision(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, read_mode="e4m3",
                  flush=16, record=None):
    """q, k [B, T, Hk, Dk]; v [B, T, Hv, Dv]; beta, g [B, T, Hv]; h0 [N, Hv, Dk, Dv] or None;
    cu_seqlens [N + 1] or None (then B rows).

    Returns (o fp64 [B, T, Hv, Dv], ht fp64 [N, Hv, Dk, Dv]).  With a list as
    ``record``, (sequence, token offset, anchor [Hv, Dk, Dv]) is appended at
    every flush, before the read copy is taken; nothing else changes."""
    if flush < 1:
        raise ValueError("flush period must be >= 1")
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
    heads = np.arange(Hv) // G

    def step(H, a, kt, vt, bt):
        H = a[:, None, None] * H
        u = vt - np.einsum("hkv,hk->hv", H, kt)
        return H + bt[:, None, None] * kt[:, :, None] * u[:, None, :]

    for n, (b, t0, t1) in enumerate(seqs):
        A = h0[n].copy()                                       # [Hv, Dk, Dv]
        R = A
        for t in range(t0, t1):
            if (t - t0) % flush == 0:
                if record is not None:
                    record.append((n, t - t0, A.copy()))
                R = read_copy(A, read_mode)
            kt, qt = k[b, t][heads], q[b, t][heads]
            a = np.exp(g[b, t])
            A = step(A, a, kt, v[b, t], beta[b, t])
            R = step(R, a, kt, v[b, t], beta[b, t])
            o[b, t] = scale * np.einsum("hkv,hk->hv", R, qt)
        ht[n] = A
    return o, ht


def two_precision_torch(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, read_mode="e4m3",
                        flush=16):
    """The same profile in differentiable fp64 torch, for the backward: the read
    copy is Q_read through the identity straight-through estimator (the
    gradient of R's snapshot reaches the anchor unchanged), everything else is
    the exact recurrence, so autograd gives the window-wise adjoint the page
    describes ("[5/8] ReplaySSM state QAT and two-precision GDN", "What does
    this PR do?": a window-wise adjoint during backward).  Plain Python loops:
    small cases only.  Inputs as two_precision (torch fp64 tensors); returns
    (o [B, T, Hv, Dv], ht [N, Hv, Dk, Dv])."""
    import torch

    from .chunked import qdq_ste

    if flush < 1:
        raise ValueError("flush period must be >= 1")
    if read_mode not in ("none", "e4m3"):
        raise ValueError("the read quantizer is E4M3 or disabled")
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    if cu_seqlens is not None:
        cu = [int(x) for x in _np(cu_seqlens)]
        seqs = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    else:
        seqs = [(b, 0, T) for b in range(B)]
    N = len(seqs)
    if h0 is None:
        h0 = torch.zeros(N, Hv, Dk, Dv, dtype=torch.float64)
    out = {}
    hts = []
    for n, (b, t0, t1) in enumerate(seqs):
        hn = []
        for h in range(Hv):
            hk = h // G
            A = h0[n, h]
            R = A
            for t in range(t0, t1):
                if (t - t0) % flush == 0:
                    # one scale per column of H over all Dk key rows
                    R = qdq_ste(A[None], read_mode, 1)[0]
                a = torch.exp(g[b, t, h])
                kt = k[b, t, hk]
                A = a * A
                A = A + beta[b, t, h] * torch.outer(kt, v[b, t, h] - A.transpose(0, 1) @ kt)
                R = a * R
                R = R + beta[b, t, h] * torch.outer(kt, v[b, t, h] - R.transpose(0, 1) @ kt)
                out[(b, t, h)] = scale * (R.transpose(0, 1) @ q[b, t, hk])
            hn.append(A)
        hts.append(torch.stack(hn, 0))
    zero = torch.zeros(Dv, dtype=torch.float64)
    o = torch.stack([torch.stack([torch.stack([out.get((b, t, h), zero) for h in range(Hv)], 0)
                                  for t in range(T)], 0) for b in range(B)], 0)
    return o, torch.stack(hts, 0)
