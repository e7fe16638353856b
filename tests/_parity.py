"""Shared tolerance checks, derived flip allowances and oracle runners for
the GPU parity tests.

Tolerances (stated once, used everywhere):
  outputs / final states: max |x - r| <= 1e-2 * max|r| + a_i, and at least
      99.9% of elements satisfy |x - r| <= 1e-2 * |r| + 1e-4 * max|r| + a_i,
      where a_i is the element's flip allowance below (zero for every element
      that no quantization flip can reach).  The absolute floor 1e-4 * max|r|
      is for reference elements near zero: the kernels' split-bf16 operands
      carry about 16 mantissa bits, so an output that is a short sum of terms
      of size up to max|r| can be off by about 2^-16 * max|r| whatever its own
      size;
  state / W codes: every differing code is one quantization step away (E4M3:
      or within 2^-5 in code units, where the grid steps by 2^-9), and at
      most 0.1% of the codes differ (at least one flip is always allowed: a
      single flip in a few hundred codes is consistent with a 1e-5 flip rate);
      state codes are compared this way in each (sequence, head) up to and
      including its first chunk (token) with a flip; the later ones carry that
      flip's perturbation, which the allowance bounds;
  flip allowance: a code one step away from the oracle's changes that
      quantized element by (the code's grid gap) x (its tile scale), both
      taken from the oracle.  That perturbation is pushed through the exact
      linear maps of the method with the oracle's own values: within a chunk
      o changes by (diag(e^gamma) Q - P W^) E + P dW^ (H^ + E) and the next
      state by R E + K~^T dW^ (H^ + E) with R = e^{gamma_L} I - K~^T W^
      (spectral norm from the oracle), and the next state quantization keeps
      only its own flips and a scale change of at most max|dH| / amax.  Token
      recurrences use (I - beta k k^T) (spectral norm <= 1) and the decay.
      Where the kernel does not report its codes (KDA, two-precision, the
      decode post readout of the last token; fp32 recurrences) every element
      whose oracle value lies within 2^-20 of the tile amax (plus any
      perturbation already propagated) of a rounding boundary counts as
      possibly flipped.  Elements before a unit's first flip get no allowance;
  gradients: relative L2 error ||x - r|| / ||r|| <= 2e-2 per tensor.
Every test that applies an allowance records how many (sequence, head) units
carried one; the session summary prints the counts.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle.chunked import chunked

REL = 1e-2
FLOOR = 1e-4
FRAC = 1e-3
CODE_FRAC = 1e-3
GRAD_L2 = 2e-2
FP_MARGIN = 2.0 ** -20   # fp32 kernels' error at a quantization input, relative to the tile amax
DEQ_SLACK = 1.0 + 2.0 ** -20   # a dequantized value is code x scale rounded to binary32

# (test name, what, units with an allowance, units, max allowance / max|ref|),
# printed by the session summary (conftest.py)
ALLOWANCE_LOG = []


def close_report(x, ref, allow=None):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    a = 0.0 if allow is None else np.asarray(allow, dtype=np.float64)
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    err = np.abs(x - ref)
    bad = err > REL * np.abs(ref) + FLOOR * mx + a
    over = err - a
    return dict(max_rel=float(over.max() / mx) if mx > 0 else float(over.max() if over.size else 0),
                frac_bad=float(bad.mean()) if bad.size else 0.0, n=int(ref.size),
                finite=bool(np.isfinite(x).all()))


def assert_close(x, ref, what="", allow=None):
    """Spec bound, each element widened by its flip allowance (if any)."""
    r = close_report(x, ref, allow)
    assert r["finite"], "%s: non-finite values" % what
    assert r["max_rel"] <= REL, "%s: max (|err| - allowance) / max|ref| = %.3e" % (what, r["max_rel"])
    assert r["frac_bad"] <= FRAC, "%s: %.3e of elements outside 1e-2 relative" % (what, r["frac_bad"])
    return r


def log_allowance(what, allow, ref, unit_axes):
    """Record how many units (indexed by unit_axes of allow) carry an allowance."""
    import os
    allow = np.asarray(allow, dtype=np.float64)
    if allow.size == 0:
        return
    ax = tuple(i for i in range(allow.ndim) if i not in unit_axes)
    per_unit = allow.max(axis=ax) if ax else allow
    mx = float(np.abs(np.asarray(ref)).max()) if np.asarray(ref).size else 0.0
    ALLOWANCE_LOG.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], what,
                          int((per_unit > 0).sum()), int(per_unit.size),
                          float(allow.max() / mx) if mx > 0 else 0.0))


# ----------------------------------------------------------------------------
# Quantization grid gaps and flip candidates (oracle values only)
# ----------------------------------------------------------------------------
_E4M3 = {}


def _e4m3_tables():
    """Per E4M3 code: its value and the distances to the next smaller and next
    larger value of the grid (0 past the ends; NaN codes have none)."""
    if not _E4M3:
        vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
        fin = np.isfinite(vals)
        grid = np.unique(vals[fin])
        lo = np.zeros(256)
        hi = np.zeros(256)
        for c in np.nonzero(fin)[0]:
            i = int(np.searchsorted(grid, vals[c]))
            lo[c] = grid[i] - grid[i - 1] if i > 0 else 0.0
            hi[c] = grid[i + 1] - grid[i] if i + 1 < grid.size else 0.0
        _E4M3.update(val=np.where(fin, vals, 0.0), lo=lo, hi=hi)
    return _E4M3


def code_gap(codes, mode):
    """Largest distance, in code units, from each code's value to an adjacent
    value of its grid: what one step away from that code changes it by (with
    the binary32 rounding of code x scale)."""
    codes = np.asarray(codes, dtype=np.uint8)
    if mode == "int8":
        return np.full(codes.shape, DEQ_SLACK)
    t = _e4m3_tables()
    return DEQ_SLACK * np.maximum(t["lo"][codes], t["hi"][codes])


def flip_candidates(x, group_cols, mode, margin):
    """Elements of x whose code another fp path could round differently.

    x: fp32 [batch, rows, cols] as the oracle quantizes it (one scale per
    batch index and block of group_cols columns); margin: absolute distance
    (scalar or broadcastable to x) within which the value may sit on the other
    side of its rounding boundary.  Returns the oracle's dequantized values,
    and sigma = (code gap) x scale where a flip is possible, else 0."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y, sc, cd = oracle.qdq_groups(x, group_cols, mode, with_codes=True)
    s = np.repeat(sc.astype(np.float64), group_cols, axis=-1)[:, None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(s > 0, x.astype(np.float64) / np.where(s > 0, s, 1.0), 0.0)
    if mode == "int8":
        val = cd.view(np.int8).astype(np.float64)
        lo = np.where(val > -127, 1.0, 0.0)
        hi = np.where(val < 127, 1.0, 0.0)
    else:
        t = _e4m3_tables()
        val, lo, hi = t["val"][cd], t["lo"][cd], t["hi"][cd]
    # distance (code units) from u to the rounding boundary on its side of val
    up = u >= val
    dist = np.where(up, np.where(hi > 0, val + hi / 2 - u, np.inf),
                    np.where(lo > 0, u - (val - lo / 2), np.inf))
    dist = np.maximum(dist, 0.0)
    possible = (s > 0) & (dist * s <= margin)
    return y.astype(np.float64), np.where(possible, DEQ_SLACK * np.maximum(lo, hi) * s, 0.0)


def tile_amax(x, group_cols):
    """amax per [rows, group_cols] tile of x [batch, rows, cols], broadcast back."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    b, r, c = x.shape
    m = x.reshape(b, r, c // group_cols, group_cols).max(axis=(1, 3))
    return np.repeat(m, group_cols, axis=-1)[:, None, :]


# ----------------------------------------------------------------------------
# Flip allowance of the chunked forward
# ----------------------------------------------------------------------------
def fwd_flip_allowance(d, inters, rec, state_flip, w_flip, lens, packed, scale, block_v, sm, wm):
    """Per-element allowances for o [B, T, Hv, Dv] and ht [N, Hv, Dk, Dv].

    state_flip: bool [n_chunks, Hv, Dk, Dv] where the kernel's state code
    differs from the oracle's (dense chunk order; after a unit's first flip its
    later codes may differ by more than one step: the carried perturbation
    bounds them); w_flip: bool [B*T, Hv, Dk] likewise for W codes.  Everything else comes from the oracle's
    intermediates (chunked(..., intermediates=True)) and its record."""
    q = d["q"].double().numpy()
    k = d["k"].double().numpy()
    B, T, Hk, Dk = k.shape
    Hv, Dv = d["v"].shape[2], d["v"].shape[3]
    G = Hv // Hk
    qf = q.reshape(B * T, Hk, Dk)
    kf = k.reshape(B * T, Hk, Dk)
    N = len(lens)
    o_al = np.zeros((B * T, Hv, Dv))
    ht_al = np.zeros((N, Hv, Dk, Dv))
    # W codes by token (empty sequences have none), in the tokens' order
    wref = np.concatenate(rec["w_codes"], 0) if wm != "none" and rec.get("w_codes") else None
    cbase = np.concatenate([[0], np.cumsum([-(-L // 64) for L in lens])]).astype(int)
    tbase = np.concatenate([[0], np.cumsum(lens)]).astype(int) if packed else \
        np.arange(N + 1) * T
    for n in range(N):
        L = lens[n]
        nch = -(-L // 64)
        inter = inters[n] if packed else inters[0]
        for h in range(Hv):
            p = h if packed else n * Hv + h
            sf = state_flip[cbase[n]:cbase[n] + nch, h] if sm != "none" else None
            wf = w_flip[tbase[n]:tbase[n] + L, h] if wm != "none" else None
            ev = [c for c in range(nch)
                  if (sf is not None and sf[c].any()) or
                  (wf is not None and wf[64 * c:64 * c + 64].any())]
            if not ev:
                continue
            prop = np.zeros(Dv)        # column 2-norms of the state perturbation
            for c in range(ev[0], nch):
                st = inter[c]
                gam = st["gamma"][p].numpy()
                Wh = st["W_hat"][p].numpy()
                Hh = st["H_hat"][p].numpy()
                Lc = gam.size
                t0 = tbase[n] + 64 * c
                qc, kc = qf[t0:t0 + Lc, h // G], kf[t0:t0 + Lc, h // G]
                if sm != "none":
                    codes = rec["state_codes"][cbase[n] + c, h]
                    sc = np.repeat(rec["state_scales"][cbase[n] + c, h].astype(np.float64), block_v)
                    # a differing code: one step (the first flip), or, once a perturbation
                    # of column norm prop reaches the quantizer, |Q(x + d) - Q(x)| <=
                    # |d| + half a grid gap on each side (at most two of the oracle's gaps)
                    E = np.where(sf[c], (2.0 if prop.any() else 1.0) * code_gap(codes, sm) *
                                 sc[None, :] + prop[None, :], 0.0)
                    if prop.any():
                        # elsewhere the quantizer keeps its codes; its scale moves with the amax
                        E = E + np.abs(Hh) * _scale_shift(Hh, prop, block_v)[None, :]
                    Ecol = np.zeros(Dv)
                else:
                    E = np.zeros((Dk, Dv))
                    Ecol = prop
                sW = np.zeros((Lc, Dk))
                if wf is not None and wf[64 * c:64 * c + Lc].any():
                    wcodes = wref[t0:t0 + Lc, h]
                    sW = np.where(wf[64 * c:64 * c + Lc],
                                  code_gap(wcodes, wm) * float(rec["w_scales"][cbase[n] + c, h]), 0.0)
                le = np.tril(np.ones((Lc, Lc), bool))
                P = np.where(le, np.exp(np.where(le, gam[:, None] - gam[None, :], 0.0)), 0.0) * (qc @ kc.T)
                M = np.exp(gam)[:, None] * qc - P @ Wh
                Habs = np.abs(Hh) + E + Ecol[None, :]
                dD = sW @ Habs                                   # |dW^ (H^ + E)|
                ob = np.abs(M) @ E + np.linalg.norm(M, axis=1)[:, None] * Ecol[None, :] + \
                    np.abs(P) @ dD
                o_al[t0:t0 + Lc, h] = abs(scale) * ob
                Kd = kc * np.exp(gam[-1] - gam)[:, None]
                R = np.exp(gam[-1]) * np.eye(Dk) - Kd.T @ Wh
                prop = np.linalg.norm(R, 2) * (np.linalg.norm(E, axis=0) + Ecol) + \
                    np.linalg.norm(Kd, 2) * np.linalg.norm(dD, axis=0)
            ht_al[n, h] = prop[None, :]
    return o_al.reshape(B, T, Hv, Dv), ht_al


# ----------------------------------------------------------------------------
# Flip allowances of the token recurrences
# ----------------------------------------------------------------------------
def token_step_norm(beta, k):
    """Spectral norm of I - beta k k^T (k not necessarily unit)."""
    kk = float(np.dot(k, k))
    return max(1.0, abs(1.0 - beta * kk))


def code_steps(a, b, mode):
    """Distance in quantization steps between two code arrays (u8)."""
    a = np.asarray(a, dtype=np.uint8)
    b = np.asarray(b, dtype=np.uint8)
    if mode == "int8":
        return np.abs(a.view(np.int8).astype(np.int32) - b.view(np.int8).astype(np.int32))
    sa = np.where(a & 0x80, -1, 1) * (a & 0x7F).astype(np.int32)
    sb = np.where(b & 0x80, -1, 1) * (b & 0x7F).astype(np.int32)
    return np.abs(sa - sb)


def assert_codes(a, b, mode, what="codes"):
    d = code_steps(a, b, mode)
    if mode == "e4m3" and d.size:
        # Below 2^-5 the E4M3 grid steps by 2^-9 (subnormals and the lowest
        # normal binade), finer than the kernel's fp32 / split-bf16 error
        # relative to the group amax (448 in code units): near-zero elements
        # may land a few codes apart.  Differences within 2^-5 in code units
        # (2^-5 s, about 7e-5 of the amax) count as one step.
        near = np.abs(oracle.e4m3_decode(np.ravel(a)).astype(np.float64) -
                      oracle.e4m3_decode(np.ravel(b)).astype(np.float64)) <= 2.0 ** -5
        d = np.where(near.reshape(d.shape) & (d > 1), 1, d)
    nflip = int((d > 0).sum())
    frac = nflip / d.size if d.size else 0.0
    assert d.max(initial=0) <= 1, "%s: a code differs by %d steps" % (what, int(d.max()))
    assert nflip <= max(1, CODE_FRAC * d.size), "%s: %.3e of codes differ" % (what, frac)
    return frac


def grad_rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


def slot_map(lengths, packed, T):
    """For each dense chunk index (sequence after sequence), its chunk slot in
    the library's context layout (see include/gdn_qdq.h)."""
    out = []
    if packed:
        start = 0
        for n, L in enumerate(lengths):
            for c in range(-(-L // 64)):
                out.append(start // 64 + n + c)
            start += L
    else:
        nt = -(-T // 64)
        for n in range(len(lengths)):
            for c in range(nt):
                out.append(n * nt + c)
    return np.array(out, dtype=np.int64)


def run_oracle(d, state_mode, w_mode, scale=1.0, record=False, block_v=64, neumann_degree=None):
    """O2 (chunked, fp64) on CPU inputs dict from synth.make_inputs."""
    return chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                   cu_seqlens=d.get("cu_seqlens"), scale=scale, state_mode=state_mode,
                   w_mode=w_mode, record=record, block_v=block_v, neumann_degree=neumann_degree)


def to_dev(d, device="cuda"):
    out = {}
    for k, v in d.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out
def decode_flip_allowance(d, rec_codes, rec_scales, gpu_flip, state_out, scale, block_v, sm,
                          readout):
    """Allowances for the decode step's o [B, T, Hv, Dv] and state [B, Hv, Dk, Dv].

    gpu_flip: bool [B, T, Hv, Dk, Dv] where the kernel's code of S^ read by
    token t differs from the oracle's (rec_codes, rec_scales).  A perturbation
    E of S^ reaches H = e^g (I - beta k k^T) S^ + ... scaled by at most e^g;
    the carried state passes it to the next token, whose quantizer keeps its
    own flips and a scale change of at most max|dS| / amax.  The post readout
    of the last token reads Q(state_out), whose codes the kernel does not
    report: its possible flips are the oracle's flip candidates."""
    q = d["q"].double().numpy()
    k = d["k"].double().numpy()
    g = d["g"].double().numpy()
    beta = d["beta"].double().numpy()
    B, T, Hk, Dk = k.shape
    Hv, Dv = d["v"].shape[2], d["v"].shape[3]
    G = Hv // Hk
    o_al = np.zeros((B, T, Hv, Dv))
    s_al = np.zeros((B, Hv, Dk, Dv))
    if sm == "none" or T == 0:
        return o_al, s_al
    S_last = np.asarray(state_out, dtype=np.float32)
    for b in range(B):
        for h in range(Hv):
            if not gpu_flip[b, :, h].any() and readout == "pre":
                continue
            prop = np.zeros(Dv)            # column 2-norms of the carried state's perturbation
            Es = []
            for t in range(T):
                sc = np.repeat(rec_scales[b, t, h].astype(np.float64), block_v)
                E = np.where(gpu_flip[b, t, h], (2.0 if prop.any() else 1.0) *
                             code_gap(rec_codes[b, t, h], sm) * sc[None, :] + prop[None, :], 0.0)
                if prop.any():
                    Sh = decode_values(rec_codes[b, t, h], sm) * sc[None, :]
                    E = E + np.abs(Sh) * _scale_shift(Sh, prop, block_v)[None, :]
                Es.append(E)
                eg = np.exp(g[b, t, h])
                prop = eg * token_step_norm(beta[b, t, h], k[b, t, h // G]) * np.linalg.norm(E, axis=0)
                if readout == "pre":
                    o_al[b, t, h] = abs(scale) * np.linalg.norm(q[b, t, h // G]) * prop
            if readout == "post":
                # o_t reads Q(H_t): the quantized state token t + 1 reads, or Q(state_out)
                xs = S_last[b, h][None]
                amax = tile_amax(xs, block_v)[0, 0]
                pt = np.repeat(prop.reshape(-1, block_v).max(-1), block_v)
                y, sig = flip_candidates(xs, block_v, sm, FP_MARGIN * amax + pt[None, :])
                last = sig[0] + np.abs(y[0]) * _scale_shift(y[0], prop, block_v)[None, :]
                for t in range(T):
                    Enext = Es[t + 1] if t + 1 < T else last
                    o_al[b, t, h] = abs(scale) * np.linalg.norm(q[b, t, h // G]) * \
                        np.linalg.norm(Enext, axis=0)
            s_al[b, h] = prop[None, :]
    return o_al, s_al


def decode_values(codes, mode):
    codes = np.asarray(codes, dtype=np.uint8)
    if mode == "int8":
        return codes.view(np.int8).astype(np.float64)
    return _e4m3_tables()["val"][codes]


def recurrence_flip_allowance(events, steps, Dk, Dv, mode, group_cols, scale, carried=True):
    """Allowance of one (sequence, head) token recurrence whose state is
    quantized at some tokens and whose codes the kernel does not report.

    events: {t: (state before quantization, fp64 [Dk, Dv])} for the tokens t
    whose state is quantized first; steps: list over tokens of (decay vector
    or scalar e^g, beta, k, q) — each token maps the state perturbation dH to
    (I - beta k k^T) diag(e^g) dH and reads o_t = scale H^T q.  At an event
    the perturbation becomes the oracle's flip candidates (margin FP_MARGIN x
    tile amax plus the perturbation already carried) and a scale change.
    With carried=False the quantized state is recomputed from an unperturbed
    source at every event (the two-precision read copy): the perturbation
    restarts there.  Returns the allowance [T, Dv] of o."""
    T = len(steps)
    o_al = np.zeros((T, Dv))
    prop = np.zeros(Dv)
    for t, (eg, bt, kt, qt) in enumerate(steps):
        if t in events:
            x = np.asarray(events[t], dtype=np.float32)[None]
            amax = tile_amax(x, group_cols)[0, 0]
            if not carried:
                prop = np.zeros(Dv)
            pt = np.repeat(prop.reshape(-1, group_cols).max(-1), group_cols)
            y, sig = flip_candidates(x, group_cols, mode, FP_MARGIN * amax + 2 * pt[None, :])
            E = sig[0] + np.maximum(np.abs(y[0]) * _scale_shift(y[0], prop, group_cols)[None, :],
                                    np.where(amax[0] > 0, 0.0, pt)[None, :])
            prop = np.linalg.norm(E, axis=0)
        prop = float(np.max(eg)) * token_step_norm(bt, kt) * prop
        o_al[t] = abs(scale) * np.linalg.norm(qt) * prop
    return o_al, prop


def sequence_allowances(d, rec, mode, group_cols, scale, g_key="g", carried=True):
    """Allowances of o [B, T, Hv, Dv] and ht [N, Hv, Dk, Dv] for a token
    recurrence oracle's record of (sequence, token offset, state before
    quantization [Hv, Dk, Dv]) events (see recurrence_flip_allowance)."""
    q = d["q"].double().numpy()
    k = d["k"].double().numpy()
    beta = d["beta"].double().numpy()
    g = d[g_key].double().numpy()
    B, T, Hk, Dk = k.shape
    Hv, Dv = d["v"].shape[2], d["v"].shape[3]
    G = Hv // Hk
    cu = d.get("cu_seqlens")
    if cu is not None:
        cu = [int(x) for x in cu.tolist()]
        seqs = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    else:
        seqs = [(b, 0, T) for b in range(B)]
    o_al = np.zeros((B, T, Hv, Dv))
    ht_al = np.zeros((len(seqs), Hv, Dk, Dv))
    if mode == "none":
        return o_al, ht_al
    for n, (b, t0, t1) in enumerate(seqs):
        ev = [(t, H) for (nn, t, H) in rec if nn == n]
        for h in range(Hv):
            steps = [(np.exp(g[b, t, h]), beta[b, t, h], k[b, t, h // G], q[b, t, h // G])
                     for t in range(t0, t1)]
            al, prop = recurrence_flip_allowance({t: H[h] for t, H in ev}, steps, Dk, Dv, mode,
                                                 group_cols, scale, carried)
            o_al[b, t0:t1, h] = al
            ht_al[n, h] = prop[None, :]
    return o_al, ht_al


def _scale_shift(Hq, prop, group_cols):
    """Bound on the change of each element of a quantized tile whose codes stay
    while the state it quantizes moves by at most prop (column 2-norms, which
    bound every element's change): the tile amax moves by at most that much, so
    the scale by at most pt / amax relative, and code x scale by |value| pt / amax
    (never more than pt).  Returned per column as the factor on |value|; a
    column whose tile amax is zero gets the factor 1 (the values there are zero
    and the allowance comes from pt)."""
    Dv = Hq.shape[-1]
    amax = np.repeat(np.abs(Hq).reshape(-1, Dv // group_cols, group_cols).max(axis=(0, 2)), group_cols)
    pt = np.repeat(np.asarray(prop).reshape(-1, group_cols).max(-1), group_cols)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(amax > 0, np.minimum(pt / np.where(amax > 0, amax, 1.0), 1.0),
                        np.where(pt > 0, 1.0, 0.0))
