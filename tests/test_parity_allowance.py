"""CPU pins of the derived flip allowances in _parity.py.

A flip is planted in the oracle itself (a quantization code moved one grid
step), the oracle is run again, and the change it causes in every output
element must lie within the allowance that _parity.py derives from the flip's
location and the unperturbed oracle's values — and the allowance must not be
vacuous (it stays within a modest factor of the largest real change, and is
zero before the flip)."""
import numpy as np
import pytest
import torch

import oracle
import oracle.chunked as oc
import oracle.decode as od
from gated_delta_rule_54_gb300 import synth

from _parity import (FP_MARGIN, code_gap, decode_flip_allowance, flip_candidates, fwd_flip_allowance,
                     sequence_allowances)


def _e4m3_neighbor(code):
    """The adjacent E4M3 code on the side of the larger grid gap (what code_gap measures)."""
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
    v = vals[code]
    fin = np.isfinite(vals)
    cands = [c for c in range(256) if fin[c] and vals[c] != v]
    lo = max((c for c in cands if vals[c] < v), key=lambda c: vals[c])
    hi = min((c for c in cands if vals[c] > v), key=lambda c: vals[c])
    return hi if vals[hi] - v >= v - vals[lo] else lo


class _FlipHook:
    """Wraps oracle.qdq_groups: on the call-th call, moves code [idx] one step."""

    def __init__(self, target_call, idx):
        self.target, self.idx, self.n = target_call, idx, 0
        self.orig = oracle.qdq_groups

    def __call__(self, x, group_cols, mode, with_codes=False):
        y, sc, cd = self.orig(x, group_cols, mode, with_codes=True)
        if self.n == self.target:
            c = int(cd[self.idx])
            sc8 = c - 256 if c >= 128 else c
            nc = _e4m3_neighbor(c) if mode == "e4m3" else (sc8 + 1 if sc8 < 127 else sc8 - 1) & 0xFF
            cd = cd.copy()
            y = y.copy()
            cd[self.idx] = nc
            grp = self.idx[-1] // group_cols
            s = sc.reshape(sc.shape[0], -1)[self.idx[0], grp]
            val = (oracle.e4m3_decode(np.array([nc], np.uint8))[0] if mode == "e4m3"
                   else float(nc - 256 if nc >= 128 else nc))
            y[self.idx] = np.float32(val) * np.float32(s)
        self.n += 1
        return (y, sc, cd) if with_codes else (y, sc)


def _check_cover(dev, allow, what, before=None):
    dev = np.abs(np.asarray(dev, dtype=np.float64))
    allow = np.asarray(allow, dtype=np.float64)
    assert (dev <= allow * (1 + 1e-9) + 1e-12 * dev.max()).all(), \
        "%s: a planted flip changes an element by more than its allowance" % what
    assert dev.max() > 0 and allow.max() <= 64 * dev.max(), \
        "%s: allowance %.3e vs largest change %.3e" % (what, allow.max(), dev.max())
    if before is not None:
        assert not allow[before].any(), "%s: allowance before the flip" % what


@pytest.mark.parametrize("site", ["state", "w"])
def test_forward_allowance_covers_a_planted_flip(site, monkeypatch):
    w = synth.small(B=2, T=200, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=41)
    d = synth.make_inputs(w)
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    o_ref, ht_ref, rec, inters = oc.chunked(*args, state_mode="e4m3", w_mode="e4m3", record=True,
                                            intermediates=True)
    nc = rec["state_codes"].shape[0]        # dense chunks: 2 sequences x 4
    # calls alternate W, state per chunk step; the batch of the call is [B*Hv]
    chunk, p = 1, 1                        # second chunk, sequence 0, head 1
    if site == "state":
        codes = rec["state_codes"][chunk, 1]
        dk, v = np.argwhere(np.abs(oracle.e4m3_decode(codes.ravel()).reshape(codes.shape)) > 100)[0]
        hook = _FlipHook(2 * chunk + 1, (p, dk, v))
    else:
        wc = rec["w_codes"][0][64 * chunk:64 * chunk + 64, 1]
        t, dk = np.argwhere(np.abs(oracle.e4m3_decode(wc.ravel()).reshape(wc.shape)) > 100)[0]
        hook = _FlipHook(2 * chunk, (p, t, dk))
    monkeypatch.setattr(oc, "qdq_groups", hook)
    o_f, ht_f, rec_f = oc.chunked(*args, state_mode="e4m3", w_mode="e4m3", record=True)
    monkeypatch.undo()
    # the flip locations as the GPU tests find them: codes that differ (the
    # planted one, and any later code its perturbation moves)
    sf = rec_f["state_codes"] != rec["state_codes"]
    wf = np.concatenate(rec_f["w_codes"], 0) != np.concatenate(rec["w_codes"], 0)
    assert sf.sum() + wf.sum() >= 1
    o_al, ht_al = fwd_flip_allowance(d, inters, rec, sf, wf, [200, 200], False, 1.0, 64,
                                     "e4m3", "e4m3")
    before = np.zeros(o_al.shape, bool)
    before[:, :64 * chunk] = True
    before[1] = True                        # the other sequence never sees the flip
    before[..., 0, :] = True                # nor the other head
    _check_cover((o_f - o_ref).numpy(), o_al, "o (%s flip)" % site, before)
    dev = np.abs((ht_f - ht_ref).numpy())
    assert (dev <= ht_al * (1 + 1e-9) + 1e-300).all()


def test_decode_allowance_covers_a_planted_flip(monkeypatch):
    w = synth.small(B=2, T=6, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=42)
    d = synth.make_inputs(w)
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    ro, rS, rc, rs = od.decode(*args, state_mode="e4m3", block_v=32, readout="pre", record=True)
    t, b, h = 2, 1, 0
    dk, v = np.argwhere(np.abs(oracle.e4m3_decode(rc[b, t, h].ravel()).reshape(64, 64)) > 100)[0]
    hook = _FlipHook(t, (b * 2 + h, dk, v))
    monkeypatch.setattr(od, "qdq_groups", hook)
    o_f, S_f, rc_f, _ = od.decode(*args, state_mode="e4m3", block_v=32, readout="pre", record=True)
    monkeypatch.undo()
    flip = rc_f != rc
    assert flip[b, t, h, dk, v]
    o_al, s_al = decode_flip_allowance(d, rc, rs, flip, rS, 1.0, 32, "e4m3", "pre")
    before = np.ones(o_al.shape, bool)
    before[b, t:, h] = False
    _check_cover(o_f - ro, o_al, "decode o", before)
    assert (np.abs(S_f - rS) <= s_al * (1 + 1e-9) + 1e-300).all()


def test_flip_candidates_find_the_value_nearest_a_boundary():
    """A value nudged onto the far side of its rounding boundary changes code
    only where flip_candidates says it may."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 64, 64)).astype(np.float32)
    y, sc, cd = oracle.qdq_groups(x, 32, "e4m3", with_codes=True)
    margin = 1e-3 * np.abs(x).max()
    _, sig = flip_candidates(x, 32, "e4m3", margin)
    xp = x + rng.uniform(-margin, margin, x.shape).astype(np.float32)
    # keep the amax elements fixed so that the scales do not move
    am = np.abs(x).reshape(3, 64, 2, 32).max(axis=(1, 3))
    keep = np.abs(x) == np.repeat(am, 32, axis=1)[:, None, :]
    xp[keep] = x[keep]
    _, sc2, cd2 = oracle.qdq_groups(xp, 32, "e4m3", with_codes=True)
    assert np.array_equal(sc, sc2)
    changed = cd2 != cd
    assert changed.any() and (sig[changed] > 0).all()
    assert np.allclose(sig[sig > 0], (code_gap(cd, "e4m3") * np.repeat(sc, 32, 1)[:, None, :])[sig > 0], rtol=1e-12)


def test_kda_allowance_covers_a_planted_flip(monkeypatch):
    """A flip planted at one of the oracle's own flip candidates (an element
    within the kernels' error margin of its rounding boundary) is covered."""
    import oracle.kda as ok
    w = synth.small(B=1, T=140, Hk=1, Hv=1, Dk=64, Dv=64, w_mode="none", h0=True, seed=43)
    d = synth.make_kda_inputs(w)
    args = (d["q"], d["k"], d["v"], d["beta"], d["g_k"], d["h0"])
    rec = []
    ro, rh = ok.kda_recurrent(*args, state_mode="int8", record=rec)
    H = rec[1][2].astype(np.float32)            # [Hv, Dk, Dv] entering token 64
    amax = np.abs(H).reshape(1, 64, 1, 64).max()
    _, sig = flip_candidates(H, 64, "int8", FP_MARGIN * amax)
    assert sig.any()
    h, dk, v = np.unravel_index(np.argmax(sig), sig.shape)
    hook = _FlipHook(1, (h, dk, v))
    monkeypatch.setattr(ok, "qdq_groups", hook)
    o_f, h_f = ok.kda_recurrent(*args, state_mode="int8")
    monkeypatch.undo()
    o_al, ht_al = sequence_allowances(d, rec, "int8", 64, 1.0, g_key="g_k")
    dev = np.abs(o_f - ro)
    assert (dev[0, :64] == 0).all()
    assert (dev <= o_al * (1 + 1e-9) + 1e-300).all()
    assert (np.abs(h_f - rh) <= ht_al * (1 + 1e-9) + 1e-300).all()
