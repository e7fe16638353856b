"""Pins for the two-precision GDN oracle (oracle/two_precision.py): a
hand-derived case (grouping of the read scale, flush timing, the anchor kept
apart from the read state), reduction to the token recurrence O1 when the read
quantizer is disabled, the anchor's independence of the read quantizer, the
one-token flush period as the decode step's "pre" readout of the anchor, the
zero-write-strength closed form, and packed sequences flushing from their own
starts."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle.decode import decode
from oracle.two_precision import two_precision
from gated_delta_rule_54_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _hand():
    with open(os.path.join(HERE, "golden", "two_precision_hand_case.json")) as f:
        c = json.load(f)
    T = len(c["beta"])
    x = dict(q=np.array(c["q"])[None, :, None, :], k=np.array(c["k"])[None, :, None, :],
             v=np.array(c["v"])[None, :, None, :], beta=np.array(c["beta"])[None, :, None],
             g=np.zeros((1, T, 1)), h0=np.array(c["h0"])[None, None])
    return c, x


def test_hand_case():
    c, x = _hand()
    o, ht = two_precision(**x, flush=c["flush"])
    assert np.array_equal(o[0, :, 0], np.array(c["o"]))
    assert np.array_equal(ht[0, 0], np.array(c["ht"]))


def test_hand_case_read_disabled():
    c, x = _hand()
    o, ht = two_precision(**x, flush=c["flush"], read_mode="none")
    assert np.array_equal(o[0, :, 0], np.array(c["o_read_disabled"]))
    assert np.array_equal(ht[0, 0], np.array(c["ht"]))


def _case(lengths=None, seed=0, Hk=2, Hv=4, T=70):
    w = synth.small(B=2 if lengths is None else 1, T=T if lengths is None else 0, Hk=Hk, Hv=Hv,
                    Dk=32, Dv=16, h0=True, seed=seed)
    return synth.make_inputs(w, lengths=lengths)


@pytest.mark.parametrize("lengths", [None, [1, 16, 37, 5]])
def test_read_disabled_is_the_token_recurrence(lengths):
    d = _case(lengths=lengths, seed=1)
    cu = d["cu_seqlens"]
    o, ht = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], cu_seqlens=cu,
                          read_mode="none", scale=0.5)
    o1, h1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], cu_seqlens=cu,
                              state_mode="none", scale=0.5)
    assert np.abs(o - o1).max() <= 1e-10 * np.abs(o1).max()
    assert np.abs(ht - h1).max() <= 1e-10 * np.abs(h1).max()


@pytest.mark.parametrize("flush", [1, 5, 16])
def test_anchor_ignores_the_read_quantizer(flush):
    d = _case(seed=2)
    args = [d[n] for n in ("q", "k", "v", "beta", "g", "h0")]
    o_q, ht_q = two_precision(*args, read_mode="e4m3", flush=flush)
    o_n, ht_n = two_precision(*args, read_mode="none", flush=flush)
    assert np.array_equal(ht_q, ht_n)          # read errors never reach the anchor
    assert not np.array_equal(o_q, o_n)        # but the outputs see them
    assert np.abs(o_q - o_n).max() <= 0.1 * np.abs(o_n).max()


def test_one_token_flush_is_the_decode_pre_readout_of_the_anchor():
    # flush period 1: every token reads Q(A_t) freshly, which is one decode step
    # (readout "pre", one scale per value row = block_v 1) on the anchor state
    d = _case(seed=3, T=9)
    args = [d[n] for n in ("q", "k", "v", "beta", "g")]
    o, _ = two_precision(*args, d["h0"], read_mode="e4m3", flush=1)
    B, T = d["B"], d["T"]
    for t in range(T):
        if t == 0:
            state = d["h0"].numpy().astype(np.float64)
        else:
            _, state = oracle.recurrent(*[x[:, :t] for x in args], d["h0"], state_mode="none")
        sl = [x[:, t:t + 1] for x in args]
        od, _ = decode(*sl, state, state_mode="e4m3", block_v=1, readout="pre")
        assert np.abs(o[:, t] - od[:, 0]).max() <= 1e-12 * max(1.0, np.abs(od).max())


def test_zero_beta_reads_the_decayed_quantized_h0():
    # beta = 0: nothing is written; with the flush period past the sequence end
    # o_t = exp(sum_{s<=t} g_s) Q(h0)^T q_t, Q one E4M3 scale per value row
    rng = np.random.default_rng(4)
    T, Dk, Dv = 12, 8, 6
    q = rng.standard_normal((1, T, 1, Dk)).astype(np.float32)
    k = rng.standard_normal((1, T, 1, Dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, Dv)).astype(np.float32)
    g = (-rng.uniform(0, 0.3, (1, T, 1))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, Dk, Dv)).astype(np.float32)
    o, ht = two_precision(q, k, v, np.zeros((1, T, 1), np.float32), g, h0, flush=T + 3)
    Qh0, sc = oracle.qdq_groups(h0[0, 0][None], 1, "e4m3")
    assert sc.shape == (1, Dv)                                  # one scale per value row
    cum = np.cumsum(g[0, :, 0].astype(np.float64))
    ref = np.exp(cum)[:, None] * (q[0, :, 0].astype(np.float64) @ Qh0[0].astype(np.float64))
    assert np.abs(o[0, :, 0] - ref).max() <= 1e-12 * np.abs(ref).max()
    assert np.abs(ht[0, 0] - np.exp(cum[-1]) * h0[0, 0]).max() <= 1e-12


def test_packed_sequences_flush_from_their_own_start():
    lengths = [3, 21, 17]
    d = _case(lengths=lengths, seed=5)
    o, ht = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                          cu_seqlens=d["cu_seqlens"], flush=4)
    cu = np.asarray(d["cu_seqlens"])
    for n in range(len(lengths)):
        a, b = int(cu[n]), int(cu[n + 1])
        on, hn = two_precision(*[d[x][:, a:b] for x in ("q", "k", "v", "beta", "g")],
                               d["h0"][n:n + 1], flush=4)
        assert np.array_equal(o[:, a:b], on)
        assert np.array_equal(ht[n], hn[0])


@pytest.mark.parametrize("rm", ["e4m3", "none"])
def test_two_precision_scales_exactly_with_values_and_state(rm):
    """Anchor and read copy are linear in (v, h0), and the read QDQ absorbs
    powers of two: scaling both by 2^k scales o and ht by exactly 2^k in fp64."""
    import torch
    w = synth.small(B=2, T=70, Hk=1, Hv=2, Dk=128, Dv=64, w_mode="none", h0=True, seed=64)
    d = synth.make_inputs(w)
    o, ht = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], read_mode=rm)
    for k in (-9, 4):
        f = 2.0 ** k
        v2 = (d["v"].float() * f).to(torch.bfloat16)
        assert torch.equal(v2.float(), d["v"].float() * f)
        o2, ht2 = two_precision(d["q"], d["k"], v2, d["beta"], d["g"], d["h0"] * f, read_mode=rm)
        assert np.array_equal(np.asarray(o2), np.asarray(o) * f)
        assert np.array_equal(np.asarray(ht2), np.asarray(ht) * f)
