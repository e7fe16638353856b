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


# ---- the differentiable form and its backward (window-wise adjoint) ----

import torch  # noqa: E402

from oracle.chunked import qdq_ste  # noqa: E402
from oracle.recurrent_torch import recurrent_torch  # noqa: E402
from oracle.two_precision import two_precision_torch  # noqa: E402


def _t64(d, names=("q", "k", "v", "beta", "g", "h0")):
    return [None if d[n] is None else d[n].to(torch.float32).to(torch.float64) for n in names]


@pytest.mark.parametrize("lengths,read_mode", [(None, "e4m3"), (None, "none"), ([1, 16, 37, 5], "e4m3")])
def test_torch_form_is_the_profile(lengths, read_mode):
    d = _case(lengths=lengths, seed=5)
    o1, h1 = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                           cu_seqlens=d["cu_seqlens"], read_mode=read_mode, scale=0.5)
    o2, h2 = two_precision_torch(*_t64(d), cu_seqlens=d["cu_seqlens"], read_mode=read_mode, scale=0.5)
    assert np.abs(o1 - o2.numpy()).max() <= 1e-12 * np.abs(o1).max()
    assert np.abs(h1 - h2.numpy()).max() <= 1e-12 * np.abs(h1).max()


def _grads(fn, xs, do, dht):
    xs = [x.clone().requires_grad_(True) for x in xs]
    o, ht = fn(*xs)
    ((o * do).sum() + (ht * dht).sum()).backward()
    return [torch.zeros_like(x) if x.grad is None else x.grad for x in xs]


def _upstream(d, seed):
    gen = torch.Generator().manual_seed(seed)
    o_shape = d["v"].shape
    do = torch.randn(*o_shape, generator=gen, dtype=torch.float64)
    dht = torch.randn(*d["h0"].shape, generator=gen, dtype=torch.float64) * 0.1
    return do, dht


def test_torch_read_disabled_gradients_are_the_token_recurrence():
    """With the read quantizer off R == A: the backward is the plain recurrence's."""
    d = _case(seed=6, T=40)
    do, dht = _upstream(d, 6)
    xs = _t64(d)
    g1 = _grads(lambda *x: two_precision_torch(*x, read_mode="none", scale=0.5, flush=16), xs, do, dht)
    g2 = _grads(lambda *x: recurrent_torch(*x, scale=0.5, state_mode="none"), xs, do, dht)
    for a, b in zip(g1, g2):
        assert torch.abs(a - b).max() <= 1e-12 * torch.abs(b).max()


def test_torch_single_window_gradients():
    """One flush (W >= T): o follows the plain recurrence from Q_read(h0) and ht
    the plain recurrence from h0, so the backward is the sum of the two plain
    recurrences' gradients, the first passing its h0 gradient through the
    identity straight-through estimator."""
    d = _case(seed=7, T=30)
    do, dht = _upstream(d, 7)
    xs = _t64(d)
    g1 = _grads(lambda *x: two_precision_torch(*x, read_mode="e4m3", scale=0.5, flush=64), xs, do, dht)

    def o_path(q, k, v, beta, g, h0):
        hq = torch.stack([qdq_ste(h0[:, h], "e4m3", 1) for h in range(h0.shape[1])], 1)
        o, _ = recurrent_torch(q, k, v, beta, g, hq, scale=0.5, state_mode="none")
        return o, torch.zeros_like(h0)

    def ht_path(q, k, v, beta, g, h0):
        _, ht = recurrent_torch(q, k, v, beta, g, h0, scale=0.5, state_mode="none")
        return torch.zeros_like(d["v"], dtype=torch.float64), ht

    ga = _grads(o_path, xs, do, dht)
    gb = _grads(ht_path, xs, do, dht)
    for x, a, b in zip(("q", "k", "v", "beta", "g", "h0"), g1, [p + r for p, r in zip(ga, gb)]):
        assert torch.abs(a - b).max() <= 1e-12 * torch.abs(b).max(), x


def test_torch_step_adjoint_closed_form():
    """One token, Dk = Dv = 1, read copy off: H1 = a (1 - b k^2) H0 + b k v,
    o = s H1 q, loss c H1 with c = s do q + dht; the gradients written out by
    hand."""
    rng = np.random.default_rng(8)
    q0, k0, v0, b0, g0, h00, do0, dh0 = rng.normal(size=8)
    b0 = 1.0 / (1.0 + np.exp(-b0))
    s = 0.7
    T = lambda x: torch.tensor([[[[x]]]], dtype=torch.float64)
    xs = [T(q0), T(k0), T(v0), torch.tensor([[[b0]]], dtype=torch.float64),
          torch.tensor([[[g0]]], dtype=torch.float64), T(h00)]
    grads = _grads(lambda *x: two_precision_torch(*x, read_mode="none", scale=s, flush=16), xs,
                   T(do0)[0], T(dh0))
    a = np.exp(g0)
    h1 = a * (1 - b0 * k0 * k0) * h00 + b0 * k0 * v0
    c = s * do0 * q0 + dh0
    want = {"q": s * do0 * h1, "k": c * (b0 * v0 - 2 * a * b0 * k0 * h00),
            "v": c * b0 * k0, "beta": c * k0 * (v0 - a * k0 * h00),
            "g": c * a * (1 - b0 * k0 * k0) * h00, "h0": c * a * (1 - b0 * k0 * k0)}
    for name, got in zip(("q", "k", "v", "beta", "g", "h0"), grads):
        assert abs(float(got.reshape(-1)[0]) - want[name]) <= 1e-12 * max(1.0, abs(want[name])), name


def test_torch_read_disabled_gradcheck():
    w = synth.small(B=1, T=5, Hk=1, Hv=1, Dk=4, Dv=3, h0=True, seed=9)
    d = synth.make_inputs(w)
    xs = [x.clone().requires_grad_(True) for x in _t64(d)]
    assert torch.autograd.gradcheck(
        lambda *x: two_precision_torch(*x, read_mode="none", scale=0.5, flush=2), xs)
