"""Pins for the decode QAT oracle (oracle/decode.py).

The decode step is pinned against the C token recurrence with a chunk of one
token (same state, same codes), the delta-rule invariant (which holds for any
quantized state), a zero-write-strength closed form, the post readout read off
the recurrence's own record of the next token's quantized state, the split
carry from a chunked prefill against a single-pass torch recurrence, and the
QDQ error bound for the post readout.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.chunked import chunked
from oracle.decode import decode
from oracle.recurrent_torch import recurrent_torch
from gated_delta_rule_54_gb300 import synth


def _inputs(B=2, T=37, Hk=1, Hv=2, Dk=32, Dv=128, seed=0):
    w = synth.small(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, h0=True, seed=seed)
    return synth.make_inputs(w)


def _rel(a, b):
    b = np.asarray(b, np.float64)
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("sm", ["none", "e4m3", "int8"])
@pytest.mark.parametrize("block_v", [16, 32, 64, 128])
def test_decode_is_token_recurrence_with_one_token_chunks(sm, block_v):
    d = _inputs(seed=block_v)
    B, T = d["B"], d["T"]
    o, S, *rec = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                        block_v=block_v, record=True)
    o1, h1, *rec1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                     state_mode=sm, block_v=block_v, chunk=1,
                                     record_states=True)
    assert _rel(o, o1) <= 1e-12
    assert _rel(S, h1) <= 1e-12
    if sm != "none":
        c1 = rec1[0].reshape(B, T, *rec1[0].shape[1:])
        s1 = rec1[1].reshape(B, T, *rec1[1].shape[1:])
        assert np.array_equal(rec[0], c1)
        assert np.array_equal(rec[1].view(np.uint32), s1.view(np.uint32))


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_post_readout_reads_the_state_the_next_token_quantizes(sm):
    d = _inputs(T=9, Hv=4, Hk=2, Dk=64, Dv=64, seed=3)
    B, T, Hv = d["B"], d["T"], 4
    o, S = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                  readout="post")
    _, h1, codes, scales = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                            state_mode=sm, chunk=1, record_states=True)
    Dk, Dv = codes.shape[2], codes.shape[3]
    codes = codes.reshape(B, T, Hv, Dk, Dv)
    scales = scales.reshape(B, T, Hv, Dv // 64)
    dec = oracle.e4m3_decode(codes) if sm == "e4m3" else codes.view(np.int8).astype(np.float32)
    q = d["q"].double().numpy()[:, :, np.arange(Hv) // 2]
    for t in range(T):
        if t + 1 < T:
            Hq = (dec[:, t + 1].reshape(B, Hv, Dk, Dv // 64, 64) *
                  scales[:, t + 1][:, :, None, :, None]).reshape(B, Hv, Dk, Dv)
        else:
            Hq = oracle.qdq_groups(h1.astype(np.float32).reshape(B * Hv, Dk, Dv), 64, sm)[0]
            Hq = Hq.reshape(B, Hv, Dk, Dv)
        ref = np.einsum("bhkv,bhk->bhv", Hq.astype(np.float64), q[:, t])
        assert _rel(o[:, t], ref) <= 1e-12


@pytest.mark.parametrize("sm", ["none", "e4m3", "int8"])
def test_delta_rule_invariant_holds_for_any_quantized_state(sm):
    # beta = 1 and |k| = 1: H^T k = exp(g) S^T k + (v - exp(g) S^T k) = v, whatever S is.
    rng = np.random.default_rng(7)
    B, T, H, D = 3, 20, 2, 32
    k = np.zeros((B, T, H, D), np.float32)
    for idx in np.ndindex(B, T, H):
        sel = rng.choice(D, 4, replace=False)
        k[idx][sel] = 0.5 * rng.choice([-1, 1], 4)
    v = rng.standard_normal((B, T, H, D)).astype(np.float32)
    g = (-rng.uniform(0, 1, (B, T, H))).astype(np.float32)
    s0 = rng.standard_normal((B, H, D, D)).astype(np.float32)
    o, _ = decode(k, k, v, np.ones((B, T, H), np.float32), g, s0, scale=0.5, state_mode=sm,
                  block_v=16)
    assert np.abs(o - 0.5 * v).max() <= 1e-12


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_post_readout_within_the_qdq_error_bound(sm):
    d = _inputs(T=6, Hv=2, Hk=2, Dk=64, Dv=128, seed=8)
    op, _ = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                   readout="pre")
    oq, _ = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                   readout="post")
    o1, h1, _, _ = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                    state_mode=sm, chunk=1, record_states=True)
    assert _rel(op, o1) <= 1e-12
    # last token: |Q(H) - H| <= amax(tile) * (2^-4 for E4M3, 1/254 for INT8) per element
    B, Hv, Dk, Dv = h1.shape
    amax = np.abs(h1.reshape(B, Hv, Dk, Dv // 64, 64)).max(axis=(2, 4))       # [B, Hv, tiles]
    bound_el = amax * (2.0 ** -4 if sm == "e4m3" else 1 / 254) * (1 + 1e-6)
    q = np.abs(d["q"].double().numpy()[:, -1])                               # [B, Hk, Dk]
    bound = q.sum(-1)[:, :, None, None] * bound_el[:, :, :, None]             # Hk == Hv here
    err = np.abs(oq[:, -1] - op[:, -1]).reshape(B, Hv, Dv // 64, 64)
    assert np.all(err <= bound + 1e-12)
    assert err.max() > 0


def test_zero_beta_is_decay_of_the_quantized_state():
    d = _inputs(T=1, seed=9)
    zero = torch.zeros_like(d["beta"])
    for sm in ("e4m3", "int8"):
        o, S = decode(d["q"], d["k"], d["v"], zero, d["g"], d["h0"], state_mode=sm, block_v=32)
        B, Hv, Dk, Dv = d["h0"].shape
        Sq = oracle.qdq_groups(d["h0"].numpy().reshape(B * Hv, Dk, Dv), 32, sm)[0]
        Sq = Sq.reshape(B, Hv, Dk, Dv).astype(np.float64)
        a = np.exp(d["g"][:, 0].double().numpy())[:, :, None, None]
        assert _rel(S, a * Sq) <= 1e-15
        q = d["q"][:, 0].double().numpy()[:, np.arange(Hv) // (Hv // d["q"].shape[2])]
        assert _rel(o[:, 0], np.einsum("bhkv,bhk->bhv", a * Sq, q)) <= 1e-12


def test_single_token_calls_chain_like_one_call():
    d = _inputs(T=5, seed=10)
    o, S = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode="int8")
    s = d["h0"].numpy().astype(np.float64)
    for t in range(5):
        sl = lambda x: x[:, t:t + 1]
        ot, s = decode(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["beta"]), sl(d["g"]),
                       s, state_mode="int8")
        assert _rel(ot[:, 0], o[:, t]) <= 1e-12
    assert _rel(s, S) <= 1e-12


@pytest.mark.parametrize("P", [0, 64, 100])
@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_split_carry_prefill_then_decode(P, sm):
    """A chunked prefill of P tokens, its final state carried into decode, equals
    one torch recurrence that quantizes before t < P with t % 64 == 0 and before
    every t >= P."""
    d = _inputs(B=1, T=140, Hk=1, Hv=2, Dk=32, Dv=64, seed=P + 1)
    x = [d[n].double() for n in ("q", "k", "v", "beta", "g")]
    h0 = d["h0"].double()
    ref_o, ref_h = recurrent_torch(*x, h0=h0, state_mode=sm,
                                   quantize_before=lambda t: t >= P or t % 64 == 0)
    pre = [a[:, :P] for a in x]
    post = [a[:, P:] for a in x]
    if P:
        o_p, ht = chunked(*pre, h0, state_mode=sm, w_mode="none")
        assert _rel(o_p.numpy(), ref_o[:, :P].numpy()) <= 1e-10
    else:
        ht = h0
    o_d, S = decode(*post, ht.numpy(), state_mode=sm)
    assert _rel(o_d, ref_o[:, P:].numpy()) <= 1e-9
    assert _rel(S, ref_h.numpy()) <= 1e-9


@pytest.mark.parametrize("sm,readout", [("e4m3", "post"), ("int8", "pre"), ("none", "pre")])
def test_decode_scales_exactly_with_values_and_state(sm, readout):
    """o and the carried state are linear in (v, state) and the QDQ absorbs
    powers of two in s and 1/s: scaling both by 2^k scales o and the state by
    exactly 2^k in fp64."""
    d = _inputs(seed=61)
    S0 = torch.randn(2, 2, 32, 128, generator=torch.Generator().manual_seed(62)) * 0.3
    o, S = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], S0, state_mode=sm, readout=readout)
    for k in (-9, 4):
        f = 2.0 ** k
        v2 = (d["v"].float() * f).to(torch.bfloat16)
        assert torch.equal(v2.float(), d["v"].float() * f)
        o2, S2 = decode(d["q"], d["k"], v2, d["beta"], d["g"], S0 * f, state_mode=sm,
                        readout=readout)
        assert np.array_equal(o2, o * f) and np.array_equal(S2, S * f)
