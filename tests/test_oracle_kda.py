"""Pins for the KDA recurrent oracle (oracle/kda.py): a hand-derived case with
distinct channel decays, reduction to the GDN token recurrence when every
channel decays alike (all QDQ modes, packed sequences, grouped heads), the
delta-rule invariant, and the zero-write-strength closed form."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.kda import kda_recurrent
from gated_delta_rule_54_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_hand_case():
    with open(os.path.join(HERE, "golden", "kda_hand_case.json")) as f:
        c = json.load(f)
    a = np.array(c["alpha"])
    q = np.array(c["q"])[None, :, None, :]
    k = np.array(c["k"])[None, :, None, :]
    v = np.array(c["v"])[None, :, None, :]
    beta = np.array(c["beta"])[None, :, None]
    g = np.log(a)[None, :, None, :]
    h0 = np.array(c["h0"])[None, None]
    o, ht = kda_recurrent(q, k, v, beta, g, h0)
    assert np.allclose(o[0, :, 0], np.array(c["o"]), atol=1e-6, rtol=0)
    assert np.allclose(ht[0, 0], np.array(c["ht"]), atol=1e-6, rtol=0)


def _gdn_case(lengths=None, sm="none", seed=0, Hk=2, Hv=4):
    w = synth.small(B=2 if lengths is None else 1, T=150 if lengths is None else 0, Hk=Hk, Hv=Hv,
                    Dk=32, Dv=64, h0=True, seed=seed)
    d = synth.make_inputs(w, lengths=lengths)
    gk = d["g"][..., None].expand(*d["g"].shape, 32).contiguous()     # same decay on every channel
    return d, gk


@pytest.mark.parametrize("sm", ["none", "e4m3", "int8"])
def test_channel_constant_decay_is_the_gdn_recurrence(sm):
    d, gk = _gdn_case(sm=sm, seed=1)
    o, ht = kda_recurrent(d["q"], d["k"], d["v"], d["beta"], gk, d["h0"], state_mode=sm)
    o1, h1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm)
    assert np.abs(o - o1).max() <= 1e-10 * np.abs(o1).max()
    assert np.abs(ht - h1).max() <= 1e-10 * np.abs(h1).max()


def test_channel_constant_decay_packed_sequences():
    lengths = [1, 64, 97, 5]
    d, gk = _gdn_case(lengths=lengths, seed=2)
    for sm in ("none", "int8"):
        o, ht = kda_recurrent(d["q"], d["k"], d["v"], d["beta"], gk, d["h0"],
                              cu_seqlens=d["cu_seqlens"], state_mode=sm, block_v=32)
        o1, h1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                  cu_seqlens=d["cu_seqlens"], state_mode=sm, block_v=32)
        assert np.abs(o - o1).max() <= 1e-10 * np.abs(o1).max()
        assert np.abs(ht - h1).max() <= 1e-10 * np.abs(h1).max()


def test_delta_rule_invariant_with_channel_decay():
    # beta = 1, |k| = 1: H^T k = v after each write, whatever the decays
    rng = np.random.default_rng(3)
    T, D = 40, 16
    k = np.zeros((1, T, 1, D), np.float32)
    for t in range(T):
        k[0, t, 0, rng.choice(D, 4, replace=False)] = 0.5 * rng.choice([-1, 1], 4)
    v = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    g = (-rng.uniform(0, 2, (1, T, 1, D))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, D, D)).astype(np.float32)
    o, _ = kda_recurrent(k, k, v, np.ones((1, T, 1), np.float32), g, h0, scale=0.5)
    assert np.abs(o[0, :, 0] - 0.5 * v[0, :, 0]).max() <= 1e-12


def test_zero_beta_is_per_channel_decay():
    rng = np.random.default_rng(4)
    T, Dk, Dv = 20, 8, 6
    q = rng.standard_normal((1, T, 1, Dk)).astype(np.float32)
    k = rng.standard_normal((1, T, 1, Dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, Dv)).astype(np.float32)
    g = (-rng.uniform(0, 0.3, (1, T, 1, Dk))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, Dk, Dv)).astype(np.float32)
    o, ht = kda_recurrent(q, k, v, np.zeros((1, T, 1), np.float32), g, h0)
    cum = np.cumsum(g[0, :, 0].astype(np.float64), 0)                   # [T, Dk]
    H0 = h0[0, 0].astype(np.float64)
    for t in range(T):
        ref = (np.exp(cum[t])[:, None] * H0).T @ q[0, t, 0].astype(np.float64)
        assert np.allclose(o[0, t, 0], ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(ht[0, 0], np.exp(cum[-1])[:, None] * H0, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("sm", ["e4m3", "int8", "none"])
def test_kda_scales_exactly_with_values_and_state(sm):
    """Linear in (v, h0), with a QDQ that absorbs powers of two: scaling both by
    2^k scales o and ht by exactly 2^k in fp64."""
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=64, Dv=64, w_mode="none", h0=True, seed=63)
    d = synth.make_kda_inputs(w)
    o, ht = kda_recurrent(d["q"], d["k"], d["v"], d["beta"], d["g_k"], d["h0"], state_mode=sm)
    for k in (-9, 4):
        f = 2.0 ** k
        v2 = (d["v"].float() * f).to(torch.bfloat16)
        assert torch.equal(v2.float(), d["v"].float() * f)
        o2, ht2 = kda_recurrent(d["q"], d["k"], v2, d["beta"], d["g_k"], d["h0"] * f,
                                state_mode=sm)
        assert np.array_equal(np.asarray(o2), np.asarray(o) * f)
        assert np.array_equal(np.asarray(ht2), np.asarray(ht) * f)
