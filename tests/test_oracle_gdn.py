"""Pins for the two GDN oracles (O1 token recurrence in C, O2 chunked WY form in torch).

Neither oracle is trusted on its own: each is checked against a hand-derived
case, closed forms (orthogonal keys, zero write strength), the delta-rule
invariant, the other formulation, structural identities of the WY form, and
finite-difference gradients.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.chunked import chunked, qdq_ste
from oracle.recurrent_torch import recurrent_torch
from gated_delta_rule_54_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _hand():
    with open(os.path.join(HERE, "golden", "hand_case_T3.json")) as f:
        c = json.load(f)
    t = lambda x: torch.tensor(x, dtype=torch.float32)
    q = t(c["q"])[None, :, None, :]
    k = t(c["k"])[None, :, None, :]
    v = t(c["v"])[None, :, None, :]
    beta = t(c["beta"])[None, :, None]
    g = torch.log(torch.tensor(c["alpha"], dtype=torch.float64)).float()[None, :, None]
    return c, q, k, v, beta, g


def test_hand_case_recurrent():
    c, q, k, v, beta, g = _hand()
    o, ht = oracle.recurrent(q, k, v, beta, g)
    # g = log(alpha) is carried in fp32, so exp(g) is alpha to ~3e-8 relative
    assert np.allclose(o[0, :, 0, :], np.array(c["o"]), atol=1e-6, rtol=0)
    # ht is H = S^T (Dk x Dv)
    assert np.allclose(ht[0, 0].T, np.array(c["S_final_v_by_k"]), atol=1e-6, rtol=0)


def test_hand_case_chunked():
    c, q, k, v, beta, g = _hand()
    for chunk in (64, 2, 1):
        o, ht = chunked(q, k, v, beta, g, chunk=chunk)
        assert np.allclose(o[0, :, 0, :].numpy(), np.array(c["o"]), atol=1e-6, rtol=0)
        assert np.allclose(ht[0, 0].T.numpy(), np.array(c["S_final_v_by_k"]), atol=1e-6)


def _unit_half_keys(rng, n, D):
    """Keys with four entries +-1/2: unit norm exactly in binary."""
    k = np.zeros((n, D), np.float32)
    for i in range(n):
        idx = rng.choice(D, 4, replace=False)
        k[i, idx] = 0.5 * rng.choice([-1, 1], 4)
    return k


def test_delta_rule_invariant_beta_one():
    # beta = 1, |k| = 1  =>  S_t k_t = v_t for any decay; read with q_t = k_t.
    rng = np.random.default_rng(0)
    T, D = 150, 16
    k = _unit_half_keys(rng, T, D)
    v = rng.standard_normal((T, D)).astype(np.float32)
    g = (-rng.uniform(0, 2, T)).astype(np.float32)
    h0 = rng.standard_normal((1, 1, D, D)).astype(np.float32)
    args = (k[None, :, None], k[None, :, None], v[None, :, None], np.ones((1, T, 1), np.float32),
            g[None, :, None], h0)
    o, _ = oracle.recurrent(*args)
    assert np.allclose(o[0, :, 0], v, atol=1e-12, rtol=0)
    o2, _ = chunked(*[torch.from_numpy(a) for a in args], chunk=64)
    assert np.allclose(o2[0, :, 0].numpy(), v, atol=1e-11, rtol=0)


def test_zero_beta_is_pure_decay():
    rng = np.random.default_rng(1)
    T, D = 70, 8
    q = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    k = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    g = (-rng.uniform(0, 0.1, (1, T, 1))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, D, D)).astype(np.float32)
    beta = np.zeros((1, T, 1), np.float32)
    o, ht = oracle.recurrent(q, k, v, beta, g, h0)
    cum = np.cumsum(g[0, :, 0].astype(np.float64))
    H0 = h0[0, 0].astype(np.float64)
    exp_o = np.exp(cum)[:, None] * (q[0, :, 0].astype(np.float64) @ H0)
    assert np.allclose(o[0, :, 0], exp_o, rtol=1e-12, atol=1e-13)
    assert np.allclose(ht[0, 0], np.exp(cum[-1]) * H0, rtol=1e-12, atol=1e-14)


def test_orthogonal_keys_closed_form():
    # keys e_0, e_1, ... (mutually orthogonal), h0 = 0: H_t^T k_j = 0 before the
    # write of token j, so o_t = sum_{j<=t} exp(sum_{s=j+1..t} g_s) b_j (k_j.q_t) v_j.
    rng = np.random.default_rng(2)
    T, D = 48, 64
    k = np.eye(D, dtype=np.float32)[:T][None, :, None]
    q = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, D)).astype(np.float32)
    b = rng.uniform(0.1, 1, (1, T, 1)).astype(np.float32)
    g = (-rng.uniform(0, 1, (1, T, 1))).astype(np.float32)
    cum = np.cumsum(g[0, :, 0].astype(np.float64))
    ref = np.zeros((T, D))
    for t in range(T):
        for j in range(t + 1):
            ref[t] += np.exp(cum[t] - cum[j]) * b[0, j, 0] * q[0, t, 0, j] * v[0, j, 0].astype(np.float64)
    o, _ = oracle.recurrent(q, k, v, b, g)
    assert np.allclose(o[0, :, 0], ref, rtol=1e-11, atol=1e-12)
    o2, _ = chunked(*[torch.from_numpy(a) for a in (q, k, v, b, g)], chunk=16)
    assert np.allclose(o2[0, :, 0].numpy(), ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("T", [1, 3, 63, 64, 65, 127, 128, 257])
def test_chunked_equals_recurrent_qdq_off(T):
    w = synth.small(T=T, B=2, Hk=2, Hv=4, Dk=32, Dv=32, h0=True, seed=T)
    d = synth.make_inputs(w)
    o1, h1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    o2, h2 = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    assert np.abs(o1 - o2.numpy()).max() <= 1e-10 * np.abs(o1).max()
    assert np.abs(h1 - h2.numpy()).max() <= 1e-10 * np.abs(h1).max()


def test_chunked_equals_recurrent_varlen_ragged():
    lengths = [1, 64, 97, 130, 5]
    w = synth.small(T=0, B=1, Hk=1, Hv=3, Dk=32, Dv=64, h0=True)
    d = synth.make_inputs(w, lengths=lengths)
    for sm in ("none", "e4m3", "int8"):
        o1, h1, c1, s1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                          cu_seqlens=d["cu_seqlens"], state_mode=sm,
                                          record_states=True)
        r = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                    cu_seqlens=d["cu_seqlens"], state_mode=sm, record=True)
        o2, h2 = r[0], r[1]
        assert np.abs(o1 - o2.numpy()).max() <= 1e-10 * np.abs(o1).max()
        assert np.abs(h1 - h2.numpy()).max() <= 1e-10 * np.abs(h1).max()
        if sm != "none":
            assert np.array_equal(c1, r[2]["state_codes"])
            assert np.array_equal(s1, r[2]["state_scales"])


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_state_qdq_recurrent_vs_chunked_codes_agree(sm):
    w = synth.small(T=300, B=2, Hk=2, Hv=4, Dk=64, Dv=128, h0=True, seed=5)
    d = synth.make_inputs(w)
    o1, h1, c1, s1 = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                      state_mode=sm, record_states=True)
    o2, h2, rec = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                          record=True)
    flips = np.mean(c1 != rec["state_codes"])
    assert flips == 0.0
    assert np.abs(o1 - o2.numpy()).max() <= 1e-10 * np.abs(o1).max()


def test_qdq_changes_output_and_none_is_unquantized():
    w = synth.small(T=130, Hk=2, Hv=2, Dk=32, Dv=64, h0=True)
    d = synth.make_inputs(w)
    a = [d[x] for x in ("q", "k", "v", "beta", "g", "h0")]
    o0, _ = chunked(*a)
    for sm, wm in (("e4m3", "none"), ("none", "e4m3"), ("int8", "e4m3")):
        o, _ = chunked(*a, state_mode=sm, w_mode=wm)
        assert (o - o0).abs().max() > 1e-4 * o0.abs().max()
    o1, _ = oracle.recurrent(*a)
    assert np.abs(o1 - o0.numpy()).max() <= 1e-10 * np.abs(o1).max()


def test_wy_structure_identities():
    w = synth.small(T=200, Hk=2, Hv=2, Dk=64, Dv=64, h0=True)
    d = synth.make_inputs(w)
    _, _, inter = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                          state_mode="e4m3", w_mode="e4m3", intermediates=True)
    for st in inter[0]:
        A, T = st["A"], st["T"]
        L = A.shape[-1]
        I = torch.eye(L, dtype=torch.float64)
        assert (T @ (I + A) - I).abs().max() <= 1e-12
        assert torch.all(torch.triu(A) == 0)
        # W-QDQ: one scale per (head, chunk) tile; its amax element lands on +-448 * scale
        Wf = st["W"].float()
        for h in range(Wf.shape[0]):
            a = Wf[h].abs().max()
            s = a / 448.0
            i = Wf[h].abs().argmax()
            assert st["W_hat"][h].flatten()[i].abs().float() == 448.0 * s


def test_orthogonal_keys_in_chunk_give_identity_solve():
    D, L = 64, 32
    k = torch.eye(D)[:L][None, :, None]
    rng = np.random.default_rng(3)
    q = torch.from_numpy(rng.standard_normal((1, L, 1, D)).astype(np.float32))
    v = torch.from_numpy(rng.standard_normal((1, L, 1, D)).astype(np.float32))
    b = torch.from_numpy(rng.uniform(0.1, 1, (1, L, 1)).astype(np.float32))
    g = torch.from_numpy((-rng.uniform(0, 1, (1, L, 1))).astype(np.float32))
    _, _, inter = chunked(q, k, v, b, g, intermediates=True)
    st = inter[0][0]
    assert torch.all(st["A"] == 0)
    assert torch.equal(st["T"][0], torch.eye(L, dtype=torch.float64))
    gam = torch.cumsum(g[0, :, 0].double(), 0)
    W_ref = (b[0, :, 0].double() * torch.exp(gam))[:, None] * k[0, :, 0].double()
    assert torch.allclose(st["W"][0], W_ref, rtol=1e-14, atol=0)


def test_u_solves_the_unit_lower_system():
    w = synth.small(T=64, Hk=1, Hv=1, Dk=32, Dv=32)
    d = synth.make_inputs(w)
    _, _, inter = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], intermediates=True)
    st = inter[0][0]
    I = torch.eye(64, dtype=torch.float64)
    bV = d["beta"][0, :, 0].double()[:, None] * d["v"][0, :, 0].double()
    assert ((I + st["A"][0]) @ st["U"][0] - bV).abs().max() <= 1e-12 * bV.abs().max()


def _small_grad_inputs(T=5, Dk=4, Dv=4, Hk=1, Hv=2, seed=0, h0=True):
    g_ = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g_, dtype=torch.float64)
    q = r(1, T, Hk, Dk) * 0.5
    k = r(1, T, Hk, Dk) * 0.5
    v = r(1, T, Hv, Dv)
    beta = torch.sigmoid(r(1, T, Hv))
    g = -torch.nn.functional.softplus(r(1, T, Hv))
    h = r(1, Hv, Dk, Dv) * 0.3 if h0 else None
    xs = [q, k, v, beta, g] + ([h] if h0 else [])
    return [x.requires_grad_(True) for x in xs]


def test_gradcheck_chunked_qdq_off():
    xs = _small_grad_inputs()

    def f(q, k, v, beta, g, h0):
        o, ht = chunked(q, k, v, beta, g, h0, chunk=4)
        return o, ht

    assert torch.autograd.gradcheck(f, xs, eps=1e-6, atol=1e-7, rtol=1e-6)


def test_chunked_grads_equal_recurrent_grads_with_state_ste():
    """Identity STE through the state QDQ: autograd of the chunked form equals
    autograd of the token recurrence with the same QDQ placement (W-QDQ off)."""
    for sm in ("none", "e4m3", "int8"):
        xs = _small_grad_inputs(T=11, Dk=8, Dv=8, Hk=1, Hv=2, seed=3)
        gen = torch.Generator().manual_seed(9)
        do = torch.randn(1, 11, 2, 8, generator=gen, dtype=torch.float64)
        dht = torch.randn(1, 2, 8, 8, generator=gen, dtype=torch.float64)
        o, ht = chunked(*xs, chunk=4, block_v=4, state_mode=sm)
        ga = torch.autograd.grad((o * do).sum() + (ht * dht).sum(), xs)
        o2, ht2 = recurrent_torch(*xs, chunk=4, block_v=4, state_mode=sm)
        assert torch.allclose(o, o2, rtol=1e-10, atol=1e-12)
        gb = torch.autograd.grad((o2 * do).sum() + (ht2 * dht).sum(), xs)
        for a, b in zip(ga, gb):
            assert torch.allclose(a, b, rtol=1e-9, atol=1e-11)


def test_qdq_ste_backward_is_identity():
    x = torch.randn(3, 8, 16, dtype=torch.float64, requires_grad=True)
    wgt = torch.randn(3, 8, 16, dtype=torch.float64)
    for mode in ("e4m3", "int8"):
        y = qdq_ste(x, mode, 8)
        (gx,) = torch.autograd.grad((y * wgt).sum(), x)
        assert torch.equal(gx, wgt)
        ref, _ = oracle.qdq_groups(x.detach().float().numpy(), 8, mode)
        assert np.array_equal(y.detach().float().numpy(), ref)


# ---- Neumann approximate inverse ("[7/7] Experimental GDN/KDA approximate-inverse QAT") ----
from oracle.chunked import neumann_inverse


def test_neumann_inverse_identities():
    """(I + A) T_d = I - (-A)^{d+1} (the residual identity of the polynomial);
    degree 0 is I; the product form prod_j (I + X^{2^j}) equals the sum for
    d = 2^m - 1; degree >= L - 1 is the exact inverse (A is nilpotent)."""
    rng = np.random.default_rng(5)
    L = 24
    A = torch.from_numpy(np.tril(rng.standard_normal((2, L, L)) * 0.3, -1))
    I = torch.eye(L, dtype=torch.float64)
    for d in (0, 1, 3, 7, 10):
        T = neumann_inverse(A, d)
        Xd1 = torch.linalg.matrix_power(-A, d + 1)
        assert ((I + A) @ T - (I - Xd1)).abs().max() <= 1e-12 * max(1.0, Xd1.abs().max().item())
    assert torch.equal(neumann_inverse(A, 0), I.expand(2, L, L))
    X = -A
    prod = (I + X) @ (I + X @ X) @ (I + torch.linalg.matrix_power(X, 4))
    assert (prod - neumann_inverse(A, 7)).abs().max() <= 1e-12 * prod.abs().max()
    exact = torch.linalg.solve_triangular(I + A, I.expand(2, L, L), upper=False, unitriangular=True)
    assert (neumann_inverse(A, L - 1) - exact).abs().max() <= 1e-10 * exact.abs().max()


def test_chunked_neumann_degree_63_is_the_exact_solve():
    w = synth.small(B=1, T=150, Hk=1, Hv=2, Dk=32, Dv=64, h0=True, seed=12)
    d = synth.make_inputs(w)
    o1, h1 = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode="e4m3",
                     w_mode="e4m3")
    o2, h2 = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode="e4m3",
                     w_mode="e4m3", neumann_degree=63)
    assert (o1 - o2).abs().max() <= 1e-9 * o1.abs().max()
    assert (h1 - h2).abs().max() <= 1e-9 * h1.abs().max()
    o3, _ = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode="e4m3",
                    w_mode="e4m3", neumann_degree=3)
    assert (o1 - o3).abs().max() > 1e-6 * o1.abs().max()   # a low degree is not the inverse


def test_gradcheck_chunked_neumann():
    """The backward differentiates the actual polynomial."""
    w = synth.small(B=1, T=20, Hk=1, Hv=1, Dk=4, Dv=3, h0=True, seed=13)
    d = synth.make_inputs(w)
    xs = [d[n].double().requires_grad_(True) for n in ("q", "k", "v", "beta", "g", "h0")]

    def f(*a):
        o, ht = chunked(*a, chunk=8, neumann_degree=3)
        return o.sum() + (ht * ht).sum()
    assert torch.autograd.gradcheck(f, xs, eps=1e-6, atol=1e-7, rtol=1e-6)


@pytest.mark.parametrize("sm,wm", [("e4m3", "e4m3"), ("int8", "e4m3"), ("none", "none")])
def test_chunked_scales_exactly_with_values_and_state(sm, wm):
    """o and ht are linear in (v, h0) and the QDQ is equivariant under powers
    of two (s and 1/s absorb them exactly), while W does not involve v: scaling
    v and h0 by 2^k scales o and ht by exactly 2^k, bit for bit in fp64."""
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=41)
    d = synth.make_inputs(w)
    o, ht = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm, w_mode=wm)
    for k in (-7, 3):
        f = 2.0 ** k
        v2 = (d["v"].float() * f).to(torch.bfloat16)
        assert torch.equal(v2.float(), d["v"].float() * f)     # exact in bf16
        o2, ht2 = chunked(d["q"], d["k"], v2, d["beta"], d["g"], d["h0"] * f, state_mode=sm,
                          w_mode=wm)
        assert torch.equal(o2, o * f) and torch.equal(ht2, ht * f)


@pytest.mark.parametrize("sm,wm", [("e4m3", "e4m3"), ("int8", "none")])
def test_chunked_packed_equals_separate_calls(sm, wm):
    """cu_seqlens only says where each sequence's rows sit: the packed call gives
    every sequence exactly the outputs and final state of a call on that
    sequence alone (chunks restart at every sequence start)."""
    lengths = [70, 130, 64, 1]
    w = synth.small(B=1, T=0, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=65)
    d = synth.make_inputs(w, lengths=lengths)
    o, ht = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                    cu_seqlens=d["cu_seqlens"], state_mode=sm, w_mode=wm)
    start = 0
    for n, L in enumerate(lengths):
        sl = lambda x: x[:, start:start + L]
        o1, ht1 = chunked(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["beta"]), sl(d["g"]),
                          d["h0"][n:n + 1], state_mode=sm, w_mode=wm)
        assert torch.equal(o1, o[:, start:start + L]) and torch.equal(ht1, ht[n:n + 1])
        start += L
