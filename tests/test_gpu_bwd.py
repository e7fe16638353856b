"""GPU parity of the identity-STE backward (gdn_chunk_bwd_ste, through the C ABI)
against autograd of the fp64 chunked oracle (which applies QDQ as
x + (Q(x) - x).detach(), i.e. the identity straight-through estimator).

Tolerance: relative L2 error <= 2e-2 per gradient tensor.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_chunk_bwd_ste, gdn_chunk_fwd_qdq, synth
from oracle.chunked import chunked

from _parity import GRAD_L2, grad_rel_l2, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


def _grads_gpu(d, sm, wm, do, dht, scale=1.0, block_v=64, neumann_degree=None):
    dd = to_dev(d)
    cu = dd["cu_seqlens"]
    o, ht, ctx = gdn_chunk_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                   cu_seqlens=cu, scale=scale, state_mode=sm, w_mode=wm,
                                   save_ctx=True, block_v=block_v, neumann_degree=neumann_degree)
    gr = gdn_chunk_bwd_ste(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], ctx, do.cuda(),
                           dht.cuda() if dht is not None else None, cu_seqlens=cu, scale=scale,
                           state_mode=sm, w_mode=wm, block_v=block_v,
                           neumann_degree=neumann_degree)
    torch.cuda.synchronize()
    return [x.cpu().double().numpy() for x in gr]


def _grads_oracle(d, sm, wm, do, dht, scale=1.0, cu=None, block_v=64, neumann_degree=None):
    N, Hv = d["N"], d["v"].shape[2]
    h0 = d["h0"] if d["h0"] is not None else torch.zeros(N, Hv, d["k"].shape[3], d["v"].shape[3])
    xs = [t.double().requires_grad_(True) for t in (d["q"], d["k"], d["v"], d["beta"], d["g"], h0)]
    o, ht = chunked(*xs, cu_seqlens=cu, scale=scale, state_mode=sm, w_mode=wm, block_v=block_v,
                    neumann_degree=neumann_degree)
    loss = (o * do.double()).sum() + ((ht * dht.double()).sum() if dht is not None else 0.0)
    return [g.numpy() for g in torch.autograd.grad(loss, xs)]


def _dO(w, d, seed=11, with_dht=True):
    gen = torch.Generator().manual_seed(seed)
    B, T = d["B"], d["T"]
    do = torch.randn(B, T, w.Hv, w.Dv, generator=gen).to(torch.bfloat16)
    dht = torch.randn(d["N"], w.Hv, w.Dk, w.Dv, generator=gen) * 0.01 if with_dht else None
    return do, dht


def _check(w, lengths=None, scale=1.0, with_dht=True, block_v=64, neumann_degree=None):
    d = synth.make_inputs(w, lengths=lengths)
    do, dht = _dO(w, d, with_dht=with_dht)
    g = _grads_gpu(d, w.state_mode, w.w_mode, do, dht, scale, block_v=block_v,
                   neumann_degree=neumann_degree)
    r = _grads_oracle(d, w.state_mode, w.w_mode, do, dht, scale, d["cu_seqlens"], block_v=block_v,
                      neumann_degree=neumann_degree)
    errs = {}
    for name, a, b in zip(NAMES, g, r):
        assert np.isfinite(a).all(), name
        errs[name] = grad_rel_l2(a, b)
    bad = {k: v for k, v in errs.items() if not v <= GRAD_L2}
    assert not bad, "relative L2 errors above %.0e: %s (all: %s)" % (GRAD_L2, bad, errs)
    return errs


MODES = [("e4m3", "e4m3"), ("int8", "e4m3"), ("none", "none"), ("e4m3", "none"),
         ("none", "e4m3"), ("int8", "int8")]


@pytest.mark.parametrize("sm,wm", MODES)
def test_bwd_modes(sm, wm):
    w = synth.small(B=2, T=200, Hk=2, Hv=2, Dk=128, Dv=128, state_mode=sm, w_mode=wm, h0=True,
                    seed=21)
    _check(w)


@pytest.mark.parametrize("block_v", [16, 32, 128])
def test_bwd_state_scale_widths(block_v):
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128, state_mode="int8", h0=True,
                    seed=40 + block_v)
    _check(w, block_v=block_v)


@pytest.mark.parametrize("degree", [1, 3, 7])
def test_bwd_neumann_solve(degree):
    """The backward differentiates the actual Neumann polynomial."""
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128, h0=True, seed=50 + degree)
    _check(w, neumann_degree=degree)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_bwd_lengths(T):
    w = synth.small(B=2, T=T, Hk=1, Hv=1, Dk=64, Dv=64, h0=True, seed=100 + T)
    _check(w)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_bwd_lengths_tensor_core_path(T):
    """Dk = Dv = 128 with both sites quantized and block_v 64 takes the tcgen05
    chunk kernel (P, Gamma o KK^T and Delta recomputed): ragged chunk tails."""
    w = synth.small(B=2, T=T, Hk=1, Hv=2, Dk=128, Dv=128, h0=True, seed=110 + T)
    _check(w, scale=128 ** -0.5, with_dht=T % 2 == 1)


def test_bwd_scan_two_blocks_per_cta():
    """80 (sequence, head) chains are more than fit twice on the SMs, so the
    reverse scan covers both value blocks in one CTA (the small cases above
    take one block per CTA)."""
    w = synth.small(B=5, T=70, Hk=16, Hv=16, Dk=128, Dv=128, h0=True, seed=61)
    _check(w)


def test_bwd_grouped_heads_int8():
    w = synth.small(B=1, T=150, Hk=2, Hv=6, Dk=128, Dv=128, state_mode="int8", h0=True, seed=22)
    _check(w)


def test_bwd_packed_ragged():
    lengths = [0, 1, 70, 128, 33, 200]
    w = synth.small(B=1, T=0, Hk=2, Hv=2, Dk=128, Dv=128, h0=True, seed=23)
    _check(w, lengths=lengths)


def test_bwd_dims_scale_and_no_dht():
    w = synth.small(B=1, T=140, Hk=1, Hv=2, Dk=64, Dv=128, h0=True, seed=24)
    _check(w, scale=64 ** -0.5, with_dht=False)
    w = synth.small(B=1, T=140, Hk=1, Hv=1, Dk=128, Dv=64, h0=False, seed=25)
    _check(w)
    w = synth.small(B=2, T=100, Hk=2, Hv=2, Dk=64, Dv=64, h0=True, seed=27)
    _check(w)


def test_bwd_deterministic():
    w = synth.small(B=2, T=260, Hk=2, Hv=4, Dk=128, Dv=128, h0=True, seed=26)
    d = synth.make_inputs(w)
    do, dht = _dO(w, d)
    a = _grads_gpu(d, "e4m3", "e4m3", do, dht)
    b = _grads_gpu(d, "e4m3", "e4m3", do, dht)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_full_fwd_bwd_workload_sampled():
    """B=8, T=4096, H=16, D=128 forward + backward in the benchmark's launch
    configuration; gradients of sampled (sequence, head) sub-problems against
    the oracle (heads and sequences are independent, so sub-problems are exact)."""
    w = synth.WORKLOADS["fwd_bwd"]
    d = synth.make_inputs(w)
    g = _grads_gpu(d, w.state_mode, w.w_mode, d["do"], d["dht"])
    for n, hk in [(0, 0), (7, 15), (3, 9)]:
        sub = dict(q=d["q"][n:n + 1, :, hk:hk + 1], k=d["k"][n:n + 1, :, hk:hk + 1],
                   v=d["v"][n:n + 1, :, hk:hk + 1], beta=d["beta"][n:n + 1, :, hk:hk + 1],
                   g=d["g"][n:n + 1, :, hk:hk + 1], h0=d["h0"][n:n + 1, hk:hk + 1], N=1)
        r = _grads_oracle(sub, w.state_mode, w.w_mode, d["do"][n:n + 1, :, hk:hk + 1],
                          d["dht"][n:n + 1, hk:hk + 1])
        got = [g[0][n:n + 1, :, hk:hk + 1], g[1][n:n + 1, :, hk:hk + 1], g[2][n:n + 1, :, hk:hk + 1],
               g[3][n:n + 1, :, hk:hk + 1], g[4][n:n + 1, :, hk:hk + 1], g[5][n:n + 1, hk:hk + 1]]
        for name, a, b in zip(NAMES, got, r):
            e = grad_rel_l2(a, b)
            assert e <= GRAD_L2, "%s (n=%d, h=%d): relative L2 %.3e" % (name, n, hk, e)


def test_autograd_op_matches_the_oracle_gradients():
    """gdn_chunk_qdq (forward + STE backward as one autograd op) against the
    oracle's autograd, with bf16 q/k/v gradients as autograd hands them back."""
    import torch
    from gated_delta_rule_54_gb300 import gdn_chunk_qdq
    from oracle.chunked import chunked
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=77)
    d = synth.make_inputs(w)
    names = ("q", "k", "v", "beta", "g", "h0")
    xs = [d[n].cuda().requires_grad_(True) for n in names]
    o, ht = gdn_chunk_qdq(*xs, state_mode="e4m3", w_mode="e4m3")
    gen = torch.Generator().manual_seed(78)
    do = torch.randn(o.shape, generator=gen).to(torch.bfloat16).float()
    dht = torch.randn(ht.shape, generator=gen) * 0.01
    ((o * do.cuda()).sum() + (ht * dht.cuda()).sum()).backward()
    rs = [d[n].double().requires_grad_(True) for n in names]
    o2, ht2 = chunked(*rs, state_mode="e4m3", w_mode="e4m3")
    ((o2 * do.double()).sum() + (ht2 * dht.double()).sum()).backward()
    for n, x, r in zip(names, xs, rs):
        gx = x.grad.double().cpu()
        rel = float((gx - r.grad).norm() / r.grad.norm())
        assert x.grad.dtype == x.dtype and torch.isfinite(gx).all()
        # bf16 gradients of q, k, v add a 2^-9 relative rounding to the STE bound
        assert rel <= GRAD_L2 + (2.0 ** -8 if x.dtype == torch.bfloat16 else 0.0), (n, rel)


def _random_case(seed):
    rng = np.random.default_rng(2000 + seed)
    Dk = int(rng.choice([64, 128]))
    Dv = int(rng.choice([64, 128]))
    Hk = int(rng.choice([1, 2]))
    Hv = Hk * int(rng.choice([1, 2]))
    sm, wm = MODES[int(rng.integers(len(MODES)))]
    block_v = int(rng.choice([16, 32, 64] + ([128] if Dv == 128 else [])))
    packed = bool(rng.integers(2))
    if packed:
        lengths = [int(x) for x in rng.integers(0, 160, size=int(rng.integers(1, 5)))]
        if sum(lengths) == 0:
            lengths[0] = 1
        w = synth.small(B=1, T=0, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, state_mode=sm, w_mode=wm, h0=True,
                        seed=400 + seed)
    else:
        lengths = None
        w = synth.small(B=int(rng.integers(1, 3)), T=int(rng.integers(1, 200)), Hk=Hk, Hv=Hv,
                        Dk=Dk, Dv=Dv, state_mode=sm, w_mode=wm, h0=bool(rng.integers(2)),
                        seed=400 + seed)
    return w, lengths, block_v, float(rng.choice([1.0, Dk ** -0.5])), bool(rng.integers(2))


@pytest.mark.parametrize("seed", range(12))
def test_bwd_randomized(seed):
    """Seeded random mixes of head dims, grouped heads, both QDQ sites' modes,
    state-scale widths, packed lengths (empty sequences included), scale and
    dht presence: every gradient within the relative L2 bound of the oracle's
    autograd (this covers the tensor-core and the warp-level paths alike)."""
    w, lengths, block_v, scale, with_dht = _random_case(seed)
    _check(w, lengths=lengths, scale=scale, with_dht=with_dht, block_v=block_v)
