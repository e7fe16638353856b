"""GPU parity of the two-precision backward (gdn_two_precision_bwd, the
window-wise adjoint, through the C ABI) against autograd of the fp64 oracle
``oracle.two_precision.two_precision_torch`` (read copy through the identity
straight-through estimator).

Tolerances, per gradient tensor, relative L2:
  * E4M3 read copy: <= 2e-2, the chunked backward's bound.  The kernels take
    the read codes from their own fp32 anchor, so a code whose oracle value
    sits within fp32 error of a rounding boundary may land one step away; the
    step enters the outputs and every gradient of its window, which the
    relative L2 bound absorbs.
  * read copy off: <= 1e-4.  Then nothing is quantized and the only difference
    is fp32 against fp64 arithmetic over a few hundred token steps (relative
    rounding 2^-24 per operation, far below this bound)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_two_precision_bwd, gdn_two_precision_fwd, synth
from oracle.two_precision import two_precision_torch

from _parity import GRAD_L2, grad_rel_l2, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dh0")
READ_OFF_L2 = 1e-4


def _upstream(d, seed=11, with_dht=True):
    gen = torch.Generator().manual_seed(seed)
    B, T, Hv, Dv = d["v"].shape
    do = torch.randn(B, T, Hv, Dv, generator=gen)
    dht = (torch.randn(d["N"], Hv, d["k"].shape[3], Dv, generator=gen) * 0.1
           if with_dht else None)
    return do, dht


def _grads_gpu(d, do, dht, rm, flush, scale):
    dd = to_dev(d)
    cu = dd["cu_seqlens"]
    o, ht, anchors = gdn_two_precision_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"],
                                           dd["h0"], cu_seqlens=cu, scale=scale, read_mode=rm,
                                           flush=flush, save_anchors=True)
    gr = gdn_two_precision_bwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], anchors,
                               do.cuda(), dht.cuda() if dht is not None else None,
                               cu_seqlens=cu, scale=scale, read_mode=rm, flush=flush)
    torch.cuda.synchronize()
    return [x.cpu().double().numpy() for x in gr]


def _grads_oracle(d, do, dht, rm, flush, scale):
    N, Hv = d["N"], d["v"].shape[2]
    h0 = d["h0"] if d["h0"] is not None else torch.zeros(N, Hv, d["k"].shape[3], d["v"].shape[3])
    xs = [t.to(torch.float32).double().requires_grad_(True)
          for t in (d["q"], d["k"], d["v"], d["beta"], d["g"], h0)]
    o, ht = two_precision_torch(*xs, cu_seqlens=d["cu_seqlens"], scale=scale, read_mode=rm,
                                flush=flush)
    loss = (o * do.double()).sum() + ((ht * dht.double()).sum() if dht is not None else 0.0)
    return [g.numpy() for g in torch.autograd.grad(loss, xs)]


def _compare(g, r, rm, what=""):
    tol = GRAD_L2 if rm == "e4m3" else READ_OFF_L2
    errs = {}
    for name, a, b in zip(NAMES, g, r):
        assert np.isfinite(a).all(), name
        errs[name] = grad_rel_l2(a, b)
    print("%s read=%s rel L2: %s" % (what, rm, {k: "%.2e" % v for k, v in errs.items()}))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, "relative L2 errors above %.0e: %s (all: %s)" % (tol, bad, errs)
    return errs


def _check(w, lengths=None, rm="e4m3", flush=16, scale=1.0, h0=True, with_dht=True, seed=11):
    d = synth.make_inputs(w, lengths=lengths)
    if not h0:
        d["h0"] = None
    do, dht = _upstream(d, seed, with_dht)
    g = _grads_gpu(d, do, dht, rm, flush, scale)
    r = _grads_oracle(d, do, dht, rm, flush, scale)
    return _compare(g, r, rm)


@pytest.mark.parametrize("rm", ["e4m3", "none"])
@pytest.mark.parametrize("flush", [1, 5, 16, 64])
def test_two_precision_bwd_modes_and_flush(rm, flush):
    # grouped heads (two value heads per key head), Dv = 128: eight column groups per cluster
    w = synth.small(B=2, T=150, Hk=2, Hv=4, Dk=128, Dv=128, w_mode="none", h0=True, seed=40 + flush)
    _check(w, rm=rm, flush=flush)


@pytest.mark.parametrize("T", [1, 3, 15, 16, 17, 70])
def test_two_precision_bwd_lengths_dv64(T):
    # Dv = 64: four column groups per cluster; windows and staged blocks with ragged tails
    w = synth.small(B=2, T=T, Hk=1, Hv=2, Dk=128, Dv=64, w_mode="none", h0=True, seed=50 + T)
    _check(w, flush=16)


def test_two_precision_bwd_packed_grouped_scaled():
    w = synth.small(B=1, T=0, Hk=2, Hv=4, Dk=128, Dv=64, w_mode="none", h0=True, seed=60)
    _check(w, lengths=[0, 5, 130, 16, 77], scale=0.125, flush=5)


def test_two_precision_bwd_no_h0_no_dht():
    w = synth.small(B=3, T=40, Hk=1, Hv=1, Dk=128, Dv=128, w_mode="none", seed=61)
    _check(w, h0=False, with_dht=False, flush=7)


@pytest.mark.parametrize("T,flush", [(100, 200), (300, 256), (40, 33)])
def test_two_precision_bwd_long_windows(T, flush):
    # one window longer than the sequence; the longest window replayed; W not a multiple of 4
    w = synth.small(B=1, T=T, Hk=1, Hv=2, Dk=128, Dv=128, w_mode="none", h0=True, seed=62 + T)
    _check(w, flush=flush)


def test_two_precision_bwd_is_repeatable():
    """Column sums go through the cluster in a fixed order: two calls agree bit
    for bit."""
    w = synth.small(B=2, T=90, Hk=2, Hv=4, Dk=128, Dv=128, w_mode="none", h0=True, seed=63)
    d = synth.make_inputs(w)
    do, dht = _upstream(d)
    a = _grads_gpu(d, do, dht, "e4m3", 16, 1.0)
    b = _grads_gpu(d, do, dht, "e4m3", 16, 1.0)
    for name, x, y in zip(NAMES, a, b):
        assert np.array_equal(x, y), name


def test_two_precision_bwd_empty_sequences_pass_dht():
    """A sequence without tokens: dh0 = dht, and no other output is touched."""
    w = synth.small(B=1, T=0, Hk=1, Hv=2, Dk=128, Dv=64, w_mode="none", h0=True, seed=64)
    d = synth.make_inputs(w, lengths=[0, 0])
    dd = to_dev(d)
    do, dht = _upstream(d)
    _, _, anchors = gdn_two_precision_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                          cu_seqlens=dd["cu_seqlens"], save_anchors=True)
    gr = gdn_two_precision_bwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], anchors, do.cuda(),
                               dht.cuda(), cu_seqlens=dd["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(gr[5].cpu(), dht)


def test_two_precision_bwd_full_size_sampled_head():
    """The two-precision workload (B4 T4096 H16 D128, E4M3 reads, 16-token
    flush) in one call; the gradients of sequence 0, head 11, against the oracle
    run on that (sequence, head) slice alone (heads do not interact: one value
    head per key head).  The oracle's autograd over 4096 tokens takes about a
    minute, so one head is sampled."""
    w = synth.WORKLOADS["two_precision"]
    assert w.Hk == w.Hv
    d = synth.make_inputs(w)
    do, dht = _upstream(d, seed=12)
    g = _grads_gpu(d, do, dht, "e4m3", 16, 1.0)
    for h in (11,):
        sub = {n: d[n][:1, :, h:h + 1] for n in ("q", "k", "v", "beta", "g")}
        sub["h0"] = d["h0"][:1, h:h + 1]
        sub["N"], sub["cu_seqlens"] = 1, None
        r = _grads_oracle(sub, do[:1, :, h:h + 1], dht[:1, h:h + 1], "e4m3", 16, 1.0)
        gs = [x[:1, :, h:h + 1] for x in g[:5]] + [g[5][:1, h:h + 1]]
        _compare(gs, r, "e4m3", "full size, head %d:" % h)


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    Dv = int(rng.choice([64, 128]))
    Hk = int(rng.choice([1, 2]))
    Hv = Hk * int(rng.choice([1, 2]))
    packed = bool(rng.integers(2))
    flush = int(rng.choice([1, 2, 3, 4, 7, 16, 17, 40, 64, 100, 256]))
    rm = str(rng.choice(["e4m3", "none"]))
    if packed:
        lengths = [int(x) for x in rng.integers(0, 90, size=int(rng.integers(1, 5)))]
        w = synth.small(B=1, T=0, Hk=Hk, Hv=Hv, Dk=128, Dv=Dv, w_mode="none", h0=True,
                        seed=200 + seed)
    else:
        lengths = None
        w = synth.small(B=int(rng.integers(1, 3)), T=int(rng.integers(1, 140)), Hk=Hk, Hv=Hv,
                        Dk=128, Dv=Dv, w_mode="none", h0=True, seed=200 + seed)
    return w, lengths, rm, flush, float(rng.choice([1.0, 0.125])), bool(rng.integers(2)), \
        bool(rng.integers(2))


@pytest.mark.parametrize("seed", range(12))
def test_two_precision_bwd_randomized(seed):
    """Seeded random mixes of shapes, flush periods (1 .. 256), packed lengths
    (zeros included), grouped heads, read modes, scale and present / absent h0
    and dht, each against the oracle's autograd."""
    w, lengths, rm, flush, scale, h0, dht = _random_case(seed)
    _check(w, lengths=lengths, rm=rm, flush=flush, scale=scale, h0=h0, with_dht=dht,
           seed=300 + seed)
