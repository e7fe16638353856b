"""GPU checks with zero tolerance, from exact invariances of the method.

Every path is linear in (v, h0) and its QDQ absorbs powers of two in the
scale and its reciprocal, so scaling v and h0 by 2^k must scale every output
by exactly 2^k in the kernels' own arithmetic; the backward is linear in its
incoming gradients; and packing sequences only moves their rows, so a packed
batch must give each sequence exactly what a call on it alone gives."""
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq, synth

from _parity import to_dev
from test_gpu_bwd import NAMES, _dO

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k", [-7, 3])
def test_paths_scale_exactly_with_values_and_state(k):
    """Every path is linear in (v, h0), its QDQ is equivariant under powers of
    two (the scale and its reciprocal absorb them exactly), and W does not
    involve v: scaling v and h0 by 2^k must scale every output by exactly 2^k,
    bit for bit, in the kernels' own arithmetic."""
    from gated_delta_rule_54_gb300 import (gdn_decode_qdq, gdn_two_precision_fwd,
                                           kda_recurrent_fwd_qdq)
    f = 2.0 ** k
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128, h0=True, seed=51)
    d = to_dev(synth.make_kda_inputs(w))
    q, kk, v, beta, g, gk, h0 = d["q"], d["k"], d["v"], d["beta"], d["g"], d["g_k"], d["h0"]
    v2 = (v.float() * f).to(torch.bfloat16)
    assert torch.equal(v2.float(), v.float() * f)
    runs = [
        lambda vv, hh: gdn_chunk_fwd_qdq(q, kk, vv, beta, g, hh, state_mode="e4m3", w_mode="e4m3")[:2],
        lambda vv, hh: gdn_chunk_fwd_qdq(q, kk, vv, beta, g, hh, state_mode="int8", w_mode="e4m3")[:2],
        lambda vv, hh: gdn_decode_qdq(q, kk, vv, beta, g, hh, state_mode="e4m3", readout="post"),
        lambda vv, hh: kda_recurrent_fwd_qdq(q, kk, vv, beta, gk, hh, state_mode="e4m3"),
        lambda vv, hh: gdn_two_precision_fwd(q, kk, vv, beta, g, hh, read_mode="e4m3", flush=16),
    ]
    for i, run in enumerate(runs):
        a = run(v, h0)
        b = run(v2, h0 * f)
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            assert torch.equal(y, x * f), (i, float((y - x * f).abs().max()))


@pytest.mark.parametrize("sm,wm,hv", [("e4m3", "e4m3", 2), ("int8", "e4m3", 4)])
def test_backward_scales_exactly_with_the_cotangents(sm, wm, hv):
    """The STE backward is linear in the incoming gradients (dO, dht) and reuses
    the forward's saved values: scaling both by 2^k scales every gradient by
    exactly 2^k, bit for bit (grouped heads included)."""
    from gated_delta_rule_54_gb300 import gdn_chunk_bwd_ste
    w = synth.small(B=2, T=150, Hk=2, Hv=hv, Dk=128, Dv=128, h0=True, seed=52)
    d = synth.make_inputs(w)
    do, dht = _dO(w, d)
    dd = to_dev(d)
    o, ht, ctx = gdn_chunk_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                   state_mode=sm, w_mode=wm, save_ctx=True)
    f = 2.0 ** -5
    do2 = (do.float() * f).to(torch.bfloat16)
    assert torch.equal(do2.float(), do.float() * f)
    args = (dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], ctx)
    a = gdn_chunk_bwd_ste(*args, do.cuda(), dht.cuda(), state_mode=sm, w_mode=wm)
    b = gdn_chunk_bwd_ste(*args, do2.cuda(), (dht * f).cuda(), state_mode=sm, w_mode=wm)
    torch.cuda.synchronize()
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(y, x * f), (name, float((y - x * f).abs().max()))


def test_packed_sequences_equal_separate_calls_bit_for_bit():
    """Packing changes only where a sequence's rows sit: a packed batch must give
    every sequence exactly the outputs, final state and gradients that a call on
    that sequence alone gives (rows past a chunk's end hold the next sequence's
    tokens in the packed call and nothing in the single one; both must be
    masked out)."""
    from gated_delta_rule_54_gb300 import gdn_chunk_bwd_ste
    lengths = [70, 130, 64, 1]
    w = synth.small(B=1, T=0, Hk=2, Hv=4, Dk=128, Dv=128, h0=True, seed=53)
    d = synth.make_inputs(w, lengths=lengths)
    dd = to_dev(d)
    gen = torch.Generator().manual_seed(54)
    do = torch.randn(d["v"].shape, generator=gen).to(torch.bfloat16).cuda()
    dht = (torch.randn(d["h0"].shape, generator=gen) * 0.01).cuda()
    o, ht, ctx = gdn_chunk_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                   cu_seqlens=dd["cu_seqlens"], save_ctx=True)
    grads = gdn_chunk_bwd_ste(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], ctx, do, dht,
                              cu_seqlens=dd["cu_seqlens"])
    torch.cuda.synchronize()
    start = 0
    for n, L in enumerate(lengths):
        sl = lambda x: x[:, start:start + L].contiguous()
        q, k, v, beta, g = (sl(dd[key]) for key in ("q", "k", "v", "beta", "g"))
        h0 = dd["h0"][n:n + 1].contiguous()
        o1, ht1, ctx1 = gdn_chunk_fwd_qdq(q, k, v, beta, g, h0, save_ctx=True)
        g1 = gdn_chunk_bwd_ste(q, k, v, beta, g, ctx1, sl(do), dht[n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(o1, o[:, start:start + L]), ("o", n)
        assert torch.equal(ht1, ht[n:n + 1]), ("ht", n)
        for name, a, b in zip(NAMES, g1, grads):
            ref = b[n:n + 1] if name == "dh0" else b[:, start:start + L]
            assert torch.equal(a, ref), (name, n, float((a - ref).abs().max()))
        start += L
