"""GPU parity of the two-precision GDN forward (gdn_two_precision_fwd, through
the C ABI) against the fp64 oracle (oracle/two_precision.py).

The anchor ht is never quantized: it is held to the forward's bounds
(max |err| <= 1e-2 max|ref|, 99.9% of elements within 1e-2 relative), and so
are the outputs, each element widened by its derived flip allowance: the
kernel quantizes its own fp32 anchor at each flush, so a read code whose oracle
value lies within the kernels' error of a rounding boundary may land one step
away; that step, times its column scale, is carried through the window's
tokens to the outputs until the next flush recomputes the read copy from the
anchor (tests/_parity.py)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_two_precision_fwd, synth
from oracle.two_precision import two_precision

from _parity import assert_close, log_allowance, sequence_allowances, to_dev

pytestmark = pytest.mark.gpu


def _run(w, lengths=None, rm="e4m3", flush=16, scale=1.0, h0=True):
    d = synth.make_inputs(w, lengths=lengths)
    if not h0:
        d["h0"] = None
    dd = to_dev(d)
    o, ht = gdn_two_precision_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                  cu_seqlens=dd["cu_seqlens"], scale=scale, read_mode=rm,
                                  flush=flush)
    torch.cuda.synchronize()
    rec = []
    ro, rh = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                           cu_seqlens=d["cu_seqlens"], scale=scale, read_mode=rm, flush=flush,
                           record=rec)
    al = sequence_allowances(d, rec, rm, 1, scale, carried=False)[0]
    return o.cpu().numpy(), ht.cpu().numpy(), ro, rh, al


def _check(o, ht, ro, rh, o_al):
    assert_close(ht, rh, "two-precision ht (anchor)")
    if o.size:
        log_allowance("two-precision o", o_al, ro, unit_axes=(0, 2))
        assert_close(o, ro, "two-precision o", allow=o_al)


@pytest.mark.parametrize("rm", ["e4m3", "none"])
@pytest.mark.parametrize("flush", [1, 16, 64])
def test_two_precision_modes_and_flush(rm, flush):
    w = synth.small(B=2, T=150, Hk=2, Hv=4, Dk=128, Dv=128, w_mode="none", h0=True, seed=flush)
    _check(*_run(w, rm=rm, flush=flush))


@pytest.mark.parametrize("T", [1, 3, 15, 16, 17, 257])
def test_two_precision_lengths(T):
    w = synth.small(B=2, T=T, Hk=1, Hv=2, Dk=128, Dv=64, w_mode="none", h0=True, seed=20 + T)
    _check(*_run(w))


def test_two_precision_packed_grouped_scaled_no_h0():
    w = synth.small(B=1, T=0, Hk=2, Hv=4, Dk=128, Dv=64, w_mode="none", h0=True, seed=30)
    _check(*_run(w, lengths=[0, 5, 130, 16, 77], scale=0.125, flush=5))
    w = synth.small(B=3, T=40, Hk=1, Hv=1, Dk=128, Dv=128, w_mode="none", seed=31)
    _check(*_run(w, h0=False, flush=7))


def test_two_precision_read_disabled_matches_the_chunked_forward():
    """With the read quantizer off the profile is the plain gated delta rule:
    the token-serial kernel and the chunked forward (no QDQ) agree."""
    from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq
    w = synth.small(B=2, T=200, Hk=2, Hv=4, Dk=128, Dv=128, w_mode="none", h0=True, seed=32)
    d = to_dev(synth.make_inputs(w))
    o1, h1 = gdn_two_precision_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   read_mode="none")
    o2, h2, _ = gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                  state_mode="none", w_mode="none")
    torch.cuda.synchronize()
    assert_close(o1.cpu().numpy(), o2.cpu().numpy(), "two-precision vs chunked o")
    assert_close(h1.cpu().numpy(), h2.cpu().numpy(), "two-precision vs chunked ht")


def test_two_precision_anchor_ignores_the_read_quantizer_on_the_gpu():
    w = synth.small(B=2, T=100, Hk=2, Hv=2, Dk=128, Dv=128, w_mode="none", h0=True, seed=33)
    d = to_dev(synth.make_inputs(w))
    args = [d[n] for n in ("q", "k", "v", "beta", "g", "h0")]
    _, h_q = gdn_two_precision_fwd(*args, read_mode="e4m3", flush=4)
    _, h_n = gdn_two_precision_fwd(*args, read_mode="none", flush=4)
    torch.cuda.synchronize()
    assert torch.equal(h_q, h_n)


def test_two_precision_full_size_one_sequence():
    """The benchmark's workload (B4 T4096 H16 D128, E4M3 reads, 16-token flush)
    in the benchmark's launch configuration; sequence 0 (all heads) against the
    oracle."""
    w = synth.WORKLOADS["two_precision"]
    d = synth.make_inputs(w)
    dd = to_dev(d)
    o, ht = gdn_two_precision_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                  read_mode="e4m3", flush=16)
    torch.cuda.synchronize()
    sub = {n: d[n][:1] for n in ("q", "k", "v", "beta", "g", "h0")}
    sub["cu_seqlens"] = None
    rec = []
    ro, rh = two_precision(*[sub[n] for n in ("q", "k", "v", "beta", "g", "h0")],
                           read_mode="e4m3", flush=16, record=rec)
    o_al = sequence_allowances(sub, rec, "e4m3", 1, 1.0, carried=False)[0]
    _check(o[:1].cpu().numpy(), ht[:1].cpu().numpy(), ro, rh, o_al)
    assert np.isfinite(o.cpu().numpy()).all() and np.isfinite(ht.cpu().numpy()).all()
