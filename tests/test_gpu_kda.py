"""GPU parity of the KDA recurrence (kda_recurrent_fwd_qdq, through the C ABI)
against the fp64 KDA oracle.

The kernel's fp32 recurrence is held to the forward's bounds (max |err| <=
1e-2 max|ref|, 99.9% of elements within 1e-2 relative), each element widened
by its derived flip allowance: with QDQ the kernel quantizes its own fp32
state, so a code whose oracle value lies within the kernels' error of a
rounding boundary may land one step away; that step, times its tile scale, is
carried through the recurrence (tests/_parity.py)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import kda_recurrent_fwd_qdq, synth
from oracle.kda import kda_recurrent

from _parity import assert_close, log_allowance, sequence_allowances, to_dev

pytestmark = pytest.mark.gpu


def _run(w, lengths=None, sm="e4m3", block_v=64, chunk=64, scale=1.0, h0=True):
    d = synth.make_kda_inputs(w, lengths=lengths)
    if not h0:
        d["h0"] = None
    dd = to_dev(d)
    o, ht = kda_recurrent_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g_k"], dd["h0"],
                                  cu_seqlens=dd["cu_seqlens"], scale=scale, state_mode=sm,
                                  block_v=block_v, chunk=chunk)
    torch.cuda.synchronize()
    rec = []
    ro, rh = kda_recurrent(d["q"], d["k"], d["v"], d["beta"], d["g_k"], d["h0"],
                           cu_seqlens=d["cu_seqlens"], scale=scale, state_mode=sm,
                           block_v=block_v, chunk=chunk, record=rec)
    al = sequence_allowances(d, rec, sm, block_v, scale, g_key="g_k")
    return d, o.cpu().numpy(), ht.cpu().numpy(), ro, rh, al


def _check(o, ht, ro, rh, al):
    o_al, ht_al = al
    if o.size:
        log_allowance("kda o", o_al, ro, unit_axes=(0, 2))
        assert_close(o, ro, "kda o", allow=o_al)
    log_allowance("kda ht", ht_al, rh, unit_axes=(0, 1))
    assert_close(ht, rh, "kda ht", allow=ht_al)


@pytest.mark.parametrize("sm", ["e4m3", "int8", "none"])
@pytest.mark.parametrize("block_v", [16, 32, 64])
def test_kda_modes_and_scale_widths(sm, block_v):
    w = synth.small(B=2, T=150, Hk=2, Hv=4, Dk=128, Dv=128, w_mode="none", h0=True, seed=block_v)
    _check(*_run(w, sm=sm, block_v=block_v)[1:])


@pytest.mark.parametrize("T", [1, 63, 64, 65, 257])
def test_kda_lengths(T):
    w = synth.small(B=2, T=T, Hk=1, Hv=2, Dk=64, Dv=64, w_mode="none", h0=True, seed=T)
    _check(*_run(w, sm="int8")[1:])


def test_kda_packed_grouped_no_h0_and_every_token_qdq():
    w = synth.small(B=1, T=0, Hk=2, Hv=4, Dk=128, Dv=64, w_mode="none", h0=True, seed=9)
    _check(*_run(w, lengths=[0, 5, 130, 64, 77], sm="e4m3", scale=0.125)[1:])
    w = synth.small(B=2, T=40, Hk=1, Hv=1, Dk=64, Dv=128, w_mode="none", seed=10)
    _check(*_run(w, sm="e4m3", chunk=1, h0=False)[1:])


def test_kda_channel_constant_decay_matches_gdn_forward():
    """With every channel decaying alike and no W QDQ, the KDA recurrence is the
    gated delta rule: the two CUDA paths agree (state QDQ off)."""
    from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq
    w = synth.small(B=2, T=200, Hk=2, Hv=2, Dk=128, Dv=128, w_mode="none", h0=True, seed=11)
    d = to_dev(synth.make_inputs(w))
    gk = d["g"][..., None].expand(*d["g"].shape, 128).contiguous()
    o1, h1 = kda_recurrent_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], gk, d["h0"],
                                   state_mode="none")
    o2, h2, _ = gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                  state_mode="none", w_mode="none")
    torch.cuda.synchronize()
    assert_close(o1.cpu().numpy(), o2.cpu().numpy(), "kda vs gdn o")
    assert_close(h1.cpu().numpy(), h2.cpu().numpy(), "kda vs gdn ht")


def test_kda_full_workload_sampled():
    """B=4, T=4096, H=16, D=128 in the benchmark's launch configuration; sampled
    (sequence, head) sub-problems against the oracle."""
    w = synth.WORKLOADS["kda"]
    d = synth.make_kda_inputs(w)
    dd = to_dev(d)
    o, ht = kda_recurrent_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g_k"], dd["h0"],
                                  state_mode=w.state_mode)
    torch.cuda.synchronize()
    o, ht = o.cpu().numpy(), ht.cpu().numpy()
    for n, h in [(0, 0), (3, 15)]:
        sl = lambda x: x[n:n + 1, :, h:h + 1]
        sub = dict(q=sl(d["q"]), k=sl(d["k"]), v=sl(d["v"]), beta=sl(d["beta"]), g_k=sl(d["g_k"]),
                   h0=d["h0"][n:n + 1, h:h + 1], cu_seqlens=None)
        rec = []
        ro, rh = kda_recurrent(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g_k"], sub["h0"],
                               state_mode=w.state_mode, record=rec)
        al = sequence_allowances(sub, rec, w.state_mode, 64, 1.0, g_key="g_k")
        _check(o[n:n + 1, :, h:h + 1], ht[n:n + 1, h:h + 1], ro, rh, al)
