"""GPU parity of the decode QAT step (gdn_decode_qdq, through the C ABI)
against the fp64 decode oracle, with the tolerances of the forward parity
tests: codes within one step and at most 0.1% of them flipped; o and the
carried state within 1e-2 relative, each element widened by its derived flip
allowance (a differing code's step times its tile scale, carried through the
token updates; tests/_parity.py).  Scales agree to 1e-4 relative (the tile
amax is computed from fp32 instead of fp64 state values)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq, gdn_decode_qdq, synth
from oracle.decode import decode
from oracle.recurrent_torch import recurrent_torch

from _parity import (assert_close, assert_codes, code_steps, decode_flip_allowance, log_allowance,
                     to_dev)

pytestmark = pytest.mark.gpu


def _inputs(B, T, Hk, Hv, Dk, Dv, seed, state=True):
    w = synth.small(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, h0=state, seed=seed)
    return synth.make_inputs(w)


def _check(d, sm, bv, readout, scale=1.0):
    dd = to_dev(d)
    o, S, codes, scales = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                         scale=scale, state_mode=sm, block_v=bv, readout=readout,
                                         record=True)
    torch.cuda.synchronize()
    s0 = d["h0"] if d["h0"] is not None else torch.zeros(S.shape)
    ro, rS, rc, rs = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], s0, scale=scale,
                            state_mode=sm, block_v=bv, readout=readout, record=True)
    T = d["T"]
    flip = None
    if sm != "none" and T > 0:
        c = codes.cpu().numpy()
        flip = code_steps(c, rc, sm) > 0
        # codes and scales of states that no earlier flip of their (row, head) reached
        reached = np.cumsum(flip.any(axis=(3, 4)), axis=1) > 0
        ok = ~np.concatenate([np.zeros_like(reached[:, :1]), reached[:, :-1]], 1)
        assert_codes(c[ok], rc[ok], sm, "decode state codes")
        assert np.allclose(scales.cpu().numpy()[ok], rs[ok], rtol=1e-4, atol=0)
    else:
        assert codes is None or codes.numel() == 0
    o_al, s_al = decode_flip_allowance(d, rc, rs, flip, rS, scale, bv, sm, readout)
    if o.numel():
        log_allowance("decode o", o_al, ro, unit_axes=(0, 2))
        assert_close(o.cpu().numpy(), ro, "decode o", allow=o_al)
    log_allowance("decode state", s_al, rS, unit_axes=(0, 1))
    assert_close(S.cpu().numpy(), rS, "decode state", allow=s_al)
    return o, S


@pytest.mark.parametrize("readout", ["pre", "post"])
@pytest.mark.parametrize("sm", ["e4m3", "int8", "none"])
def test_decode_modes_and_readouts(sm, readout):
    _check(_inputs(3, 5, 2, 4, 128, 128, seed=1), sm, 64, readout)


@pytest.mark.parametrize("bv", [16, 32, 64, 128])
def test_decode_state_scale_widths(bv):
    _check(_inputs(2, 4, 1, 2, 128, 128, seed=bv), "e4m3", bv, "post")
    _check(_inputs(2, 3, 2, 2, 64, 128, seed=bv + 1), "int8", bv, "pre")


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (64, 128), (128, 64)])
def test_decode_head_dims(Dk, Dv):
    _check(_inputs(2, 3, 1, 2, Dk, Dv, seed=Dk + Dv), "e4m3", 64, "pre")
    _check(_inputs(2, 3, 1, 2, Dk, Dv, seed=Dk + Dv + 1), "int8", 32, "post", scale=Dk ** -0.5)


def test_decode_zero_state_zero_tokens_and_in_place():
    d = _inputs(2, 3, 2, 2, 128, 128, seed=7, state=False)
    _check(d, "e4m3", 64, "pre")                       # state_in NULL -> zeros, scale 0 first
    dd = to_dev(_inputs(2, 0, 2, 2, 128, 128, seed=8))
    o, S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"])
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(S, dd["h0"])   # T == 0 copies the state
    dd = to_dev(_inputs(2, 4, 2, 2, 128, 128, seed=9))
    ref_o, ref_S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"])
    st = dd["h0"].clone()
    o, S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], st, state_out=st)
    torch.cuda.synchronize()
    assert S.data_ptr() == st.data_ptr()
    assert torch.equal(o, ref_o) and torch.equal(st, ref_S)


def test_decode_single_token_calls_equal_one_call():
    dd = to_dev(_inputs(4, 6, 2, 4, 128, 128, seed=10))
    o, S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                          state_mode="int8", readout="post")
    st = dd["h0"].clone()
    for t in range(6):
        sl = lambda x: x[:, t:t + 1].contiguous()
        ot, st = gdn_decode_qdq(sl(dd["q"]), sl(dd["k"]), sl(dd["v"]), sl(dd["beta"]),
                                sl(dd["g"]), st, state_mode="int8", readout="post")
        assert torch.equal(ot[:, 0], o[:, t])
    assert torch.equal(st, S)


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_decode_long_trajectory(sm):
    """257 tokens of decode from a nonzero state with grouped heads."""
    d = _inputs(2, 257, 1, 2, 128, 128, seed=11)
    dd = to_dev(d)
    o, S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                          state_mode=sm)
    ro, rS = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm)
    # one-step code flips accumulate over a long trajectory; each stays within
    # one quantization step of its element, so whole units are held to 2^-3
    for b in range(2):
        for h in range(2):
            a, r = o[b, :, h].cpu().numpy(), ro[b, :, h]
            assert np.abs(a - r).max() <= 2.0 ** -3 * np.abs(r).max()
            a, r = S[b, h].cpu().numpy(), rS[b, h]
            assert np.abs(a - r).max() <= 2.0 ** -3 * np.abs(r).max()
    assert_close(o.cpu().numpy()[:, :8], ro[:, :8], "first tokens")


@pytest.mark.parametrize("P", [64, 100])
def test_split_carry_prefill_into_decode(P):
    """Chunked prefill of P tokens on the GPU, its ht carried into GPU decode,
    against the single-pass torch recurrence that quantizes before t < P with
    t % 64 == 0 and before every t >= P."""
    d = _inputs(1, 130, 1, 2, 128, 128, seed=P)
    dd = to_dev(d)
    pre = {n: dd[n][:, :P].contiguous() for n in ("q", "k", "v", "beta", "g")}
    post = {n: dd[n][:, P:].contiguous() for n in ("q", "k", "v", "beta", "g")}
    o_p, ht, _ = gdn_chunk_fwd_qdq(pre["q"], pre["k"], pre["v"], pre["beta"], pre["g"], dd["h0"],
                                   state_mode="e4m3", w_mode="none")
    o_d, S = gdn_decode_qdq(post["q"], post["k"], post["v"], post["beta"], post["g"], ht,
                            state_mode="e4m3")
    torch.cuda.synchronize()
    x = [d[n].double() for n in ("q", "k", "v", "beta", "g")]
    ref_o, ref_h = recurrent_torch(*x, h0=d["h0"].double(), state_mode="e4m3",
                                   quantize_before=lambda t: t >= P or t % 64 == 0)
    o = torch.cat([o_p.cpu(), o_d.cpu()], 1).double()
    for h in range(2):
        r = ref_o[:, :, h].numpy()
        assert np.abs(o[:, :, h].numpy() - r).max() <= 2.0 ** -3 * np.abs(r).max()
        r = ref_h[:, h].numpy()
        assert np.abs(S[:, h].cpu().numpy() - r).max() <= 2.0 ** -3 * np.abs(r).max()
    assert_close(o[:, :P].numpy(), ref_o[:, :P].numpy(), "prefill part")


def test_full_decode_workload_sampled():
    """B=256, H=16, D=128, one token, in the benchmark's launch configuration;
    sampled rows against the oracle (rows are independent)."""
    w = synth.WORKLOADS["decode"]
    d = synth.make_inputs(w)
    dd = to_dev(d)
    o, S = gdn_decode_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                          state_mode=w.state_mode)
    torch.cuda.synchronize()
    for b in (0, 131, 255):
        sl = lambda x: x[b:b + 1]
        ro, rS = decode(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["beta"]), sl(d["g"]),
                        sl(d["h0"]), state_mode=w.state_mode)
        assert_close(o[b:b + 1].cpu().numpy(), ro, "decode o row %d" % b)
        assert_close(S[b:b + 1].cpu().numpy(), rS, "decode state row %d" % b)
