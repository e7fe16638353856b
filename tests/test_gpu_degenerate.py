"""GPU parity of the forward and the STE backward on the method's degenerate
inputs, against the fp64 oracle: write strength beta = 0 (W = 0, so the W
quantizer takes its zero-amax path, A = 0 and T = I), no decay (g = 0), zero
queries (o = 0 exactly), zero keys (no writes reach the state: pure decay),
and zero values with a zero initial state (every state tile has amax 0).

With beta = 0 or k = 0 the state only decays: at the workload's decay rates it
leaves binary32's range within three chunks, so the state quantizer meets
tiles whose amax is so small that the scale's reciprocal overflows.  Both
sides then take the group as scaled to zero (signed-zero codes, scale 0), and
everything stays finite."""
import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq, synth

from _parity import GRAD_L2, assert_close, grad_rel_l2, sequence_allowances, to_dev
from test_gpu_bwd import NAMES, _dO, _grads_gpu, _grads_oracle
from test_gpu_fwd import _check_case

pytestmark = pytest.mark.gpu

KINDS = ["beta0", "g0", "q0", "k0", "zero_v_h0"]
NORMAL_MIN = 2.0 ** -126    # smallest normal binary32


def _inputs(kind, seed):
    w = synth.small(B=2, T=150, Hk=2, Hv=2, Dk=64, Dv=64, h0=kind != "zero_v_h0", seed=seed)
    d = synth.make_inputs(w)
    if kind == "beta0":
        d["beta"].zero_()
    elif kind == "g0":
        d["g"].zero_()
    elif kind == "q0":
        d["q"].zero_()
    elif kind == "k0":
        d["k"].zero_()
    elif kind == "zero_v_h0":
        d["v"].zero_()
    return w, d


@pytest.mark.parametrize("kind", KINDS)
def test_forward_degenerate(kind):
    w, d = _inputs(kind, seed=90 + KINDS.index(kind))
    o, ht = _check_case(w, d=d)
    o = o.cpu().numpy()
    assert np.isfinite(o).all()
    if kind in ("q0", "zero_v_h0"):
        assert not o.any()                   # no query or nothing stored: o is exactly zero


def test_forward_zero_values_and_state_outputs_exact_zero():
    w, d = _inputs("zero_v_h0", seed=94)
    dd = to_dev(d)
    o, ht, _ = gdn_chunk_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                 state_mode="e4m3", w_mode="e4m3")
    torch.cuda.synchronize()
    assert not o.cpu().numpy().any() and not ht.cpu().numpy().any()


@pytest.mark.parametrize("kind", KINDS)
def test_backward_degenerate(kind):
    w, d = _inputs(kind, seed=95 + KINDS.index(kind))
    do, dht = _dO(w, d)
    g = _grads_gpu(d, "e4m3", "e4m3", do, dht)
    r = _grads_oracle(d, "e4m3", "e4m3", do, dht)
    for name, a, b in zip(NAMES, g, r):
        assert np.isfinite(a).all(), (kind, name)
        if np.linalg.norm(b) < NORMAL_MIN:
            # the exact gradient lies below binary32's normal range (e.g. dh0
            # with q = 0: only dht reaches h0, through 150 tokens of decay);
            # an fp32 kernel can only hold it to an absolute error of that size
            assert np.linalg.norm(a - b) <= NORMAL_MIN, (kind, name)
        else:
            assert grad_rel_l2(a, b) <= GRAD_L2, (kind, name, grad_rel_l2(a, b))


# ---- the token-serial paths through the same threshold: beta = 0 and a
#      constant decay of e^-1.5 per token, so the state's tile amax crosses
#      the point where the scale's reciprocal overflows within 64 tokens ----

def _pure_decay(d, g_key):
    d["beta"].zero_()
    d[g_key].fill_(-1.5)
    return d


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_decode_pure_decay_through_the_scale_threshold(sm):
    from oracle.decode import decode
    from test_gpu_decode import _check as decode_check, _inputs as decode_inputs
    d = _pure_decay(decode_inputs(2, 96, 1, 2, 128, 128, seed=31), "g")
    rs = decode(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                block_v=64, readout="post", record=True)[3]
    assert (rs[:, 0] > 0).all() and (rs[:, -1] == 0).all()   # the threshold is crossed
    o, S = decode_check(d, sm, 64, "post")
    assert np.isfinite(o.cpu().numpy()).all()
    assert not S.cpu().numpy().any()          # the quantized state became exactly zero


@pytest.mark.parametrize("sm", ["e4m3", "int8"])
def test_kda_pure_decay_through_the_scale_threshold(sm):
    from gated_delta_rule_54_gb300 import kda_recurrent_fwd_qdq
    from oracle.kda import kda_recurrent
    from test_gpu_kda import _check as kda_check
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128, w_mode="none", h0=True, seed=32)
    d = _pure_decay(synth.make_kda_inputs(w), "g_k")
    dd = to_dev(d)
    o, ht = kda_recurrent_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g_k"], dd["h0"],
                                  state_mode=sm)
    torch.cuda.synchronize()
    rec = []
    ro, rh = kda_recurrent(d["q"], d["k"], d["v"], d["beta"], d["g_k"], d["h0"], state_mode=sm,
                           record=rec)
    o, ht = o.cpu().numpy(), ht.cpu().numpy()
    assert np.isfinite(o).all() and not ht.any() and not np.asarray(rh).any()
    kda_check(o, ht, ro, rh, sequence_allowances(d, rec, sm, 64, 1.0, g_key="g_k"))


def test_two_precision_pure_decay_through_the_scale_threshold():
    from gated_delta_rule_54_gb300 import gdn_two_precision_fwd
    from oracle.two_precision import two_precision
    w = synth.small(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128, w_mode="none", h0=True, seed=33)
    d = _pure_decay(synth.make_inputs(w), "g")
    dd = to_dev(d)
    o, ht = gdn_two_precision_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                  read_mode="e4m3", flush=16)
    torch.cuda.synchronize()
    ro, rh = two_precision(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], read_mode="e4m3",
                           flush=16)
    o, ht = o.cpu().numpy(), ht.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    # The anchor is never quantized: it decays below binary32's range, where the
    # fp32 kernel can only hold the oracle's value rounded to binary32.
    assert_close(ht, np.asarray(rh).astype(np.float32), "anchor ht")
    # Reads after the read copy's amax passed the threshold are exactly zero.
    late = o[:, 64:]
    assert not late.any() and not np.asarray(ro)[:, 64:].any()
    assert_close(o, ro, "two-precision o")
