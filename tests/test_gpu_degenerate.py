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

from _parity import GRAD_L2, grad_rel_l2, to_dev
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
