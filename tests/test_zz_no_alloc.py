"""GPU: the allocation-free backward entry point (gdn_chunk_bwd_ste_noalloc).

It serves callers that cannot allocate device memory when they run the
backward (a runtime that reserved the device's memory for its own pool, or
code where an allocation would synchronize the device): they pass inputs and
outputs only, and the scratch comes from a fixed array inside the library.
Checked through the C ABI against the workspace-taking gdn_chunk_bwd_ste on
the same inputs.  Both run the same deterministic kernels, so the gradients
must be bit-identical.  The array keeps the previous call's contents, so the
calls alternate between two different problems (grouped heads, then an INT8
state at other head dims): whatever one call leaves in the array is wrong for
the next, and any stale byte that leaked through would show.  Collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_54_gb300 import api, gdn_chunk_bwd_ste, gdn_chunk_fwd_qdq, synth
from gated_delta_rule_54_gb300._lib import load


pytestmark = pytest.mark.gpu

GDN_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
GDN_ERR_WORKSPACE_TOO_SMALL = -5


def _case(w, seed):
    d = synth.make_inputs(w)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(d["B"], d["T"], w.Hv, w.Dv, generator=gen).to(torch.bfloat16).cuda()
    dht = (torch.randn(d["N"], w.Hv, w.Dk, w.Dv, generator=gen) * 0.01).cuda()
    _, _, ctx = gdn_chunk_fwd_qdq(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"], dev["h0"],
                                  state_mode=w.state_mode, w_mode=w.w_mode, save_ctx=True)
    return dev, do, dht, ctx


def _noalloc(w, dev, do, dht, ctx):
    lib = load()
    p = api.make_problem(dev["q"], dev["k"], dev["v"], None, 1.0, w.state_mode, w.w_mode)
    f32 = dict(device="cuda", dtype=torch.float32)
    outs = [torch.full(dev["q"].shape, float("nan"), **f32), torch.full(dev["k"].shape, float("nan"), **f32),
            torch.full(dev["v"].shape, float("nan"), **f32), torch.full(dev["beta"].shape, float("nan"), **f32),
            torch.full(dev["g"].shape, float("nan"), **f32),
            torch.full((dev["N"], w.Hv, w.Dk, w.Dv), float("nan"), **f32)]
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.gdn_chunk_bwd_ste_noalloc(
        ctypes.byref(p), P(dev["q"]), P(dev["k"]), P(dev["v"]), P(dev["beta"]), P(dev["g"]), P(ctx),
        P(do), P(dht), *[P(t) for t in outs], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, outs


CASES = [
    synth.small(B=2, T=200, Hk=2, Hv=4, Dk=128, Dv=128, h0=True, seed=41),   # grouped heads
    synth.small(B=1, T=300, Hk=2, Hv=2, Dk=64, Dv=64, state_mode="int8", h0=True, seed=42),
]


def test_noalloc_equals_workspace_backward_across_alternating_problems():
    runs = []
    for i, w in enumerate(CASES):
        dev, do, dht, ctx = _case(w, 7 + i)
        p = api.make_problem(dev["q"], dev["k"], dev["v"], None, 1.0, w.state_mode, w.w_mode)
        assert api.gdn_bwd_workspace_bytes(p) <= GDN_NOALLOC_SCRATCH_BYTES
        ref = gdn_chunk_bwd_ste(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"], ctx, do, dht,
                                state_mode=w.state_mode, w_mode=w.w_mode)
        torch.cuda.synchronize()
        runs.append((w, dev, do, dht, ctx, ref))
    # A, B, A, B: each noalloc call follows one that filled the array with another problem
    for call in range(4):
        w, dev, do, dht, ctx, ref = runs[call % 2]
        st, outs = _noalloc(w, dev, do, dht, ctx)
        assert st == 0, "call %d returned %d" % (call, st)
        for name, a, b in zip(("dq", "dk", "dv", "dbeta", "dg", "dh0"), outs, ref):
            assert torch.isfinite(a).all(), "%s call %d" % (name, call)
            assert torch.equal(a, b), "%s call %d differs from the workspace backward" % (name, call)


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    # 8192 tokens x 16 heads x 128 x 128 needs a 64 MiB state-gradient buffer
    w = synth.small(B=1, T=8192, Hk=16, Hv=16, Dk=128, Dv=128, seed=43)
    dev, do, dht, ctx = _case(w, 8)
    p = api.make_problem(dev["q"], dev["k"], dev["v"], None, 1.0, w.state_mode, w.w_mode)
    assert api.gdn_bwd_workspace_bytes(p) > GDN_NOALLOC_SCRATCH_BYTES
    st, outs = _noalloc(w, dev, do, dht, ctx)
    assert st == GDN_ERR_WORKSPACE_TOO_SMALL
    assert torch.isnan(outs[0]).all()   # nothing was launched
