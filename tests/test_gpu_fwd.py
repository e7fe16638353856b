"""GPU parity of the forward (gdn_chunk_fwd_qdq, through the C ABI) against the fp64 oracle.

Small cases span several chunks and ragged tails and are compared element by
element; the full-size workloads run in the benchmark's launch configuration
and are compared on sampled (sequence, key-head group) sub-problems that the
oracle computes independently.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_54_gb300 import gdn_chunk_fwd_qdq, make_problem, split_ctx, synth

from _parity import (assert_close, assert_codes, code_steps, fwd_flip_allowance, log_allowance,
                     run_oracle, slot_map, to_dev)
from oracle.chunked import chunked

pytestmark = pytest.mark.gpu


def _gpu_fwd(d, sm, wm, scale=1.0, save_ctx=True, block_v=64, neumann_degree=None):
    dd = to_dev(d)
    o, ht, ctx = gdn_chunk_fwd_qdq(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"],
                                   cu_seqlens=dd["cu_seqlens"], scale=scale, state_mode=sm,
                                   w_mode=wm, save_ctx=save_ctx, block_v=block_v,
                                   neumann_degree=neumann_degree)
    torch.cuda.synchronize()
    return dd, o, ht, ctx


def _check_case(w, lengths=None, scale=1.0, block_v=64, neumann_degree=None, d=None):
    """Forward of workload w (or of the given inputs d, made for w) against the
    oracle: state / W codes and scales of every chunk, chunk vectors, and o and
    ht element by element, each element widened by its derived flip allowance
    (zero before a unit's first flipped code)."""
    if d is None:
        d = synth.make_inputs(w, lengths=lengths)
    sm, wm = w.state_mode, w.w_mode
    dd, o, ht, ctx = _gpu_fwd(d, sm, wm, scale, block_v=block_v, neumann_degree=neumann_degree)
    o_ref, ht_ref, rec, inters = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                         cu_seqlens=d.get("cu_seqlens"), scale=scale,
                                         state_mode=sm, w_mode=wm, record=True,
                                         intermediates=True, block_v=block_v,
                                         neumann_degree=neumann_degree)
    p = make_problem(dd["q"], dd["k"], dd["v"], dd["cu_seqlens"], scale, sm, wm, block_v=block_v,
                     neumann_degree=neumann_degree)
    seg = split_ctx(ctx, p)
    packed = lengths is not None
    lens = list(lengths) if packed else [w.T] * w.B
    smap = slot_map(lens, packed, d["T"])
    state_flip = w_flip = None
    if sm != "none":
        codes = seg["h_codes"].cpu().numpy()[smap]
        state_flip = code_steps(codes, rec["state_codes"], sm) > 0
        # A flip feeds the later states of its (sequence, head), their codes and
        # amax with them: those are no independent check (the allowance bounds
        # their effect); every other chunk's codes and scale are.
        chunk_seq = np.concatenate([[n] * (-(-L // 64)) for n, L in enumerate(lens)] or [[]])
        any_flip = state_flip.reshape(len(smap), w.Hv, -1).any(-1)
        indep = np.ones(any_flip.shape, bool)
        for ci, h in zip(*np.nonzero(any_flip)):
            indep[(chunk_seq == chunk_seq[ci]) & (np.arange(len(smap)) > ci), h] = False
        assert_codes(codes[indep], np.asarray(rec["state_codes"])[indep], sm, "state codes")
        sc = seg["h_scales"].cpu().numpy()[smap]
        assert np.allclose(sc[indep], np.asarray(rec["state_scales"])[indep], rtol=1e-2, atol=0)
    else:
        hf = seg["h_full"].cpu().numpy()[smap]
        assert hf.shape[0] == len(smap)
    if wm != "none":
        wc = seg["w_codes"].cpu().numpy().reshape(-1, w.Hv, w.Dk)
        wref = np.concatenate(rec["w_codes"], 0).reshape(-1, w.Hv, w.Dk)
        assert_codes(wc, wref, wm, "W codes")
        ws = seg["w_scales"].cpu().numpy()[smap]
        assert np.allclose(ws, rec["w_scales"], rtol=1e-3, atol=0)
        w_flip = code_steps(wc, wref, wm) > 0
    # chunk vectors: gamma, e^gamma, e^{gamma_L - gamma}, beta, beta e^gamma per (chunk, head)
    cv = seg["chunk_vectors"].cpu().numpy()[smap]
    g64 = d["g"].double().numpy().reshape(-1, w.Hv)
    b64 = d["beta"].double().numpy().reshape(-1, w.Hv)
    start = 0
    ci = 0
    for L in lens:
        for c0 in range(0, L, 64):
            Lc = min(64, L - c0)
            gam = np.zeros((64, w.Hv))
            gam[:Lc] = np.cumsum(g64[start + c0:start + c0 + Lc], 0)
            gam[Lc:] = gam[Lc - 1]
            bet = np.zeros((64, w.Hv))
            bet[:Lc] = b64[start + c0:start + c0 + Lc]
            ref = np.stack([gam, np.exp(gam), np.exp(gam[63] - gam), bet, bet * np.exp(gam)], 0)
            assert np.allclose(cv[ci].transpose(1, 2, 0), ref, rtol=2e-5, atol=1e-6), "chunk vectors"
            ci += 1
        start += L
    o_al, ht_al = fwd_flip_allowance(d, inters, rec, state_flip, w_flip, lens, packed, scale,
                                     block_v, sm, wm)
    o_ref, ht_ref = o_ref.numpy(), ht_ref.numpy()
    if o.numel():
        log_allowance("o", o_al, o_ref, unit_axes=(0, 2) if not packed else (2,))
        assert_close(o.cpu().numpy(), o_ref, "o", allow=o_al)
    log_allowance("ht", ht_al, ht_ref, unit_axes=(0, 1))
    assert_close(ht.cpu().numpy(), ht_ref, "ht", allow=ht_al)
    return o, torch.from_numpy(o_ref)


MODES = [("e4m3", "e4m3"), ("int8", "e4m3"), ("none", "none"), ("e4m3", "none"),
         ("none", "e4m3"), ("int8", "int8"), ("int8", "none"), ("e4m3", "int8"), ("none", "int8")]


@pytest.mark.parametrize("sm,wm", MODES)
def test_fwd_modes(sm, wm):
    w = synth.small(B=2, T=200, Hk=2, Hv=4, Dk=128, Dv=128, state_mode=sm, w_mode=wm, h0=True,
                    seed=3)
    _check_case(w)


@pytest.mark.parametrize("block_v", [16, 32, 128])
@pytest.mark.parametrize("sm,wm", [("e4m3", "e4m3"), ("int8", "e4m3"), ("int8", "int8")])
def test_fwd_state_scale_widths(sm, wm, block_v):
    """[Dk, block_v] state-scale tiles other than 64 ("[2/4] GDN/KDA decode QAT
    with INT8 recurrent state", "Testing": all state scale widths); 128 spans
    both value blocks."""
    w = synth.small(B=2, T=150, Hk=2, Hv=2, Dk=128, Dv=128, state_mode=sm, w_mode=wm, h0=True,
                    seed=block_v)
    _check_case(w, block_v=block_v)
    w = synth.small(B=1, T=0, Hk=1, Hv=2, Dk=64, Dv=128, state_mode=sm, w_mode=wm, h0=True,
                    seed=block_v + 1)
    _check_case(w, lengths=[70, 1, 129], block_v=block_v)


@pytest.mark.parametrize("degree", [0, 3, 7])
def test_fwd_neumann_solve(degree):
    """Neumann approximate inverse of an explicit degree ("[7/7] Experimental
    GDN/KDA approximate-inverse QAT")."""
    w = synth.small(B=2, T=150, Hk=2, Hv=2, Dk=128, Dv=128, h0=True, seed=60 + degree)
    _check_case(w, neumann_degree=degree)


def test_fwd_neumann_degree_63_is_the_exact_solve():
    w = synth.small(B=1, T=130, Hk=1, Hv=2, Dk=128, Dv=128, h0=True, seed=70)
    d = synth.make_inputs(w)
    _, o1, h1, _ = _gpu_fwd(d, "none", "none")
    _, o2, h2, _ = _gpu_fwd(d, "none", "none", neumann_degree=63)
    assert_close(o2.cpu().numpy(), o1.cpu().numpy(), "degree 63 o")
    assert_close(h2.cpu().numpy(), h1.cpu().numpy(), "degree 63 ht")


@pytest.mark.parametrize("T", [1, 3, 63, 64, 65, 127, 128, 257])
def test_fwd_lengths(T):
    w = synth.small(B=2, T=T, Hk=1, Hv=2, Dk=64, Dv=64, h0=(T % 2 == 1), seed=T)
    _check_case(w)


@pytest.mark.parametrize("Dk,Dv", [(64, 128), (128, 64), (64, 64)])
def test_fwd_head_dims(Dk, Dv):
    w = synth.small(B=1, T=190, Hk=2, Hv=2, Dk=Dk, Dv=Dv, h0=True, seed=Dk + Dv)
    _check_case(w)


def test_fwd_grouped_heads_int8_state():
    w = synth.small(B=2, T=150, Hk=2, Hv=8, Dk=128, Dv=128, state_mode="int8", h0=True, seed=9)
    _check_case(w)


def test_fwd_packed_ragged_with_empty_sequence():
    lengths = [0, 1, 64, 97, 130, 5, 200, 0, 63]
    w = synth.small(B=1, T=0, Hk=2, Hv=4, Dk=128, Dv=128, h0=True, seed=4)
    _check_case(w, lengths=lengths)


def test_fwd_scale_and_tiny_workload():
    _check_case(synth.WORKLOADS["tiny"])
    w = synth.small(B=1, T=130, Hk=1, Hv=1, Dk=128, Dv=128, h0=True, seed=5)
    _check_case(w, scale=128 ** -0.5)


def test_fwd_qdq_sensitivity_and_disabled_path():
    w = synth.small(B=1, T=256, Hk=2, Hv=2, Dk=128, Dv=128, h0=True, seed=6)
    d = synth.make_inputs(w)
    _, o_q, _, _ = _gpu_fwd(d, "e4m3", "e4m3")
    _, o_n, _, _ = _gpu_fwd(d, "none", "none")
    assert (o_q - o_n).abs().max().item() > 1e-3 * o_n.abs().max().item()
    o1, _ = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    assert_close(o_n.cpu().numpy(), o1, "disabled path vs token recurrence")


def test_fwd_without_optional_outputs_and_zero_tokens():
    w = synth.small(B=2, T=100, Hk=1, Hv=1, Dk=64, Dv=64, seed=7)
    d = to_dev(synth.make_inputs(w))
    o, ht, ctx = gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"],
                                   output_final_state=False, save_ctx=False)
    o2, _, _ = gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], save_ctx=True)
    assert ht is None and ctx is None
    assert torch.equal(o, o2)   # deterministic, and saving the context changes nothing
    # zero tokens: ht == h0, untouched by QDQ
    z = {k: (v[:, :0].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 and k not in ("h0",) else v)
         for k, v in d.items()}
    h0 = torch.randn(2, 1, 64, 64, device="cuda")
    o, ht, _ = gdn_chunk_fwd_qdq(z["q"], z["k"], z["v"], z["beta"], z["g"], h0)
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(ht, h0)


@pytest.mark.parametrize("sm,wm", [("e4m3", "e4m3"), ("int8", "e4m3"), ("int8", "int8"),
                                   ("e4m3", "int8")])
def test_fwd_forward_only_equals_training_forward(sm, wm):
    """Without the backward's context (save_ctx = 0: no T, Gamma o KK^T, P, Delta
    images and, on the fused path, no state codes; the fused kernel then runs as
    its own variant, with the work split differently between its warps) the
    forward computes exactly the same o and ht, in every mode pair."""
    for w, lens in ((synth.small(B=2, T=200, Hk=2, Hv=4, Dk=128, Dv=128, state_mode=sm, w_mode=wm,
                                 h0=True, seed=12), None),
                    (synth.small(B=1, T=0, Hk=1, Hv=2, Dk=128, Dv=128, state_mode=sm, w_mode=wm,
                                 h0=True, seed=13), [70, 0, 129, 64]),
                    (synth.small(B=1, T=150, Hk=1, Hv=2, Dk=64, Dv=128, state_mode=sm, w_mode=wm,
                                 h0=True, seed=14), None)):
        d = to_dev(synth.make_inputs(w, lengths=lens))
        args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
        o1, h1, ctx = gdn_chunk_fwd_qdq(*args, cu_seqlens=d["cu_seqlens"], state_mode=sm, w_mode=wm,
                                        save_ctx=True)
        o2, h2, none = gdn_chunk_fwd_qdq(*args, cu_seqlens=d["cu_seqlens"], state_mode=sm,
                                         w_mode=wm, save_ctx=False)
        torch.cuda.synchronize()
        assert none is None
        assert torch.equal(o1, o2) and torch.equal(h1, h2)


# ----------------------------------------------------------------------------
# Full-size workloads, in the benchmark's launch configuration, on samples.
# ----------------------------------------------------------------------------
def _sample_check(name, picks):
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w)
    dd, o, ht, ctx = _gpu_fwd(d, w.state_mode, w.w_mode, save_ctx=False)
    o = o.cpu()
    ht = ht.cpu()
    G = w.Hv // w.Hk
    cu = d["cu_seqlens"]
    for n, hk in picks:
        if cu is None:
            q, k = d["q"][n:n + 1], d["k"][n:n + 1]
            v, b, g = d["v"][n:n + 1], d["beta"][n:n + 1], d["g"][n:n + 1]
            o_gpu = o[n:n + 1]
        else:
            a, e = int(cu[n]), int(cu[n + 1])
            q, k = d["q"][:, a:e], d["k"][:, a:e]
            v, b, g = d["v"][:, a:e], d["beta"][:, a:e], d["g"][:, a:e]
            o_gpu = o[:, a:e]
        hv = slice(hk * G, (hk + 1) * G)
        h0 = d["h0"][n:n + 1, hv] if d["h0"] is not None else None
        o_ref, ht_ref = run_oracle(dict(q=q[:, :, hk:hk + 1], k=k[:, :, hk:hk + 1],
                                        v=v[:, :, hv], beta=b[:, :, hv], g=g[:, :, hv], h0=h0),
                                   w.state_mode, w.w_mode)
        assert_close(o_gpu[:, :, hv].numpy(), o_ref.numpy(), "%s o (n=%d, hk=%d)" % (name, n, hk))
        assert_close(ht[n:n + 1, hv].numpy(), ht_ref.numpy(), "%s ht (n=%d, hk=%d)" % (name, n, hk))


def test_full_single_layer_sampled():
    _sample_check("layer", [(0, 0), (3, 15), (2, 7)])


def test_full_grouped_int8_sampled():
    _sample_check("grouped_int8", [(0, 0), (1, 15)])


def test_full_packed_varlen_sampled():
    lens = synth.varlen_lengths(32768)
    picks = [(0, 0), (len(lens) - 1, 31), (int(np.argmax(lens)), 5), (int(np.argmin(lens)), 17)]
    _sample_check("varlen", picks)


def test_no_bounded_wait_gave_up():
    """No forward kernel of the runs above ended early on a TMA wait."""
    from gated_delta_rule_54_gb300 import _lib
    assert _lib.load().gdn_device_error(1) == 0


def _unswizzle(img):
    """[..., 4096] bf16 tile images -> [..., 64, 64]."""
    i = np.arange(64)[:, None]
    j = np.arange(64)[None, :]
    idx = i * 64 + 8 * ((j // 8) ^ (i % 8)) + j % 8
    return img[..., idx]


def test_fwd_saved_backward_tiles():
    """T, Gamma o KK^T, P and Delta saved for the backward, against the oracle's
    intermediates and their definitions (bf16 storage: 2^-8 relative)."""
    from oracle.chunked import chunked
    w = synth.small(B=1, T=150, Hk=1, Hv=2, Dk=64, Dv=64, h0=True, seed=31)
    d = synth.make_inputs(w)
    dd, o, ht, ctx = _gpu_fwd(d, "e4m3", "e4m3")
    p = make_problem(dd["q"], dd["k"], dd["v"], None, 1.0, "e4m3", "e4m3")
    seg = split_ctx(ctx, p)
    imgs = {k: _unswizzle(seg[k].float().cpu().numpy()) for k in ("t_img", "gkk_img", "p_img")}
    _, _, inter = chunked(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                          state_mode="e4m3", w_mode="e4m3", intermediates=True)
    q = d["q"].double().numpy()[0, :, 0]
    k = d["k"].double().numpy()[0, :, 0]
    for c, st in enumerate(inter[0]):
        L = st["T"].shape[-1]
        sl = slice(64 * c, 64 * c + L)
        for h in range(2):
            gam = st["gamma"][h].numpy()
            G = np.exp(gam[:, None] - gam[None, :])
            kk = np.tril(G * (k[sl] @ k[sl].T), -1)
            pp = np.tril(G * (q[sl] @ k[sl].T))
            T = st["T"][h].numpy()
            for name, ref in (("t_img", T), ("gkk_img", kk), ("p_img", pp)):
                x = imgs[name][c, h]
                assert np.abs(x[:L, :L] - ref).max() <= 2 ** -7 * np.abs(ref).max(), (name, c, h)
                if name != "t_img":
                    assert not x[L:].any(), (name, c, h)   # rows past the chunk end are zero
            assert np.array_equal(imgs["t_img"][c, h, L:, L:], np.eye(64 - L))
            # Delta = U - W^ H^ of the (single, Dv = 64) value block, rounded to bf16
            dimg = _unswizzle(seg["d_img"][:, :, 0].float().cpu().numpy())[c, h]
            dref = st["Delta"][h].numpy()
            assert np.abs(dimg[:L] - dref).max() <= 2 ** -7 * np.abs(dref).max(), ("d_img", c, h)
            assert not dimg[L:].any(), ("d_img", c, h)
