"""Thin Python binding of the C ABI (``include/gdn_qdq.h``): argument marshalling only.

PyTorch provides device memory and the current CUDA stream; every step of
the computation runs in the CUDA library.  There is no CPU or PyTorch
fallback: a missing library or a rejected configuration raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from ._lib import (DTYPES, QDQ_MODES, READOUTS, GdnDecodeProblem, GdnError, GdnProblem,  # noqa: F401
                   GdnTwoPrecisionProblem, check, load)

_DT = {torch.bfloat16: DTYPES["bf16"], torch.float16: DTYPES["fp16"], torch.float32: DTYPES["fp32"]}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _mode(m) -> int:
    if isinstance(m, str):
        if m not in QDQ_MODES:
            raise ValueError("QDQ mode must be one of %s, got %r" % (sorted(QDQ_MODES), m))
        return QDQ_MODES[m]
    return int(m)


def make_problem(q, k, v, cu_seqlens=None, scale=1.0, state_mode="e4m3", w_mode="e4m3",
                 block_v=64, chunk=64, N=None, neumann_degree=None, save_ctx=True) -> GdnProblem:
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    p = GdnProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv = B, T, Hk, Hv, Dk, Dv
    p.N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (B if N is None else N)
    p.cu_seqlens = cu_seqlens.data_ptr() if cu_seqlens is not None else None
    p.scale = float(scale)
    p.state_mode, p.w_mode = _mode(state_mode), _mode(w_mode)
    p.block_v, p.chunk = block_v, chunk
    p.dtype = _DT.get(q.dtype, 99)
    p.solve = 0 if neumann_degree is None else 1
    p.solve_degree = 0 if neumann_degree is None else int(neumann_degree)
    p.save_ctx = 1 if save_ctx else 0
    return p


def _check_dev(name, t, device):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError("%s must be a CUDA tensor on %s" % (name, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def gdn_validate(p: GdnProblem) -> int:
    return load().gdn_validate(ctypes.byref(p))


def gdn_ctx_bytes(p: GdnProblem) -> int:
    return int(load().gdn_ctx_bytes(ctypes.byref(p)))


def gdn_num_chunk_slots(p: GdnProblem) -> int:
    return int(load().gdn_num_chunk_slots(ctypes.byref(p)))


def gdn_bwd_workspace_bytes(p: GdnProblem) -> int:
    return int(load().gdn_bwd_workspace_bytes(ctypes.byref(p)))


def gdn_chunk_fwd_qdq(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, state_mode="e4m3",
                      w_mode="e4m3", output_final_state=True, save_ctx=False, out=None,
                      block_v=64, neumann_degree=None):
    """Forward.  q, k [B,T,Hk,Dk] bf16; v [B,T,Hv,Dv] bf16; beta, g [B,T,Hv] f32;
    h0 [N,Hv,Dk,Dv] f32 or None; cu_seqlens [N+1] int32 or None (B == 1).

    Returns (o [B,T,Hv,Dv] f32, ht [N,Hv,Dk,Dv] f32 or None, ctx uint8 or None).
    With ``save_ctx`` the forward writes the backward's context and returns
    it; without, it runs forward only with a smaller scratch context (not
    returned).  ``out`` may pass preallocated (o, ht, ctx) buffers (ctx of
    gdn_ctx_bytes for the same save_ctx; returned then).
    """
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("h0", h0),
                    ("cu_seqlens", cu_seqlens)):
        _check_dev(name, t, dev)
    p = make_problem(q, k, v, cu_seqlens, scale, state_mode, w_mode, block_v=block_v,
                     neumann_degree=neumann_degree, save_ctx=save_ctx)
    check("gdn_validate", lib.gdn_validate(ctypes.byref(p)))
    B, T, Hv, Dv = v.shape
    if out is not None:
        o, ht, ctx = out
    else:
        o = torch.empty(B, T, Hv, Dv, device=dev, dtype=torch.float32)
        ht = (torch.empty(p.N, Hv, k.shape[3], Dv, device=dev, dtype=torch.float32)
              if output_final_state else None)
        ctx = torch.empty(int(lib.gdn_ctx_bytes(ctypes.byref(p))), device=dev, dtype=torch.uint8)
    st = lib.gdn_chunk_fwd_qdq(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                               _ptr(h0), _ptr(o), _ptr(ht), _ptr(ctx), _stream(dev))
    check("gdn_chunk_fwd_qdq", st)
    return o, ht, (ctx if save_ctx or out is not None else None)


def gdn_chunk_bwd_ste(q, k, v, beta, g, ctx, do, dht=None, cu_seqlens=None, scale=1.0,
                      state_mode="e4m3", w_mode="e4m3", need_dh0=True, workspace=None, out=None,
                      block_v=64, neumann_degree=None):
    """Identity-STE backward.  Returns (dq, dk, dv, dbeta, dg, dh0 or None).

    ``out`` may pass preallocated (dq, dk, dv, dbeta, dg, dh0) buffers."""
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("ctx", ctx),
                    ("do", do), ("dht", dht), ("cu_seqlens", cu_seqlens)):
        _check_dev(name, t, dev)
    if do.dtype != torch.bfloat16:
        raise GdnError("gdn_chunk_bwd_ste", -2)
    p = make_problem(q, k, v, cu_seqlens, scale, state_mode, w_mode, block_v=block_v,
                     neumann_degree=neumann_degree)
    check("gdn_validate", lib.gdn_validate(ctypes.byref(p)))
    f32 = dict(device=dev, dtype=torch.float32)
    if out is not None:
        dq, dk, dv, dbeta, dg, dh0 = out
    else:
        dq = torch.empty(k.shape, **f32)
        dk = torch.empty(k.shape, **f32)
        dv = torch.empty(v.shape, **f32)
        dbeta = torch.empty(beta.shape, **f32)
        dg = torch.empty(g.shape, **f32)
        dh0 = torch.empty(p.N, v.shape[2], k.shape[3], v.shape[3], **f32) if need_dh0 else None
    need = int(lib.gdn_bwd_workspace_bytes(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    st = lib.gdn_chunk_bwd_ste(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                               _ptr(ctx), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(dbeta), _ptr(dg), _ptr(dh0), _ptr(workspace),
                               ctypes.c_size_t(workspace.numel()), _stream(dev))
    check("gdn_chunk_bwd_ste", st)
    return dq, dk, dv, dbeta, dg, dh0


def kda_recurrent_fwd_qdq(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0,
                          state_mode="e4m3", block_v=64, chunk=64, output_final_state=True):
    """KDA recurrence with per-key-channel decay g [B,T,Hv,Dk] f32 and the state QDQ every
    ``chunk`` tokens.  q, k [B,T,Hk,Dk] bf16; v [B,T,Hv,Dv] bf16; beta [B,T,Hv] f32;
    h0 [N,Hv,Dk,Dv] f32 or None.  Returns (o [B,T,Hv,Dv] f32, ht [N,Hv,Dk,Dv] f32 or None)."""
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("h0", h0),
                    ("cu_seqlens", cu_seqlens)):
        _check_dev(name, t, dev)
    p = make_problem(q, k, v, cu_seqlens, scale, state_mode, "none", block_v=block_v, chunk=chunk)
    B, T, Hv, Dv = v.shape
    o = torch.empty(B, T, Hv, Dv, device=dev, dtype=torch.float32)
    ht = (torch.empty(p.N, Hv, k.shape[3], Dv, device=dev, dtype=torch.float32)
          if output_final_state else None)
    st = lib.kda_recurrent_fwd_qdq(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                   _ptr(g), _ptr(h0), _ptr(o), _ptr(ht), _stream(dev))
    check("kda_recurrent_fwd_qdq", st)
    return o, ht


def make_two_precision_problem(q, k, v, cu_seqlens=None, scale=1.0, read_mode="e4m3",
                               flush=16) -> GdnTwoPrecisionProblem:
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    p = GdnTwoPrecisionProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv = B, T, Hk, Hv, Dk, Dv
    p.N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    p.cu_seqlens = _ptr(cu_seqlens)
    p.scale = float(scale)
    p.read_mode = _mode(read_mode)
    p.flush = int(flush)
    p.dtype = _DT.get(q.dtype, 99)
    return p


def gdn_two_precision_anchor_bytes(p: GdnTwoPrecisionProblem) -> int:
    return int(load().gdn_two_precision_anchor_bytes(ctypes.byref(p)))


def gdn_two_precision_fwd(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0,
                          read_mode="e4m3", flush=16, output_final_state=True, out=None,
                          save_anchors=False):
    """Two-precision GDN forward: fp32 recurrence anchor, E4M3 read copy (one scale per
    value row over the 128 key channels) re-derived from the anchor every ``flush`` tokens
    and read by the outputs only.  q, k [B,T,Hk,128] bf16; v [B,T,Hv,Dv] bf16; beta, g
    [B,T,Hv] f32; h0 [N,Hv,128,Dv] f32 or None.  Returns (o [B,T,Hv,Dv] f32,
    ht [N,Hv,128,Dv] f32 = the anchor, or None); ``out`` may pass preallocated (o, ht).
    With ``save_anchors`` a third value is returned: the anchor entering every window,
    which gdn_two_precision_bwd takes."""
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("h0", h0),
                    ("cu_seqlens", cu_seqlens)):
        _check_dev(name, t, dev)
    p = make_two_precision_problem(q, k, v, cu_seqlens, scale, read_mode, flush)
    check("gdn_two_precision_validate", lib.gdn_two_precision_validate(ctypes.byref(p)))
    B, T, Hv, Dv = v.shape
    if out is not None:
        o, ht = out
    else:
        o = torch.empty(B, T, Hv, Dv, device=dev, dtype=torch.float32)
        ht = (torch.empty(p.N, Hv, k.shape[3], Dv, device=dev, dtype=torch.float32)
              if output_final_state else None)
    anchors = None
    if save_anchors:
        nb = int(lib.gdn_two_precision_anchor_bytes(ctypes.byref(p)))
        anchors = torch.empty(max(nb // 4, 4), device=dev, dtype=torch.float32)
    st = lib.gdn_two_precision_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                   _ptr(g), _ptr(h0), _ptr(o), _ptr(ht), _ptr(anchors),
                                   _stream(dev))
    check("gdn_two_precision_fwd", st)
    return (o, ht, anchors) if save_anchors else (o, ht)


def gdn_two_precision_bwd(q, k, v, beta, g, anchors, do, dht=None, cu_seqlens=None, scale=1.0,
                          read_mode="e4m3", flush=16, need_dh0=True, workspace=None, out=None):
    """Window-wise adjoint of the two-precision forward (identity straight-through at the
    read copy).  ``anchors`` from gdn_two_precision_fwd(..., save_anchors=True) on the
    same inputs; do [B,T,Hv,Dv] f32; dht [N,Hv,128,Dv] f32 or None.  Returns
    (dq, dk, dv, dbeta, dg, dh0 or None); ``out`` may pass them preallocated."""
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g),
                    ("anchors", anchors), ("do", do), ("dht", dht), ("cu_seqlens", cu_seqlens)):
        _check_dev(name, t, dev)
    if do.dtype != torch.float32:
        raise GdnError("gdn_two_precision_bwd", -2)
    p = make_two_precision_problem(q, k, v, cu_seqlens, scale, read_mode, flush)
    check("gdn_two_precision_validate", lib.gdn_two_precision_validate(ctypes.byref(p)))
    f32 = dict(device=dev, dtype=torch.float32)
    if out is not None:
        dq, dk, dv, dbeta, dg, dh0 = out
    else:
        dq = torch.empty(k.shape, **f32)
        dk = torch.empty(k.shape, **f32)
        dv = torch.empty(v.shape, **f32)
        dbeta = torch.empty(beta.shape, **f32)
        dg = torch.empty(g.shape, **f32)
        dh0 = torch.empty(p.N, v.shape[2], k.shape[3], v.shape[3], **f32) if need_dh0 else None
    need = int(lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    st = lib.gdn_two_precision_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                   _ptr(g), _ptr(anchors), _ptr(do), _ptr(dht), _ptr(dq),
                                   _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(dh0),
                                   _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                   _stream(dev))
    check("gdn_two_precision_bwd", st)
    return dq, dk, dv, dbeta, dg, dh0


def make_decode_problem(q, k, v, scale=1.0, state_mode="e4m3", block_v=64,
                        readout="pre") -> GdnDecodeProblem:
    B, T, Hk, Dk = k.shape
    Hv, Dv = v.shape[2], v.shape[3]
    p = GdnDecodeProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv = B, T, Hk, Hv, Dk, Dv
    p.scale = float(scale)
    p.state_mode = _mode(state_mode)
    p.block_v = block_v
    if readout not in READOUTS:
        raise ValueError("readout must be one of %s, got %r" % (sorted(READOUTS), readout))
    p.readout = READOUTS[readout]
    p.dtype = _DT.get(q.dtype, 99)
    return p


def gdn_decode_qdq(q, k, v, beta, g, state_in=None, scale=1.0, state_mode="e4m3", block_v=64,
                   readout="pre", record=False, state_out=None, out=None):
    """Decode QAT step over T tokens per row.  q, k [B,T,Hk,Dk] bf16; v [B,T,Hv,Dv] bf16;
    beta, g [B,T,Hv] f32; state_in [B,Hv,Dk,Dv] f32 or None (zeros).

    Returns (o [B,T,Hv,Dv] f32, state_out [B,Hv,Dk,Dv] f32) and, with ``record``,
    (codes u8 [B,T,Hv,Dk,Dv], scales f32 [B,T,Hv,Dv/block_v]) of the quantized
    state each token read.  ``state_out`` may be ``state_in`` (in-place update);
    ``out`` may pass a preallocated o.
    """
    lib = load()
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g),
                    ("state_in", state_in), ("state_out", state_out)):
        _check_dev(name, t, dev)
    p = make_decode_problem(q, k, v, scale, state_mode, block_v, readout)
    check("gdn_decode_validate", lib.gdn_decode_validate(ctypes.byref(p)))
    B, T, Hv, Dv = v.shape
    Dk = k.shape[3]
    o = torch.empty(B, T, Hv, Dv, device=dev, dtype=torch.float32) if out is None else out
    if state_out is None:
        state_out = torch.empty(B, Hv, Dk, Dv, device=dev, dtype=torch.float32)
    codes = scales = None
    if record and p.state_mode != 0:
        codes = torch.empty(B, T, Hv, Dk, Dv, device=dev, dtype=torch.uint8)
        scales = torch.empty(B, T, Hv, Dv // block_v, device=dev, dtype=torch.float32)
    st = lib.gdn_decode_qdq(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                            _ptr(state_in), _ptr(o), _ptr(state_out), _ptr(codes), _ptr(scales),
                            _stream(dev))
    check("gdn_decode_qdq", st)
    if record:
        return o, state_out, codes, scales
    return o, state_out


def _fake_qdq(fn_name, x, group_cols, with_codes=False, out=None):
    lib = load()
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    if x.dim() == 1:
        b, r, c = 1, 1, x.shape[0]
    elif x.dim() == 2:
        b, r, c = 1, x.shape[0], x.shape[1]
    else:
        b, r, c = x[..., 0, 0].numel(), x.shape[-2], x.shape[-1]
    y = torch.empty_like(x) if out is None else out
    scales = torch.empty(b, c // group_cols if group_cols > 0 else 0, device=x.device,
                         dtype=torch.float32)
    codes = torch.empty(x.shape, device=x.device, dtype=torch.uint8) if with_codes else None
    st = getattr(lib, fn_name)(_ptr(x), _ptr(y), _ptr(scales), _ptr(codes), b, r, c, group_cols,
                               _stream(x.device))
    check(fn_name, st)
    return (y, scales, codes) if with_codes else (y, scales)


def fake_qdq_e4m3(x, group_cols, with_codes=False, out=None):
    """Grouped dynamic E4M3 fake QDQ of a [batch, rows, cols] float32 CUDA tensor."""
    return _fake_qdq("fake_qdq_e4m3", x, group_cols, with_codes, out)


def fake_qdq_int8(x, group_cols, with_codes=False, out=None):
    """Grouped dynamic INT8 fake QDQ of a [batch, rows, cols] float32 CUDA tensor."""
    return _fake_qdq("fake_qdq_int8", x, group_cols, with_codes, out)


def split_ctx(ctx: torch.Tensor, p: GdnProblem):
    """Views of the forward's context segments present for problem p (offsets
    from gdn_ctx_offset)."""
    lib = load()
    B, T, Hv, Dk, Dv = p.B, p.T, p.Hv, p.Dk, p.Dv
    ns = gdn_num_chunk_slots(p)
    f32, bf16 = torch.float32, torch.bfloat16
    segs = [  # name, segment id, dtype, shape
        ("w_codes", 0, torch.uint8, (B, T, Hv, Dk)),
        ("w_scales", 1, f32, (ns, Hv)),
        ("w_full", 2, f32, (B, T, Hv, Dk)),
        ("chunk_vectors", 3, f32, (ns, Hv, 5, 64)),
        ("t_img", 4, bf16, (ns, Hv, 64 * 64)),      # bf16 64x64 tiles as swizzled images
        ("gkk_img", 5, bf16, (ns, Hv, 64 * 64)),
        ("p_img", 6, bf16, (ns, Hv, 64 * 64)),
        ("d_img", 7, bf16, (ns, Hv, Dv // 64, 64 * 64)),   # Delta of each value block
        ("tu_img", 8, bf16, (ns, Hv, 2, 64 * 64)),
        ("h_codes", 9, torch.uint8, (ns, Hv, Dk, Dv)),
        ("h_scales", 10, f32, (ns, Hv, Dv // p.block_v)),
        ("h_full", 11, f32, (ns, Hv, Dk, Dv)),
    ]
    out = {}
    for name, sid, dt, shape in segs:
        off = int(lib.gdn_ctx_offset(ctypes.byref(p), sid))
        if off < 0:
            continue
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dt).element_size()
        out[name] = ctx[off:off + nbytes].view(dt).view(*shape)
    return out
