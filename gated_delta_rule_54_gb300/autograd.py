"""PyTorch autograd entry to the chunked forward and its identity-STE backward.

``gdn_chunk_qdq(q, k, v, beta, g, h0, ...)`` returns (o, ht) like
``gdn_chunk_fwd_qdq`` and, when any input requires grad, records one node
whose backward calls ``gdn_chunk_bwd_ste`` on the context the forward saved
(the quantized W and chunk states: the straight-through rule of the "[1/4]
GDN state/W QAT foundation" page reuses them, with no second quantizer call).
Argument marshalling only: both directions run in the CUDA library.

The backward's incoming dO is cast to bf16 (the kernel's operand type) and the
gradients of the bf16 q, k, v come back in bf16, as autograd requires
gradients in their inputs' dtype; beta, g and h0 keep fp32 gradients.
"""
from __future__ import annotations

import torch

from .api import gdn_chunk_bwd_ste, gdn_chunk_fwd_qdq


class _GdnChunkQDQ(torch.autograd.Function):
    @staticmethod
    def forward(fctx, q, k, v, beta, g, h0, cu_seqlens, scale, state_mode, w_mode, block_v,
                neumann_degree):
        o, ht, saved = gdn_chunk_fwd_qdq(q, k, v, beta, g, h0, cu_seqlens=cu_seqlens, scale=scale,
                                         state_mode=state_mode, w_mode=w_mode,
                                         output_final_state=True, save_ctx=True, block_v=block_v,
                                         neumann_degree=neumann_degree)
        fctx.save_for_backward(q, k, v, beta, g, saved, cu_seqlens)
        fctx.has_h0 = h0 is not None
        fctx.cfg = (scale, state_mode, w_mode, block_v, neumann_degree)
        return o, ht

    @staticmethod
    def backward(fctx, do, dht):
        q, k, v, beta, g, saved, cu_seqlens = fctx.saved_tensors
        scale, state_mode, w_mode, block_v, neumann_degree = fctx.cfg
        if do is None:
            do = torch.zeros(v.shape, device=v.device, dtype=torch.bfloat16)
        dq, dk, dv, dbeta, dg, dh0 = gdn_chunk_bwd_ste(
            q, k, v, beta, g, saved, do.to(torch.bfloat16).contiguous(),
            None if dht is None else dht.float().contiguous(), cu_seqlens=cu_seqlens, scale=scale,
            state_mode=state_mode, w_mode=w_mode, need_dh0=fctx.has_h0, block_v=block_v,
            neumann_degree=neumann_degree)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dbeta, dg,
                dh0 if fctx.has_h0 else None, None, None, None, None, None, None)


def gdn_chunk_qdq(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, state_mode="e4m3",
                  w_mode="e4m3", block_v=64, neumann_degree=None):
    """Differentiable chunked gated delta rule with state / W fake QDQ.

    q, k [B,T,Hk,Dk] bf16; v [B,T,Hv,Dv] bf16; beta, g [B,T,Hv] f32 (contiguous
    CUDA tensors); h0 [N,Hv,Dk,Dv] f32 or None; cu_seqlens [N+1] int32 or None.
    Returns (o [B,T,Hv,Dv] f32, ht [N,Hv,Dk,Dv] f32)."""
    return _GdnChunkQDQ.apply(q, k, v, beta, g, h0, cu_seqlens, scale, state_mode, w_mode,
                              block_v, neumann_degree)
