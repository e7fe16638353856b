"""GB300-native (sm_103a) chunked gated delta rule with state / W fake QDQ.

The compute lives in the CUDA library ``libgdn_qdq.so`` (C ABI in
``include/gdn_qdq.h``); this package is its thin binding:

  gdn_chunk_fwd_qdq   forward (chunk 64, exact solve, state + W QDQ)
  gdn_chunk_bwd_ste   identity straight-through backward
  gdn_chunk_qdq       the two as one PyTorch autograd op (forward + STE backward)
  gdn_decode_qdq      decode QAT token steps (state QDQ before every token)
  kda_recurrent_fwd_qdq  KDA (per-key-channel decay) recurrence with state QDQ
  gdn_two_precision_fwd  two-precision profile: fp32 anchor, E4M3 read copy for outputs
  gdn_two_precision_bwd  its window-wise adjoint (straight-through read copy)
  fake_qdq_e4m3 / fake_qdq_int8   the grouped QDQ primitive

``synth`` holds the seeded synthetic-input generators.
"""
from .api import (fake_qdq_e4m3, fake_qdq_int8, gdn_bwd_workspace_bytes, gdn_chunk_bwd_ste,  # noqa: F401
                  gdn_chunk_fwd_qdq, gdn_ctx_bytes, gdn_decode_qdq, gdn_num_chunk_slots,
                  gdn_two_precision_anchor_bytes, gdn_two_precision_bwd, gdn_two_precision_fwd,
                  gdn_validate, kda_recurrent_fwd_qdq, make_decode_problem,
                  make_problem, make_two_precision_problem, split_ctx)
from ._lib import GdnError, load  # noqa: F401
from .autograd import gdn_chunk_qdq  # noqa: F401
