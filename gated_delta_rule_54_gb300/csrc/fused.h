// Fused state scan + outputs of the chunked forward (host interface).
//
// For Dk = Dv = 128 with both QDQ sites on, block_v 64 and the exact solve,
// the forward runs as two launches: the chunk-local prep (A, T, W and its QDQ,
// the chunk vectors; T diag(beta) as hi + lo bf16 tiles) and one fused kernel
// per (sequence, value
// head, 64-column value block) that walks the chunks and, per chunk, forms
// U = T diag(beta) V, quantizes the state, forms Delta = U - W^ H^, the state
// update and the outputs, all on the tensor cores with accumulators in tensor
// memory.  Nothing but o (and, when the backward's context is saved, the codes
// and tile images) leaves the kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_qdq.h"

namespace gdn {

struct FusedParams {
  // 2-D TMA maps: k, q [tokens, Hk*128] bf16, v [tokens, Hv*128] bf16 (64 x 64
  // boxes, 128-byte swizzle); W codes [tokens, Hv*128] u8 (64 rows x 128 bytes)
  CUtensorMap tm_k, tm_q, tm_v, tm_wc;
  const void* tu_img;     // [n_slots, Hv, 2, 4096] bf16 T diag(beta) hi, lo tile images
  const float* cvec;      // [n_slots, Hv, 5 * 64] chunk vectors
  const float* w_scales;  // [n_slots, Hv]
  const float* h0;        // [N, Hv, 128, 128] or null
  float* o;               // [tokens, Hv, 128]
  float* ht;              // [N, Hv, 128, 128] or null
  uint8_t* h_codes;       // [n_slots, Hv, 128, 128] state codes, or null (not saved)
  float* h_scales;        // [n_slots, Hv, 2] or null
  void* pb;               // bf16 P images [n_slots, Hv, 4096], or null
  void* db;               // bf16 Delta images [n_slots, Hv, 2, 4096], or null
  const int32_t* cu_seqlens;
  int64_t T, nt_fixed;
  int Hv, G, N;
  float scale;
};

// grid (2, Hv, N); false: unsupported mode pair or launch failure
// after_prep: the chunk prep was launched just before on st (the scan then
// starts as its programmatic dependent; otherwise as an ordinary launch)
gdn_status launch_fused_scan(const FusedParams& p, int state_mode, int w_mode, cudaStream_t st,
                             bool after_prep);

// nonzero if a fused-scan kernel's bounded wait gave up (cleared when reset)
int fused_device_error(bool reset);

}  // namespace gdn
