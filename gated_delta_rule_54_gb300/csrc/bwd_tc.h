// Chunk-parallel gradients of the identity-STE backward on the Blackwell
// tensor cores (host interface).
//
// For Dk = Dv = 128 with both QDQ sites on and the exact solve, one CTA per
// (chunk slot, value head) forms every gradient of the chunk with tcgen05
// products (fp32 accumulators in tensor memory, bf16 operands in shared
// memory), recomputing P, Gamma o KK^T and Delta from Q, K, V, the saved T
// diag(beta) images and the W / state codes instead of reading them back.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_qdq.h"

namespace gdn {

struct BwdTcParams {
  // 2-D TMA maps: q, k [tokens, Hk*128] bf16; v, dO [tokens, Hv*128] bf16 (64 x 64
  // boxes, 128-byte swizzle); W codes [tokens, Hv*128] u8 (64 rows x 128 bytes)
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_wc;
  const uint8_t* h_codes;  // [n_slots, Hv, 128, 128] state codes entering each chunk
  const float* h_scales;   // [n_slots, Hv, 128 / block_v]
  const float* w_scales;   // [n_slots, Hv]
  const float* cvec;       // [n_slots, Hv, 5 * 64] chunk vectors
  const void* tb;          // [n_slots, Hv] 8 KiB T images
  const void* tu_img;      // [n_slots, Hv] 16 KiB T diag(beta) hi, lo images
  const void* ws_dh;       // [n_slots, Hv] 32 KiB state-gradient panels (the reverse scan's)
  float* dq;               // [tokens, HH, 128]: dq itself, or per value head (grouped heads)
  float* dk;
  float* dv;               // [tokens, Hv, 128]
  float* dbeta;            // [tokens, Hv]
  float* dg;
  const int32_t* cu_seqlens;
  int64_t T, nt_fixed;
  int64_t n_slots;         // chunk slots (set by the launcher)
  int Hv, G, N, HH;        // HH: heads of the dq / dk arrays (Hk, or Hv when grouped)
  int bv_log2;             // log2(block_v)
  float scale;
};

// Reverse scan of the state gradient on the tensor cores (Dk = Dv = 128, W
// site quantized): one CTA per (sequence, value head) carries dH (fp32) through
// the chunks in reverse and stores the dH' entering every chunk in the
// workspace, as the swizzled [128][64] tile image of each value block.
struct BwdScanTcParams {
  CUtensorMap tm_q, tm_k, tm_do, tm_wc;  // as in BwdTcParams
  const void* pb;          // [n_slots, Hv] 8 KiB P images (the forward's)
  const float* w_scales;   // [n_slots, Hv]
  const float* cvec;       // [n_slots, Hv, 5 * 64]
  const float* dht;        // [N, Hv, 128, 128] or null (zero)
  float* dh0;              // [N, Hv, 128, 128] or null
  void* ws_dh;             // [n_slots, Hv] 32 KiB state-gradient panels
  const int32_t* cu_seqlens;
  int64_t T, nt_fixed;
  int Hv, G, N;
  float scale;
};

// grid (Hv, N); false on an unsupported W mode or a launch failure
gdn_status launch_bwd_scan_tc(const BwdScanTcParams& p, int w_mode, cudaStream_t st);
int bwd_scan_tc_device_error(bool reset);

// persistent: one CTA per SM walks the (chunk slot, value head) tiles; false on
// an unsupported mode pair or a launch failure
gdn_status launch_bwd_chunk_tc(const BwdTcParams& p, int state_mode, int w_mode, int64_t n_slots,
                               cudaStream_t st);

// nonzero if the kernel's bounded wait gave up (cleared when reset)
int bwd_tc_device_error(bool reset);

}  // namespace gdn
