// Internal launchers behind the C ABI (host side; arguments already validated).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_qdq.h"

namespace gdn {

constexpr int kChunkLen = 64;  // chunk length and state-scale tile width
// per (chunk, value head) vectors the forward's chunk prep saves in the
// context: gamma, e^gamma, e^{gamma_L - gamma}, beta, beta e^gamma (64 each)
constexpr int kCvecFloats = 5 * 64;
// bf16 [64][64] chunk tiles the forward saves for the backward, each stored as
// the 8 KiB shared-memory image (64-column swizzled rows): T = (I + A)^-1,
// Gamma o KK^T (strictly lower), P = Gamma o QK^T (lower incl. diagonal)
constexpr int kTileImgBytes = 64 * 64 * 2;

// Derived sizes of a validated problem.
struct Dims {
  int64_t B, T, N, n_slots, nt_fixed;  // nt_fixed = ceil(T/64) for fixed-length rows
  int Hk, Hv, Dk, Dv;
  bool packed;
};

// Byte offsets of the context segments (see gdn_ctx_bytes); -1 where absent.
struct CtxLayout {
  int64_t w_codes = -1, w_scales = -1, w_full = -1, cvec = -1, tb = -1, gkk = -1, pb = -1,
          db = -1, tu_img = -1, h_codes = -1, h_scales = -1, h_full = -1;
  size_t total = 0;
};

Dims dims_of(const gdn_problem& p);
CtxLayout ctx_layout(const gdn_problem& p);
// the fused two-launch forward applies (Dk = Dv = 128, both sites quantized,
// block_v 64, exact solve)
bool fused_fwd(const gdn_problem& p);

gdn_status launch_fake_qdq(int mode, const float* x, float* y, float* scales, uint8_t* codes,
                           int64_t batch, int64_t rows, int64_t cols, int64_t group_cols,
                           cudaStream_t st);

gdn_status launch_fwd(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const float* h0,
                      float* o, float* ht, void* ctx, cudaStream_t st);

// nonzero if a forward (backward) kernel's bounded wait for a TMA transfer
// gave up (cleared when reset); -1 if the flag could not be read
int fwd_device_error(bool reset);
int bwd_device_error(bool reset);

// 2-D row-major TMA map: `cols` elements per row (contiguous), `rows` rows of
// `row_bytes` bytes; boxes of box_cols x box_rows elements; false on failure
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols,
              uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle sw);

gdn_status launch_kda(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const float* h0,
                      float* o, float* ht, cudaStream_t st);

size_t bwd_workspace_bytes(const gdn_problem& p, const Dims& d);

gdn_status launch_bwd(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const void* ctx,
                      const void* dO, const float* dht, float* dq, float* dk, float* dv,
                      float* dbeta, float* dg, float* dh0, void* ws, cudaStream_t st);

}  // namespace gdn
