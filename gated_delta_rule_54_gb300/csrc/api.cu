// C ABI entry points: host-side validation, size queries and dispatch.
// Everything here runs on the host; nothing is launched until a problem has
// passed validation (first QAT page, "What does this PR do?": unsupported
// formats and FP32 inputs are rejected before launch).
#include <cuda_runtime.h>

#include "../../include/gdn_qdq.h"
#include "fused.h"
#include "launch.h"

namespace gdn {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Dims dims_of(const gdn_problem& p) {
  Dims d;
  d.B = p.B;
  d.T = p.T;
  d.Hk = p.Hk;
  d.Hv = p.Hv;
  d.Dk = p.Dk;
  d.Dv = p.Dv;
  d.packed = p.cu_seqlens != nullptr;
  d.N = d.packed ? p.N : p.B;
  d.nt_fixed = (p.T + kChunkLen - 1) / kChunkLen;
  d.n_slots = d.packed ? (p.T / kChunkLen + p.N) : p.B * d.nt_fixed;
  return d;
}

bool fused_fwd(const gdn_problem& p) {
  return p.Dk == 128 && p.Dv == 128 && p.state_mode != GDN_QDQ_NONE &&
         p.w_mode != GDN_QDQ_NONE && p.block_v == 64 && p.solve == GDN_SOLVE_EXACT;
}

CtxLayout ctx_layout(const gdn_problem& p) {
  const Dims d = dims_of(p);
  CtxLayout L;
  size_t off = 0;
  const size_t tokens = (size_t)(d.B * d.T);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return (int64_t)at;
  };
  if (p.w_mode != GDN_QDQ_NONE) {
    L.w_codes = take(tokens * d.Hv * d.Dk);
    L.w_scales = take(sizeof(float) * (size_t)d.n_slots * d.Hv);
  } else {
    L.w_full = take(sizeof(float) * tokens * d.Hv * d.Dk);
  }
  L.cvec = take(sizeof(float) * (size_t)d.n_slots * d.Hv * kCvecFloats);
  // the fused forward's backward recomputes Gamma o KK^T and Delta on the
  // tensor cores; the others read them back
  const bool fused = fused_fwd(p);
  if (p.save_ctx) {
    L.tb = take((size_t)d.n_slots * d.Hv * kTileImgBytes);
    if (!fused) L.gkk = take((size_t)d.n_slots * d.Hv * kTileImgBytes);
    L.pb = take((size_t)d.n_slots * d.Hv * kTileImgBytes);
    if (!fused) L.db = take((size_t)d.n_slots * d.Hv * (d.Dv / 64) * kTileImgBytes);
  }
  if (fused) L.tu_img = take((size_t)d.n_slots * d.Hv * 2 * kTileImgBytes);
  const size_t per_slot = (size_t)d.n_slots * d.Hv * d.Dk * d.Dv;
  if (p.state_mode != GDN_QDQ_NONE) {
    if (p.save_ctx || !fused) {
      L.h_codes = take(per_slot);
      L.h_scales = take(sizeof(float) * (size_t)d.n_slots * d.Hv * (d.Dv / p.block_v));
    }
  } else {
    L.h_full = take(sizeof(float) * per_slot);
  }
  L.total = off;
  return L;
}

static bool valid_mode(int m) {
  return m == GDN_QDQ_NONE || m == GDN_QDQ_E4M3 || m == GDN_QDQ_INT8;
}

static gdn_status validate(const gdn_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Dk <= 0 || p->Dv <= 0)
    return GDN_ERR_INVALID_ARG;
  if (!valid_mode(p->state_mode) || !valid_mode(p->w_mode)) return GDN_ERR_INVALID_ARG;
  if (p->dtype != GDN_DTYPE_BF16) {
    if (p->dtype == GDN_DTYPE_FP16 || p->dtype == GDN_DTYPE_FP32) return GDN_ERR_UNSUPPORTED_DTYPE;
    return GDN_ERR_INVALID_ARG;
  }
  if (p->chunk != kChunkLen) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->block_v != 16 && p->block_v != 32 && p->block_v != 64 && p->block_v != 128)
    return GDN_ERR_UNSUPPORTED_MODE;
  if (p->solve != GDN_SOLVE_EXACT && p->solve != GDN_SOLVE_NEUMANN) return GDN_ERR_INVALID_ARG;
  if (p->solve == GDN_SOLVE_NEUMANN && (p->solve_degree < 0 || p->solve_degree > 63))
    return GDN_ERR_UNSUPPORTED_MODE;  // degree 63 is already the exact inverse
  if ((p->Dk != 64 && p->Dk != 128) || (p->Dv != 64 && p->Dv != 128))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->block_v > p->Dv) return GDN_ERR_UNSUPPORTED_MODE;
  if (p->Hv % p->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->cu_seqlens) {
    if (p->B != 1 || p->N < 1) return GDN_ERR_INVALID_ARG;
  } else if (p->N != p->B) {
    return GDN_ERR_INVALID_ARG;
  }
  if (p->T > ((int64_t)1 << 31) - 1 || p->B * p->T > ((int64_t)1 << 31) - 1)
    return GDN_ERR_UNSUPPORTED_SHAPE;  // token indices are int32 on the device
  if (!(p->scale == p->scale)) return GDN_ERR_INVALID_ARG;  // NaN scale
  if (p->save_ctx != 0 && p->save_ctx != 1) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

static bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15) == 0; }

// The KDA recurrence shares the problem description; its own rules: no W site,
// any QDQ period (`chunk` >= 1), state scale widths 16, 32 or 64.
static gdn_status validate_kda(const gdn_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  gdn_problem c = *p;
  if (c.w_mode != GDN_QDQ_NONE) return GDN_ERR_UNSUPPORTED_MODE;
  if (c.chunk < 1) return GDN_ERR_INVALID_ARG;
  if (c.block_v != 16 && c.block_v != 32 && c.block_v != 64) return GDN_ERR_UNSUPPORTED_MODE;
  c.chunk = kChunkLen;
  const gdn_status s = validate(&c);
  if (s != GDN_OK) return s;
  if (c.N > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;  // grid z
  return GDN_OK;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

const char* gdn_status_string(int s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer, negative size or bad enum";
    case GDN_ERR_UNSUPPORTED_DTYPE: return "GDN_ERR_UNSUPPORTED_DTYPE: q/k/v/dO must be bf16";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "GDN_ERR_UNSUPPORTED_SHAPE: Dk/Dv must be 64 or 128, Hv % Hk == 0, chunk 64";
    case GDN_ERR_UNSUPPORTED_MODE: return "GDN_ERR_UNSUPPORTED_MODE: QDQ mode or block_v not supported";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "GDN_ERR_WORKSPACE_TOO_SMALL";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a kernel launch failed";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED: pointers must be 16-byte aligned";
    default: return "unknown gdn_status";
  }
}

int gdn_abi_version(void) { return GDN_QDQ_ABI_VERSION; }

int gdn_device_error(int reset) {
  const int f = fwd_device_error(reset != 0), b = bwd_device_error(reset != 0);
  const int u = fused_device_error(reset != 0);
  return (f < 0 || b < 0 || u < 0) ? -1 : (f | b | u);
}

gdn_status gdn_validate(const gdn_problem* p) { return validate(p); }

int64_t gdn_num_chunk_slots(const gdn_problem* p) {
  if (validate(p) != GDN_OK) return -1;
  return dims_of(*p).n_slots;
}

size_t gdn_ctx_bytes(const gdn_problem* p) {
  if (validate(p) != GDN_OK) return 0;
  return ctx_layout(*p).total;
}

int64_t gdn_ctx_offset(const gdn_problem* p, int segment) {
  if (validate(p) != GDN_OK) return -1;
  const CtxLayout L = ctx_layout(*p);
  switch (segment) {
    case GDN_CTX_W_CODES: return L.w_codes;
    case GDN_CTX_W_SCALES: return L.w_scales;
    case GDN_CTX_W_FULL: return L.w_full;
    case GDN_CTX_CVEC: return L.cvec;
    case GDN_CTX_T_IMG: return L.tb;
    case GDN_CTX_GKK_IMG: return L.gkk;
    case GDN_CTX_P_IMG: return L.pb;
    case GDN_CTX_D_IMG: return L.db;
    case GDN_CTX_TU_IMG: return L.tu_img;
    case GDN_CTX_H_CODES: return L.h_codes;
    case GDN_CTX_H_SCALES: return L.h_scales;
    case GDN_CTX_H_FULL: return L.h_full;
    default: return -1;
  }
}

gdn_status gdn_chunk_fwd_qdq(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* beta, const float* g, const float* h0, float* o,
                             float* ht, void* ctx, void* stream) {
  gdn_status s = validate(p);
  if (s != GDN_OK) return s;
  const Dims d = dims_of(*p);
  if (d.B * d.T > 0 && (!q || !k || !v || !beta || !g || !o)) return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, (const void*)h0,
                          (const void*)o, (const void*)ht, (const void*)ctx,
                          (const void*)p->cu_seqlens})
    if (ptr && !aligned16(ptr)) return GDN_ERR_MISALIGNED;
  if (d.B * d.T > 0 && !ctx) return GDN_ERR_INVALID_ARG;
  if (ctx && ((uintptr_t)ctx & 255)) return GDN_ERR_MISALIGNED;
  if (d.N == 0 || (d.B * d.T == 0 && !ht)) return GDN_OK;
  return launch_fwd(*p, d, q, k, v, beta, g, h0, o, ht, ctx, (cudaStream_t)stream);
}

gdn_status kda_recurrent_fwd_qdq(const gdn_problem* p, const void* q, const void* k,
                                 const void* v, const float* beta, const float* g,
                                 const float* h0, float* o, float* ht, void* stream) {
  const gdn_status s = validate_kda(p);
  if (s != GDN_OK) return s;
  gdn_problem c = *p;
  c.chunk = kChunkLen;
  c.block_v = kChunkLen;
  const Dims d = dims_of(c);
  if (d.B * d.T > 0 && (!q || !k || !v || !beta || !g || !o)) return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, (const void*)h0,
                          (const void*)o, (const void*)ht, (const void*)p->cu_seqlens})
    if (ptr && !aligned16(ptr)) return GDN_ERR_MISALIGNED;
  if (d.N == 0 || (d.B * d.T == 0 && !ht)) return GDN_OK;
  return launch_kda(*p, d, q, k, v, beta, g, h0, o, ht, (cudaStream_t)stream);
}

size_t gdn_bwd_workspace_bytes(const gdn_problem* p) {
  if (validate(p) != GDN_OK) return 0;
  return bwd_workspace_bytes(*p, dims_of(*p));
}

gdn_status gdn_chunk_bwd_ste(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* beta, const float* g, const void* ctx, const void* dO,
                             const float* dht, float* dq, float* dk, float* dv, float* dbeta,
                             float* dg, float* dh0, void* workspace, size_t workspace_bytes,
                             void* stream) {
  gdn_status s = validate(p);
  if (s != GDN_OK) return s;
  if (!p->save_ctx) return GDN_ERR_INVALID_ARG;  // a forward-only context has no backward data
  const Dims d = dims_of(*p);
  const bool any_tokens = d.B * d.T > 0;
  if (any_tokens && (!q || !k || !v || !beta || !g || !ctx || !dO || !dq || !dk || !dv ||
                     !dbeta || !dg))
    return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, ctx, dO,
                          (const void*)dht, (const void*)dq, (const void*)dk, (const void*)dv,
                          (const void*)dbeta, (const void*)dg, (const void*)dh0, (const void*)workspace,
                          (const void*)p->cu_seqlens})
    if (ptr && !aligned16(ptr)) return GDN_ERR_MISALIGNED;
  const size_t need = bwd_workspace_bytes(*p, d);
  if (workspace_bytes < need || (need > 0 && !workspace)) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (d.N == 0) return GDN_OK;
  return launch_bwd(*p, d, q, k, v, beta, g, ctx, dO, dht, dq, dk, dv, dbeta, dg, dh0,
                    workspace, (cudaStream_t)stream);
}

static gdn_status fake_qdq_common(int mode, const float* x, float* y, float* scales,
                                  uint8_t* codes, int64_t batch, int64_t rows, int64_t cols,
                                  int64_t group_cols, void* stream) {
  if (batch < 0 || rows < 0 || cols < 0 || group_cols <= 0 || cols % group_cols != 0)
    return GDN_ERR_INVALID_ARG;
  if (batch * (cols / group_cols) == 0) return GDN_OK;
  if (!x || !y || !scales) return GDN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(scales) || (codes && !aligned16(codes)))
    return GDN_ERR_MISALIGNED;
  return launch_fake_qdq(mode, x, y, scales, codes, batch, rows, cols, group_cols,
                         (cudaStream_t)stream);
}

gdn_status fake_qdq_e4m3(const float* x, float* y, float* scales, uint8_t* codes, int64_t batch,
                         int64_t rows, int64_t cols, int64_t group_cols, void* stream) {
  return fake_qdq_common(GDN_QDQ_E4M3, x, y, scales, codes, batch, rows, cols, group_cols,
                         stream);
}

gdn_status fake_qdq_int8(const float* x, float* y, float* scales, uint8_t* codes, int64_t batch,
                         int64_t rows, int64_t cols, int64_t group_cols, void* stream) {
  return fake_qdq_common(GDN_QDQ_INT8, x, y, scales, codes, batch, rows, cols, group_cols,
                         stream);
}

}  // extern "C"
