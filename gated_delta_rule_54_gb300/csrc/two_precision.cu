// Two-precision GDN forward: an fp32 recurrence anchor and a dynamic E4M3 read
// copy that only the outputs see ("[5/8] ReplaySSM state QAT and
// two-precision GDN", "What does this PR do?": FP32 recurrence anchor, dynamic
// FP8 E4M3 read copy grouped by the 128 key channels of each value row, a
// recompute from the raw inputs and the anchor at every 16-token flush, read
// errors never overwriting the anchor; GDN, K = 128).  With H = S^T (Dk x Dv),
// t counted from the sequence start and W the flush period:
//     if t % W == 0:  R <- Q_read(A)      (one E4M3 scale per column of H)
//     A <- e^{g_t} A + beta_t k_t (v_t - e^{g_t} A^T k_t)^T
//     R <- e^{g_t} R + beta_t k_t (v_t - e^{g_t} R^T k_t)^T
//     o_t = scale R^T q_t;    ht = A
//
// Every column of H evolves independently given the token vectors, so a warp
// owns four columns over all 128 key rows (lane l holds rows 4l..4l+3) and
// walks the tokens with both states in registers; no block-wide barrier is on
// the token path.  Per token one warp reduction serves three column sums: the
// readout R^T q of this token and A^T k, R^T k of the next one (taken after
// the flush when the next token starts a window).  The sixteen partial sums
// are reduced by halving exchanges (16 shuffles) that leave value j in lanes
// 2j and 2j+1; the next token's sums are gathered back from there (8
// shuffles).  Token vectors are fetched four tokens ahead into a register
// ring.
#include "common.cuh"
#include "launch.h"
#include "two_precision.cuh"

namespace gdn {

namespace {

constexpr int kTpWarps = 4;   // warps per CTA
constexpr int kTpRing = 4;    // tokens in flight per warp

struct TpParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *beta, *g, *h0;
  float *o, *ht;
  float* anchors;  // [slots, Hv, 128, Dv] the anchor entering every window, or null
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, flush;
  float scale;
};

// one token's inputs as a lane needs them: k and q at its four key rows, v at
// the warp's four value columns (bf16, as stored), beta and g
struct TokVec {
  uint2 k, q, v;
  float b, g;
};

template <int RM>
__global__ void __launch_bounds__(kTpWarps * 32) gdn_two_precision_kernel(const TpParams p) {
  constexpr bool READQ = RM != GDN_QDQ_NONE;
  constexpr int NV = READQ ? 16 : 8;   // reduced values per token
  constexpr int LPV = 32 / NV;         // lanes holding each reduced value
  // value slots: A^T k' (0..3), R^T k' (4..7, READQ), R^T q (4..7, or 8..11 with READQ)
  constexpr int J_KA = 0, J_KR = 4, J_O = READQ ? 8 : 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = (blockIdx.x * kTpWarps + warp) * kTpCols;
  const int h = blockIdx.y, n = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);
  int64_t tok0;
  int L;
  if (p.cu_seqlens) {
    tok0 = p.cu_seqlens[n];
    L = (int)(p.cu_seqlens[n + 1] - tok0);
  } else {
    tok0 = (int64_t)n * p.T;
    L = (int)p.T;
  }

  float A[kTpRows][kTpCols], R[kTpRows][kTpCols];
  const int64_t sbase = (((int64_t)n * p.Hv + h) * kTpDk + kTpRows * lane) * p.Dv + c0;
#pragma unroll
  for (int r = 0; r < kTpRows; ++r) {
    const float4 x = p.h0 ? *reinterpret_cast<const float4*>(p.h0 + sbase + (int64_t)r * p.Dv)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    A[r][0] = x.x;
    A[r][1] = x.y;
    A[r][2] = x.z;
    A[r][3] = x.w;
  }

  auto load = [&](int lt) {
    TokVec tv;
    if (lt < L) {
      const int64_t t = tok0 + lt;
      tv.k = __ldg(reinterpret_cast<const uint2*>(p.k + (t * p.Hk + hk) * kTpDk + kTpRows * lane));
      tv.q = __ldg(reinterpret_cast<const uint2*>(p.q + (t * p.Hk + hk) * kTpDk + kTpRows * lane));
      tv.v = __ldg(reinterpret_cast<const uint2*>(p.v + (t * p.Hv + h) * p.Dv + c0));
      tv.b = __ldg(p.beta + t * p.Hv + h);
      tv.g = __ldg(p.g + t * p.Hv + h);
    } else {
      tv.k = tv.q = tv.v = make_uint2(0u, 0u);
      tv.b = tv.g = 0.f;
    }
    return tv;
  };

  // R <- Q_read(A)
  auto flush_read = [&]() {
    if constexpr (READQ) tp_read_copy<RM>(A, R);
  };
  // the anchor entering window w, kept for the backward
  const int64_t slot0 = tp_anchor_slot(tok0, n, 0, p.flush);
  auto save_anchor = [&](int w) {
    if (!p.anchors) return;
    float* dst = p.anchors + (((slot0 + w) * p.Hv + h) * kTpDk + kTpRows * lane) * p.Dv + c0;
#pragma unroll
    for (int r = 0; r < kTpRows; ++r)
      *reinterpret_cast<float4*>(dst + (int64_t)r * p.Dv) = make_float4(A[r][0], A[r][1], A[r][2], A[r][3]);
  };

  TokVec ring[kTpRing];
#pragma unroll
  for (int i = 0; i < kTpRing; ++i) ring[i] = load(i);

  // the first token's column sums A^T k, R^T k
  float kSA[kTpCols], kSR[kTpCols];
  if (L > 0) {
    save_anchor(0);
    flush_read();
    float kr[kTpRows];
    bf16x4(ring[0].k, kr);
    float x[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) x[j] = 0.f;
#pragma unroll
    for (int c = 0; c < kTpCols; ++c)
#pragma unroll
      for (int r = 0; r < kTpRows; ++r) {
        x[J_KA + c] = fmaf(kr[r], A[r][c], x[J_KA + c]);
        if constexpr (READQ) x[J_KR + c] = fmaf(kr[r], R[r][c], x[J_KR + c]);
      }
    const float s = warp_reduce_scatter<NV>(x, lane);
#pragma unroll
    for (int c = 0; c < kTpCols; ++c) {
      kSA[c] = __shfl_sync(0xffffffffu, s, (J_KA + c) * LPV);
      kSR[c] = READQ ? __shfl_sync(0xffffffffu, s, (J_KR + c) * LPV) : kSA[c];
    }
  }

  int left = p.flush;  // tokens of the current window not yet written
  for (int base = 0; base < L; base += kTpRing) {
#pragma unroll
    for (int i = 0; i < kTpRing; ++i) {
      const int lt = base + i;
      if (lt >= L) break;
      const TokVec cur = ring[i];
      const float a = expf(cur.g);
      float kr[kTpRows], qr[kTpRows], vv[kTpCols];
      bf16x4(cur.k, kr);
      bf16x4(cur.q, qr);
      bf16x4(cur.v, vv);
      // ---- the token's write into the anchor and the read state ----
#pragma unroll
      for (int c = 0; c < kTpCols; ++c) {
        const float uA = vv[c] - a * kSA[c];
        const float uR = vv[c] - a * kSR[c];
#pragma unroll
        for (int r = 0; r < kTpRows; ++r) {
          const float bk = cur.b * kr[r];
          A[r][c] = fmaf(bk, uA, a * A[r][c]);
          if constexpr (READQ) R[r][c] = fmaf(bk, uR, a * R[r][c]);
        }
      }
      // ---- this token's readout and the next token's column sums ----
      float x[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) x[j] = 0.f;
#pragma unroll
      for (int c = 0; c < kTpCols; ++c)
#pragma unroll
        for (int r = 0; r < kTpRows; ++r) x[J_O + c] = fmaf(qr[r], READQ ? R[r][c] : A[r][c], x[J_O + c]);
      const bool more = lt + 1 < L;
      if (more && --left == 0) {  // the next token starts a window
        save_anchor((lt + 1) / p.flush);
        flush_read();
        left = p.flush;
      }
      if (more) {
        float nk[kTpRows];
        bf16x4(ring[(i + 1) % kTpRing].k, nk);
#pragma unroll
        for (int c = 0; c < kTpCols; ++c)
#pragma unroll
          for (int r = 0; r < kTpRows; ++r) {
            x[J_KA + c] = fmaf(nk[r], A[r][c], x[J_KA + c]);
            if constexpr (READQ) x[J_KR + c] = fmaf(nk[r], R[r][c], x[J_KR + c]);
          }
      }
      const float s = warp_reduce_scatter<NV>(x, lane);
#pragma unroll
      for (int c = 0; c < kTpCols; ++c) {
        kSA[c] = __shfl_sync(0xffffffffu, s, (J_KA + c) * LPV);
        kSR[c] = READQ ? __shfl_sync(0xffffffffu, s, (J_KR + c) * LPV) : kSA[c];
      }
      // lanes J_O * LPV + c * LPV hold the readout of column c
      const int jo = lane / LPV - J_O;
      if (lane % LPV == 0 && jo >= 0 && jo < kTpCols)
        p.o[((tok0 + lt) * p.Hv + h) * p.Dv + c0 + jo] = p.scale * s;
      ring[i] = load(lt + kTpRing);
    }
  }

  if (p.ht) {
#pragma unroll
    for (int r = 0; r < kTpRows; ++r)
      *reinterpret_cast<float4*>(p.ht + sbase + (int64_t)r * p.Dv) =
          make_float4(A[r][0], A[r][1], A[r][2], A[r][3]);
  }
}

gdn_status launch_two_precision(const gdn_two_precision_problem& p, int64_t N, const void* q,
                                const void* k, const void* v, const float* beta, const float* g,
                                const float* h0, float* o, float* ht, float* anchors,
                                cudaStream_t st) {
  TpParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.h0 = h0;
  prm.o = o;
  prm.ht = ht;
  prm.anchors = anchors;
  prm.cu_seqlens = p.cu_seqlens;
  prm.T = p.T;
  prm.Hk = p.Hk;
  prm.Hv = p.Hv;
  prm.Dv = p.Dv;
  prm.flush = p.flush;
  prm.scale = p.scale;
  const dim3 grid((unsigned)(p.Dv / (kTpWarps * kTpCols)), (unsigned)p.Hv, (unsigned)N);
  if (p.read_mode == GDN_QDQ_E4M3)
    gdn_two_precision_kernel<GDN_QDQ_E4M3><<<grid, kTpWarps * 32, 0, st>>>(prm);
  else
    gdn_two_precision_kernel<GDN_QDQ_NONE><<<grid, kTpWarps * 32, 0, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status validate_two_precision(const gdn_two_precision_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Dk <= 0 || p->Dv <= 0)
    return GDN_ERR_INVALID_ARG;
  if (p->read_mode != GDN_QDQ_NONE && p->read_mode != GDN_QDQ_E4M3) {
    if (p->read_mode == GDN_QDQ_INT8) return GDN_ERR_UNSUPPORTED_MODE;  // FP8 or disabled only
    return GDN_ERR_INVALID_ARG;
  }
  if (p->dtype != GDN_DTYPE_BF16) {
    if (p->dtype == GDN_DTYPE_FP16 || p->dtype == GDN_DTYPE_FP32) return GDN_ERR_UNSUPPORTED_DTYPE;
    return GDN_ERR_INVALID_ARG;
  }
  if (p->flush < 1) return GDN_ERR_INVALID_ARG;
  if (p->Dk != kTpDk || (p->Dv != 64 && p->Dv != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->Hv % p->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->cu_seqlens) {
    if (p->B != 1 || p->N < 1) return GDN_ERR_INVALID_ARG;
  } else if (p->N != p->B) {
    return GDN_ERR_INVALID_ARG;
  }
  if (p->N > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;  // grid z
  if (p->T > ((int64_t)1 << 31) - 1 || p->B * p->T > ((int64_t)1 << 31) - 1)
    return GDN_ERR_UNSUPPORTED_SHAPE;  // token counts are int32 on the device
  if (!(p->scale == p->scale)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

int64_t two_precision_anchor_slots(const gdn_two_precision_problem* p) {
  return p->B * p->T / p->flush + p->N;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_two_precision_validate(const gdn_two_precision_problem* p) {
  return validate_two_precision(p);
}

size_t gdn_two_precision_anchor_bytes(const gdn_two_precision_problem* p) {
  if (validate_two_precision(p) != GDN_OK) return 0;
  return (size_t)two_precision_anchor_slots(p) * p->Hv * kTpDk * p->Dv * sizeof(float);
}

gdn_status gdn_two_precision_fwd(const gdn_two_precision_problem* p, const void* q,
                                 const void* k, const void* v, const float* beta,
                                 const float* g, const float* h0, float* o, float* ht,
                                 float* anchors, void* stream) {
  const gdn_status s = validate_two_precision(p);
  if (s != GDN_OK) return s;
  if (p->B * p->T > 0 && (!q || !k || !v || !beta || !g || !o)) return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, (const void*)h0,
                          (const void*)o, (const void*)ht, (const void*)anchors,
                          (const void*)p->cu_seqlens})
    if (ptr && ((uintptr_t)ptr & 15)) return GDN_ERR_MISALIGNED;
  if (p->N == 0 || (p->B * p->T == 0 && !ht)) return GDN_OK;
  return launch_two_precision(*p, p->N, q, k, v, beta, g, h0, o, ht, anchors,
                              static_cast<cudaStream_t>(stream));
}

}  // extern "C"
