// KDA recurrent forward with the state fake QDQ at chunk boundaries ("[1/4]
// GDN state/W QAT foundation", "What does this PR do?": KDA has a recurrent
// reference only; "[2/4] GDN/KDA decode QAT with INT8 recurrent state": the
// E4M3 / INT8 state quantizer with per-head [Dk, block_v] scales).  The
// published Kimi Delta Attention recurrence, H = S^T (Dk x Dv), with a decay
// per key channel:
//     if t % chunk == 0:  H <- Q(H)                  (t from the sequence start)
//     H <- diag(exp(g_t)) H;  H <- H + beta_t k_t (v_t - H^T k_t)^T;  o_t = scale H^T q_t
//
// The columns of H evolve independently given the token vectors, so one CTA
// owns a [Dk x 64] column block of one (sequence, value head) and walks its
// tokens in order with the block in registers: 256 threads, thread (rg, cq)
// holds columns 4cq..4cq+3 of rows rg, rg + 16, ...  Per token two block
// barriers: the column sums H^T k (after the decay) and H^T q reduce across
// the 16 row groups in shared memory.  The next token's vectors are fetched
// into registers while the current token computes.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kKdaThreads = 256;
constexpr int kKdaWarps = kKdaThreads / 32;
constexpr int kKdaC4 = 16;                         // column quads of the 64-column block
constexpr int kKdaRG = kKdaThreads / kKdaC4;       // row groups

struct KdaParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *beta, *g, *h0;
  float *o, *ht;
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, block_v, chunk;
  float scale;
};

__device__ __forceinline__ float4 fma4s(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

template <int MODE>
__device__ __forceinline__ float4 qdq4v(float4 x, float s, float r, bool zero) {
  if (zero) return x;
  return make_float4(__fmul_rn(qdq_code_value<MODE>(qdq_code<MODE>(x.x, r)), s),
                     __fmul_rn(qdq_code_value<MODE>(qdq_code<MODE>(x.y, r)), s),
                     __fmul_rn(qdq_code_value<MODE>(qdq_code<MODE>(x.z, r)), s),
                     __fmul_rn(qdq_code_value<MODE>(qdq_code<MODE>(x.w, r)), s));
}

// column sums over the 16 row groups of per-thread partials (4 columns);
// red: shared [kKdaWarps][64].  Valid for every thread after the barrier.
__device__ __forceinline__ float4 kda_colsum(float4 p, int lane, int warp, float (*red)[64]) {
  p.x += __shfl_xor_sync(0xffffffffu, p.x, 16);
  p.y += __shfl_xor_sync(0xffffffffu, p.y, 16);
  p.z += __shfl_xor_sync(0xffffffffu, p.z, 16);
  p.w += __shfl_xor_sync(0xffffffffu, p.w, 16);
  if (lane < 16) *reinterpret_cast<float4*>(&red[warp][lane * 4]) = p;
  __syncthreads();
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  const int cq = lane & 15;
#pragma unroll
  for (int w = 0; w < kKdaWarps; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(&red[w][cq * 4]);
    s.x += x.x;
    s.y += x.y;
    s.z += x.z;
    s.w += x.w;
  }
  return s;
}

template <int DK, int MODE>
__global__ void __launch_bounds__(kKdaThreads, 1) kda_recurrent_kernel(const KdaParams p) {
  constexpr int RPT = DK / kKdaRG;  // rows per thread
  constexpr bool QUANT = MODE != GDN_QDQ_NONE;
  __shared__ __align__(16) float red[2][kKdaWarps][64];
  __shared__ float amx[kKdaWarps][4];
  __shared__ __align__(16) float tv[2][3][DK];    // k, q, e^g of a token (two tokens in turn)
  __shared__ __align__(16) float tvv[2][64 + 4];  // v block and beta

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % kKdaC4, rg = tid / kKdaC4;
  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
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
  const int tile = (cq * 4) / p.block_v;
  const int64_t sbase = ((int64_t)n * p.Hv + h) * DK * p.Dv + vb * 64 + cq * 4;

  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = p.h0 ? *reinterpret_cast<const float4*>(p.h0 + sbase + (int64_t)(rg + kKdaRG * i) * p.Dv)
                : make_float4(0.f, 0.f, 0.f, 0.f);

  // the next token's vectors in registers: threads < DK hold k, q, g of one
  // key channel; threads < 64 one value; thread 64 (or 0 when DK == 64) beta
  float k_nx = 0.f, q_nx = 0.f, g_nx = 0.f, v_nx = 0.f, b_nx = 0.f;
  auto fetch = [&](int lt) {
    const int64_t t = tok0 + lt;
    if (tid < DK) {
      k_nx = __bfloat162float(p.k[(t * p.Hk + hk) * DK + tid]);
      q_nx = __bfloat162float(p.q[(t * p.Hk + hk) * DK + tid]);
      g_nx = p.g[(t * p.Hv + h) * DK + tid];
    }
    if (tid < 64) v_nx = __bfloat162float(p.v[(t * p.Hv + h) * p.Dv + vb * 64 + tid]);
    if (tid == 64 % DK) b_nx = p.beta[t * p.Hv + h];
  };
  auto publish = [&](int buf) {
    if (tid < DK) {
      tv[buf][0][tid] = k_nx;
      tv[buf][1][tid] = q_nx;
      tv[buf][2][tid] = expf(g_nx);
    }
    if (tid < 64) tvv[buf][tid] = v_nx;
    if (tid == 64 % DK) tvv[buf][64] = b_nx;
  };
  if (L > 0) {
    fetch(0);
    publish(0);
  }
  __syncthreads();

  for (int lt = 0; lt < L; ++lt) {
    const int buf = lt & 1;
    const int64_t t = tok0 + lt;
    if (lt + 1 < L) fetch(lt + 1);

    // ---- state QDQ at chunk boundaries, per [Dk, block_v] tile ----
    if constexpr (QUANT) {
      if (lt % p.chunk == 0) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i)
          m = fmaxf(m, fmaxf(fmaxf(fabsf(S[i].x), fabsf(S[i].y)), fmaxf(fabsf(S[i].z), fabsf(S[i].w))));
        for (int o = 1; o < p.block_v / 4; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (lane < 16 && (cq * 4) % p.block_v == 0) amx[warp][tile] = m;
        __syncthreads();
        float a = amx[0][tile];
#pragma unroll
        for (int w = 1; w < kKdaWarps; ++w) a = fmaxf(a, amx[w][tile]);
        float s, r;
        qdq_scale<MODE>(a, s, r);
#pragma unroll
        for (int i = 0; i < RPT; ++i) S[i] = qdq4v<MODE>(S[i], s, r, a == 0.f);
      }
    }

    // ---- decay per key channel, then H^T k ----
    const float* kv = tv[buf][0];
    const float* qv = tv[buf][1];
    const float* ev = tv[buf][2];
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = rg + kKdaRG * i;
      const float e = ev[row];
      S[i] = make_float4(S[i].x * e, S[i].y * e, S[i].z * e, S[i].w * e);
      part = fma4s(kv[row], S[i], part);
    }
    const float4 kS = kda_colsum(part, lane, warp, red[0]);
    const float4 vv = *reinterpret_cast<const float4*>(&tvv[buf][cq * 4]);
    const float bt = tvv[buf][64];
    const float4 u = make_float4(vv.x - kS.x, vv.y - kS.y, vv.z - kS.z, vv.w - kS.w);

    // ---- write, then the readout H^T q ----
    part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = rg + kKdaRG * i;
      S[i] = fma4s(bt * kv[row], u, S[i]);
      part = fma4s(qv[row], S[i], part);
    }
    // the next token's vectors go to the other buffer before the barrier below
    if (lt + 1 < L) publish(buf ^ 1);
    const float4 os = kda_colsum(part, lane, warp, red[1]);
    if (tid < kKdaC4) {
      const float sc = p.scale;
      *reinterpret_cast<float4*>(p.o + (t * p.Hv + h) * p.Dv + vb * 64 + cq * 4) =
          make_float4(sc * os.x, sc * os.y, sc * os.z, sc * os.w);
    }
  }

  if (p.ht) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      *reinterpret_cast<float4*>(p.ht + sbase + (int64_t)(rg + kKdaRG * i) * p.Dv) = S[i];
  }
}

template <int DK>
gdn_status launch_kda_t(const KdaParams& prm, int mode, const Dims& d, cudaStream_t st) {
  const dim3 grid((unsigned)(d.Dv / 64), (unsigned)d.Hv, (unsigned)d.N);
  if (mode == GDN_QDQ_NONE)
    kda_recurrent_kernel<DK, GDN_QDQ_NONE><<<grid, kKdaThreads, 0, st>>>(prm);
  else if (mode == GDN_QDQ_E4M3)
    kda_recurrent_kernel<DK, GDN_QDQ_E4M3><<<grid, kKdaThreads, 0, st>>>(prm);
  else
    kda_recurrent_kernel<DK, GDN_QDQ_INT8><<<grid, kKdaThreads, 0, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status launch_kda(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const float* h0,
                      float* o, float* ht, cudaStream_t st) {
  KdaParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.h0 = h0;
  prm.o = o;
  prm.ht = ht;
  prm.cu_seqlens = p.cu_seqlens;
  prm.T = d.T;
  prm.Hk = d.Hk;
  prm.Hv = d.Hv;
  prm.Dv = d.Dv;
  prm.block_v = p.block_v;
  prm.chunk = p.chunk;
  prm.scale = p.scale;
  if (d.N == 0) return GDN_OK;
  return d.Dk == 128 ? launch_kda_t<128>(prm, p.state_mode, d, st)
                     : launch_kda_t<64>(prm, p.state_mode, d, st);
}

}  // namespace gdn
