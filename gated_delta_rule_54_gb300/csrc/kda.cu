// KDA recurrent forward with the state fake QDQ at chunk boundaries ("[1/4]
// GDN state/W QAT foundation", "What does this PR do?": KDA has a recurrent
// reference only; "[2/4] GDN/KDA decode QAT with INT8 recurrent state": the
// E4M3 / INT8 state quantizer with per-head [Dk, block_v] scales).  The
// published Kimi Delta Attention recurrence, H = S^T (Dk x Dv), with a decay
// per key channel:
//     if t % chunk == 0:  H <- Q(H)                  (t from the sequence start)
//     H <- diag(exp(g_t)) H;  H <- H + beta_t k_t (v_t - H^T k_t)^T;  o_t = scale H^T q_t
//
// The columns of H evolve independently given the token vectors, so a warp
// owns four value columns over all Dk key rows (lane l: rows RPL l .. RPL l +
// RPL - 1, RPL = Dk / 32) and walks the tokens with its part of H in
// registers; a CTA of 16 warps covers one 64-column value block, which holds
// every [Dk, block_v] scale tile whole.  No block barrier is on the token
// path: per token one warp reduction (halving exchanges, 9 shuffles) serves
// this token's readout H^T q and the next token's H^T (e^{g'} o k'), whose
// four sums are gathered back to every lane (4 shuffles).  The state QDQ
// (every `chunk` tokens) takes the tile amax through shared memory with one
// block barrier (its buffer alternates, so no second barrier is needed).
// Token vectors are fetched four tokens ahead into a register ring.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kKdaWarps = 16;                  // one 64-column value block
constexpr int kKdaThreads = kKdaWarps * 32;
constexpr int kKdaCols = 4;                    // value columns per warp
constexpr int kKdaRing = 4;                    // tokens in flight per warp

struct KdaParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *beta, *g, *h0;
  float *o, *ht;
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, block_v, chunk;
  float scale;
};

// one token's inputs as a lane needs them: k, q and g at its RPL key rows,
// v at the warp's four value columns, beta
template <int RPL>
struct KdaTok {
  uint32_t k[RPL / 2], q[RPL / 2];
  float g[RPL];
  uint2 v;
  float b;
};

template <int RPL>
__device__ __forceinline__ void unpack_rows(const uint32_t (&u)[RPL / 2], float (&x)[RPL]) {
  if constexpr (RPL == 4) {
    bf16x4(make_uint2(u[0], u[1]), x);
  } else {
    bf16x2(u[0], x);
  }
}

template <int DK, int MODE>
__global__ void __launch_bounds__(kKdaThreads, 1) kda_recurrent_kernel(const KdaParams p) {
  constexpr int RPL = DK / 32;  // key rows per lane
  constexpr bool QUANT = MODE != GDN_QDQ_NONE;
  __shared__ float amx[2][kKdaWarps];  // per-warp amax, alternate buffers

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blockIdx.x * 64 + warp * kKdaCols;
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

  float H[RPL][kKdaCols];
  const int64_t sbase = (((int64_t)n * p.Hv + h) * DK + RPL * lane) * p.Dv + c0;
#pragma unroll
  for (int r = 0; r < RPL; ++r) {
    const float4 x = p.h0 ? *reinterpret_cast<const float4*>(p.h0 + sbase + (int64_t)r * p.Dv)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    H[r][0] = x.x;
    H[r][1] = x.y;
    H[r][2] = x.z;
    H[r][3] = x.w;
  }

  auto load = [&](int lt) {
    KdaTok<RPL> tv;
    if (lt < L) {
      const int64_t t = tok0 + lt;
      const int64_t kq = (t * p.Hk + hk) * DK + RPL * lane;
      const int64_t gr = (t * p.Hv + h) * DK + RPL * lane;
      if constexpr (RPL == 4) {
        const uint2 kk = __ldg(reinterpret_cast<const uint2*>(p.k + kq));
        const uint2 qq = __ldg(reinterpret_cast<const uint2*>(p.q + kq));
        const float4 gg = __ldg(reinterpret_cast<const float4*>(p.g + gr));
        tv.k[0] = kk.x; tv.k[1] = kk.y;
        tv.q[0] = qq.x; tv.q[1] = qq.y;
        tv.g[0] = gg.x; tv.g[1] = gg.y; tv.g[2] = gg.z; tv.g[3] = gg.w;
      } else {
        tv.k[0] = __ldg(reinterpret_cast<const uint32_t*>(p.k + kq));
        tv.q[0] = __ldg(reinterpret_cast<const uint32_t*>(p.q + kq));
        const float2 gg = __ldg(reinterpret_cast<const float2*>(p.g + gr));
        tv.g[0] = gg.x; tv.g[1] = gg.y;
      }
      tv.v = __ldg(reinterpret_cast<const uint2*>(p.v + (t * p.Hv + h) * p.Dv + c0));
      tv.b = __ldg(p.beta + t * p.Hv + h);
    } else {
#pragma unroll
      for (int i = 0; i < RPL / 2; ++i) tv.k[i] = tv.q[i] = 0u;
#pragma unroll
      for (int i = 0; i < RPL; ++i) tv.g[i] = 0.f;
      tv.v = make_uint2(0u, 0u);
      tv.b = 0.f;
    }
    return tv;
  };

  // H <- Q(H) per [Dk, block_v] tile: the warp's four columns lie in one tile
  // of block_v / 4 warps; their amax meet in shared memory
  int par = 0;
  auto qdq = [&]() {
    if constexpr (QUANT) {
      float m = 0.f;
#pragma unroll
      for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int c = 0; c < kKdaCols; ++c) m = fmaxf(m, fabsf(H[r][c]));
      m = warp_max(m);
      if (lane == 0) amx[par][warp] = m;
      __syncthreads();
      const int wpt = p.block_v / kKdaCols;  // warps per tile
      const int w0 = warp - warp % wpt;
      float a = 0.f;
      for (int w = w0; w < w0 + wpt; ++w) a = fmaxf(a, amx[par][w]);
      par ^= 1;
      float s, rcp;
      qdq_scale<MODE>(a, s, rcp);
      if (a != 0.f) {
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
          for (int c = 0; c < kKdaCols; ++c)
            H[r][c] = __fmul_rn(qdq_code_value<MODE>(qdq_code<MODE>(H[r][c], rcp)), s);
      }
    }
  };

  KdaTok<RPL> ring[kKdaRing];
#pragma unroll
  for (int i = 0; i < kKdaRing; ++i) ring[i] = load(i);

  // the first token: QDQ at t = 0, its decays and its column sums H^T (e^g o k)
  float kS[kKdaCols], dec[RPL];
  if (L > 0) {
    qdq();
    float kr[RPL];
    unpack_rows<RPL>(ring[0].k, kr);
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.f;
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      dec[r] = expf(ring[0].g[r]);
      const float kd = dec[r] * kr[r];
#pragma unroll
      for (int c = 0; c < kKdaCols; ++c) x[c] = fmaf(kd, H[r][c], x[c]);
    }
    const float s = warp_reduce_scatter<8>(x, lane);
#pragma unroll
    for (int c = 0; c < kKdaCols; ++c) kS[c] = __shfl_sync(0xffffffffu, s, c * 4);
  }

  int left = p.chunk;  // tokens of the current QDQ period not yet written
  for (int base = 0; base < L; base += kKdaRing) {
#pragma unroll
    for (int i = 0; i < kKdaRing; ++i) {
      const int lt = base + i;
      if (lt >= L) break;
      const KdaTok<RPL> cur = ring[i];
      float kr[RPL], qr[RPL], vv[kKdaCols];
      unpack_rows<RPL>(cur.k, kr);
      unpack_rows<RPL>(cur.q, qr);
      bf16x4(cur.v, vv);
      // ---- the token's write: H <- diag(e^g) H + beta k (v - (diag(e^g) H)^T k)^T ----
#pragma unroll
      for (int c = 0; c < kKdaCols; ++c) {
        const float u = vv[c] - kS[c];
#pragma unroll
        for (int r = 0; r < RPL; ++r) H[r][c] = fmaf(cur.b * kr[r], u, dec[r] * H[r][c]);
      }
      // ---- this token's readout, then the next token's column sums ----
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.f;
#pragma unroll
      for (int c = 0; c < kKdaCols; ++c)
#pragma unroll
        for (int r = 0; r < RPL; ++r) x[4 + c] = fmaf(qr[r], H[r][c], x[4 + c]);
      const bool more = lt + 1 < L;
      if (more && --left == 0) {  // the next token starts a QDQ period
        qdq();
        left = p.chunk;
      }
      if (more) {
        const KdaTok<RPL>& nx = ring[(i + 1) % kKdaRing];
        float nk[RPL];
        unpack_rows<RPL>(nx.k, nk);
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
          dec[r] = expf(nx.g[r]);
          const float kd = dec[r] * nk[r];
#pragma unroll
          for (int c = 0; c < kKdaCols; ++c) x[c] = fmaf(kd, H[r][c], x[c]);
        }
      }
      const float s = warp_reduce_scatter<8>(x, lane);
#pragma unroll
      for (int c = 0; c < kKdaCols; ++c) kS[c] = __shfl_sync(0xffffffffu, s, c * 4);
      // lanes 16, 20, 24, 28 hold the readouts of the four columns
      if (lane >= 16 && (lane & 3) == 0)
        p.o[((tok0 + lt) * p.Hv + h) * p.Dv + c0 + ((lane >> 2) - 4)] = p.scale * s;
      ring[i] = load(lt + kKdaRing);
    }
  }

  if (p.ht) {
#pragma unroll
    for (int r = 0; r < RPL; ++r)
      *reinterpret_cast<float4*>(p.ht + sbase + (int64_t)r * p.Dv) =
          make_float4(H[r][0], H[r][1], H[r][2], H[r][3]);
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
