// Decode QAT: gated delta rule token steps with a state fake QDQ before every
// token ("[2/4] GDN/KDA decode QAT with INT8 recurrent state", "What does this
// PR do?": token-state writes after an exact chunked prefill; E4M3 or signed
// symmetric INT8 with per-head [Dk, block_v] scales; "Testing": both readouts,
// split carry, all state scale widths).  Per value head, with H = S^T:
//     S^ = Q(S);  H = exp(g) S^ + beta k (v - exp(g) S^^T k)^T;
//     o = scale H^T q (pre) or scale Q(H)^T q (post);  S <- H.
//
// One CTA owns the W columns of one (row, value head) state, Dk x W fp32 (<=
// 64 KB), held in registers for all the call's tokens: the state is read from
// HBM once and written once per call, so the step is bound by HBM traffic.
// Every column's update and readout involve only that column (and the
// [Dk, block_v] tile it belongs to), so with block_v <= 64 a 128-wide state is
// split into two 64-column CTAs of 256 threads: four CTAs per SM keep more
// state loads in flight while others compute.  Thread (rg, cq) holds columns
// 4cq..4cq+3 of rows rg, rg + RG, ... (a warp load covers whole rows of the
// block, coalesced).  Column dot products reduce across the RG row groups
// through shared memory; tile maxima reduce with shuffles inside a warp and
// shared memory across warps.
#include "common.cuh"

namespace gdn {

namespace {


struct DecodeParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *beta, *g, *state_in;
  float *o, *state_out, *scales;
  uint8_t* codes;
  int64_t B, T;
  int Hk, Hv, block_v;
  float scale;
};

__device__ __forceinline__ float4 f4_fma(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

__device__ __forceinline__ float max_abs4(float4 x) {
  return fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
}

template <int MODE>
__device__ __forceinline__ float qdq1(float x, float s, float r, bool zero, uint8_t& c) {
  if (zero) {
    c = qdq_zero_code<MODE>(x);
    return x;
  }
  c = qdq_code<MODE>(x, r);
  return __fmul_rn(qdq_code_value<MODE>(c), s);
}

template <int MODE>
__device__ __forceinline__ float4 qdq4(float4 x, float s, float r, bool zero, uint32_t& c4) {
  uint8_t c0, c1, c2, c3;
  float4 y;
  y.x = qdq1<MODE>(x.x, s, r, zero, c0);
  y.y = qdq1<MODE>(x.y, s, r, zero, c1);
  y.z = qdq1<MODE>(x.z, s, r, zero, c2);
  y.w = qdq1<MODE>(x.w, s, r, zero, c3);
  c4 = (uint32_t)c0 | ((uint32_t)c1 << 8) | ((uint32_t)c2 << 16) | ((uint32_t)c3 << 24);
  return y;
}

// Per-tile amax of the CTA's state.  Every thread returns the amax of the
// [Dk, block_v] tile its columns fall in.  amx: shared [NW][8].
template <int C4, int NW>
__device__ __forceinline__ float tile_amax(float m, int block_v, int lane, int warp, int tile,
                                           float (*amx)[8]) {
  // lanes of one tile and one row group differ in the low log2(block_v/4) bits
  for (int o = 1; o < block_v / 4 && o < C4; o <<= 1)
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if constexpr (C4 < 32) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, C4));  // two row groups
  const int cq = lane % C4;
  if (lane < C4 && (cq * 4) % block_v == 0) amx[warp][tile] = m;
  __syncthreads();
  float a = amx[0][tile];
#pragma unroll
  for (int w = 1; w < NW; ++w) a = fmaxf(a, amx[w][tile]);
  return a;
}

// Column sums over all rows of per-thread partials p (4 columns), returned
// to every thread for its own columns.  red: shared [NW][W].
template <int C4, int W, int NW>
__device__ __forceinline__ float4 column_sum(float4 p, int lane, int warp, float (*red)[W],
                                             bool all_threads) {
  if constexpr (C4 < 32) {
    p.x += __shfl_xor_sync(0xffffffffu, p.x, C4);
    p.y += __shfl_xor_sync(0xffffffffu, p.y, C4);
    p.z += __shfl_xor_sync(0xffffffffu, p.z, C4);
    p.w += __shfl_xor_sync(0xffffffffu, p.w, C4);
  }
  const int cq = lane % C4;
  if (lane < C4) *reinterpret_cast<float4*>(&red[warp][cq * 4]) = p;
  __syncthreads();
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (all_threads) {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(&red[w][cq * 4]);
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
  }
  return s;
}

// DV: the state's value width (row stride); W: the CTA's columns (DV, or 64
// with blockIdx.z the 64-column block); NT: threads.
template <int DK, int DV, int W, int NT, int MODE, bool POST>
__global__ void __launch_bounds__(NT, 1024 / NT) gdn_decode_kernel(const DecodeParams p) {
  constexpr int NW = NT / 32;             // warps
  constexpr int C4 = W / 4;               // column quads
  constexpr int RG = NT / C4;             // row groups
  constexpr int RPT = DK / RG;            // rows per thread
  constexpr bool QUANT = MODE != GDN_QDQ_NONE;
  static_assert(RPT >= 1 && DK % RG == 0 && DK <= NT, "layout");

  __shared__ __align__(16) float red[2][NW][W];
  __shared__ float amx[2][NW][8];
  __shared__ float ks[DK], qs[DK];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % C4, rg = tid / C4;
  const int h = blockIdx.x;
  const int64_t b = blockIdx.y;
  const int c0 = (int)blockIdx.z * W + cq * 4;  // this thread's first column
  const int hk = h / (p.Hv / p.Hk);
  const int tile = c0 / p.block_v;
  const int64_t sbase = (b * p.Hv + h) * (int64_t)DK * DV;

  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int64_t e = sbase + (int64_t)(rg + RG * i) * DV + c0;
    S[i] = p.state_in ? __ldg(reinterpret_cast<const float4*>(p.state_in + e))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // token vectors of the next token, prefetched into registers
  auto tok_of = [&](int64_t t) { return b * p.T + t; };
  __nv_bfloat16 k_nx = __float2bfloat16(0.f), q_nx = k_nx;
  uint2 v_nx = make_uint2(0u, 0u);
  float beta_nx = 0.f, g_nx = 0.f;
  auto prefetch = [&](int64_t t) {
    const int64_t tk = tok_of(t);
    if (tid < DK) {
      k_nx = p.k[(tk * p.Hk + hk) * DK + tid];
      q_nx = p.q[(tk * p.Hk + hk) * DK + tid];
    }
    v_nx = *reinterpret_cast<const uint2*>(p.v + (tk * p.Hv + h) * DV + c0);
    beta_nx = p.beta[tk * p.Hv + h];
    g_nx = p.g[tk * p.Hv + h];
  };
  if (p.T > 0) prefetch(0);

  float s_c = 0.f, r_c = 0.f, a_c = 0.f;  // scale, reciprocal, amax of the next token's Q
  bool cached = false;

  for (int64_t t = 0; t < p.T; ++t) {
    const int64_t tk = tok_of(t);
    if (tid < DK) {
      ks[tid] = __bfloat162float(k_nx);
      qs[tid] = __bfloat162float(q_nx);
    }
    const uint2 vraw = v_nx;
    const float bt = beta_nx, gt = g_nx;
    if (t + 1 < p.T) prefetch(t + 1);

    // ---- S^ = Q(S) per [Dk, block_v] tile ----
    if constexpr (QUANT) {
      if (!cached) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) m = fmaxf(m, max_abs4(S[i]));
        a_c = tile_amax<C4, NW>(m, p.block_v, lane, warp, tile, amx[0]);
        qdq_scale<MODE>(a_c, s_c, r_c);
      }
      const bool zero = a_c == 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        uint32_t c4;
        S[i] = qdq4<MODE>(S[i], s_c, r_c, zero, c4);
        if (p.codes) {
          const int64_t e = ((tk * p.Hv + h) * DK + rg + RG * i) * DV + c0;
          *reinterpret_cast<uint32_t*>(p.codes + e) = c4;
        }
      }
      if (p.scales && rg == 0 && c0 % p.block_v == 0)
        p.scales[(tk * p.Hv + h) * (DV / p.block_v) + tile] = s_c;
    }
    __syncthreads();  // ks, qs visible; amx[0] reads done

    // ---- decay, k-projection, delta write ----
    const float a = expf(gt);
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      S[i].x *= a;
      S[i].y *= a;
      S[i].z *= a;
      S[i].w *= a;
      part = f4_fma(ks[rg + RG * i], S[i], part);
    }
    const float4 kS = column_sum<C4, W, NW>(part, lane, warp, red[0], true);
    const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vraw.x));
    const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vraw.y));
    const float4 u = make_float4(v01.x - kS.x, v01.y - kS.y, v23.x - kS.z, v23.y - kS.w);
#pragma unroll
    for (int i = 0; i < RPT; ++i) S[i] = f4_fma(bt * ks[rg + RG * i], u, S[i]);

    // ---- readout ----
    part = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (POST && QUANT) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) m = fmaxf(m, max_abs4(S[i]));
      a_c = tile_amax<C4, NW>(m, p.block_v, lane, warp, tile, amx[1]);
      qdq_scale<MODE>(a_c, s_c, r_c);
      cached = true;
      const bool zero = a_c == 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        uint32_t c4;
        part = f4_fma(qs[rg + RG * i], qdq4<MODE>(S[i], s_c, r_c, zero, c4), part);
      }
    } else {
#pragma unroll
      for (int i = 0; i < RPT; ++i) part = f4_fma(qs[rg + RG * i], S[i], part);
    }
    const float4 os = column_sum<C4, W, NW>(part, lane, warp, red[1], rg == 0);
    if (rg == 0) {
      const float sc = p.scale;
      *reinterpret_cast<float4*>(p.o + (tk * p.Hv + h) * DV + c0) =
          make_float4(sc * os.x, sc * os.y, sc * os.z, sc * os.w);
    }
  }

#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int64_t e = sbase + (int64_t)(rg + RG * i) * DV + c0;
    *reinterpret_cast<float4*>(p.state_out + e) = S[i];
  }
}

template <int DK, int DV, int MODE, bool POST>
gdn_status launch_t(const DecodeParams& prm, cudaStream_t st) {
  if constexpr (DV == 128) {
    if (prm.block_v <= 64) {
      // two 64-column CTAs of 256 threads per state (every scale tile inside one)
      const dim3 grid((unsigned)prm.Hv, (unsigned)prm.B, 2u);
      gdn_decode_kernel<DK, DV, 64, 256, MODE, POST><<<grid, 256, 0, st>>>(prm);
      return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
  }
  const dim3 grid((unsigned)prm.Hv, (unsigned)prm.B, 1u);
  gdn_decode_kernel<DK, DV, DV, 512, MODE, POST><<<grid, 512, 0, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int DK, int DV>
gdn_status dispatch(const DecodeParams& prm, int mode, bool post, cudaStream_t st) {
  if (mode == GDN_QDQ_NONE) return launch_t<DK, DV, GDN_QDQ_NONE, false>(prm, st);
  if (mode == GDN_QDQ_E4M3)
    return post ? launch_t<DK, DV, GDN_QDQ_E4M3, true>(prm, st)
                : launch_t<DK, DV, GDN_QDQ_E4M3, false>(prm, st);
  return post ? launch_t<DK, DV, GDN_QDQ_INT8, true>(prm, st)
              : launch_t<DK, DV, GDN_QDQ_INT8, false>(prm, st);
}

bool aligned(const void* ptr, uintptr_t a) { return ((uintptr_t)ptr & (a - 1)) == 0; }

gdn_status validate_decode(const gdn_decode_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hk <= 0 || p->Hv <= 0) return GDN_ERR_INVALID_ARG;
  if (p->state_mode != GDN_QDQ_NONE && p->state_mode != GDN_QDQ_E4M3 &&
      p->state_mode != GDN_QDQ_INT8)
    return GDN_ERR_INVALID_ARG;
  if (p->readout != GDN_READOUT_PRE && p->readout != GDN_READOUT_POST) return GDN_ERR_INVALID_ARG;
  if (p->dtype != GDN_DTYPE_BF16) {
    if (p->dtype == GDN_DTYPE_FP16 || p->dtype == GDN_DTYPE_FP32) return GDN_ERR_UNSUPPORTED_DTYPE;
    return GDN_ERR_INVALID_ARG;
  }
  if ((p->Dk != 64 && p->Dk != 128) || (p->Dv != 64 && p->Dv != 128))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->Hv % p->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (p->block_v != 16 && p->block_v != 32 && p->block_v != 64 && p->block_v != 128)
    return GDN_ERR_UNSUPPORTED_MODE;
  if (p->block_v > p->Dv) return GDN_ERR_UNSUPPORTED_MODE;
  if (p->B > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;  // grid y
  if (!(p->scale == p->scale)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // namespace

}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_decode_validate(const gdn_decode_problem* p) { return validate_decode(p); }

gdn_status gdn_decode_qdq(const gdn_decode_problem* p, const void* q, const void* k,
                          const void* v, const float* beta, const float* g,
                          const float* state_in, float* o, float* state_out, uint8_t* codes,
                          float* scales, void* stream) {
  const gdn_status s = validate_decode(p);
  if (s != GDN_OK) return s;
  const bool tokens = p->B * p->T > 0;
  if (tokens && (!q || !k || !v || !beta || !g || !o)) return GDN_ERR_INVALID_ARG;
  if (p->B > 0 && !state_out) return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, (const void*)state_in,
                          (const void*)o, (const void*)state_out, (const void*)codes,
                          (const void*)scales})
    if (ptr && !aligned(ptr, 16)) return GDN_ERR_MISALIGNED;
  // state_out may be state_in itself; any other overlap would race
  if (state_in && state_out && state_in != state_out) {
    const size_t bytes = sizeof(float) * (size_t)p->B * p->Hv * p->Dk * p->Dv;
    const uintptr_t a = (uintptr_t)state_in, c = (uintptr_t)state_out;
    if (a < c + bytes && c < a + bytes) return GDN_ERR_INVALID_ARG;
  }
  if (p->B == 0) return GDN_OK;
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.state_in = state_in;
  prm.o = o;
  prm.state_out = state_out;
  prm.codes = p->state_mode != GDN_QDQ_NONE ? codes : nullptr;
  prm.scales = p->state_mode != GDN_QDQ_NONE ? scales : nullptr;
  prm.B = p->B;
  prm.T = p->T;
  prm.Hk = p->Hk;
  prm.Hv = p->Hv;
  prm.block_v = p->block_v;
  prm.scale = p->scale;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool post = p->readout == GDN_READOUT_POST;
  if (p->Dk == 128)
    return p->Dv == 128 ? dispatch<128, 128>(prm, p->state_mode, post, st)
                        : dispatch<128, 64>(prm, p->state_mode, post, st);
  return p->Dv == 128 ? dispatch<64, 128>(prm, p->state_mode, post, st)
                      : dispatch<64, 64>(prm, p->state_mode, post, st);
}

}  // extern "C"
