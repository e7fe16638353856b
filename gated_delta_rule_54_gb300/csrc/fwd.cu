// Fused forward of the chunked gated delta rule with state / W fake QDQ.
//
// Method: GatedDeltaNet chunked training form with QDQ at the recurrent-state
// and WY "W" sites ("[1/4] GDN state/W QAT foundation", "What does this PR
// do?": chunk 64, dynamic E4M3, exact triangular solve, quantized W saved for
// backward; "Usage": state tiles [Dk, block_v = 64], W groups per (batch,
// head, chunk); "[2/4] GDN/KDA decode QAT with INT8 recurrent state": INT8
// variant).  Per chunk of L <= 64 tokens with state H (Dk x Dv, H = S^T):
//   gamma = cumsum(g);  A = strict-lower(beta_i e^{gamma_i-gamma_j} k_i.k_j);
//   T = (I + A)^-1;  W = T diag(beta e^gamma) K;  U = T diag(beta) V;
//   W^ = Q_W(W);  H^ = Q_S(H);  Delta = U - W^ H^;
//   O = scale (diag(e^gamma) Q H^ + (lower-incl(e^{gamma_i-gamma_j} q_i.k_j)) Delta);
//   H <- e^{gamma_L} H^ + (diag(e^{gamma_L - gamma}) K)^T Delta.
//
// GB300 design: one CTA (8 warps) per (sequence, value head, 64-wide value
// block) walks its chunks in order; the fp32 state tile [Dk x 64] never
// leaves registers.  Everything chunk-local (KK^T, the solve, W, U, QK^T) is
// recomputed per CTA, so HBM traffic is the algorithmic minimum: q, k, v,
// beta, g in, o (+ final state, + optional saved context) out.  Contractions
// run on tensor cores in bf16 with fp32 accumulation.  Operands that are not
// exactly bf16 (T, Delta, the decayed Delta, P, and unquantized W / H) are
// split into hi + lo bf16 halves so the state path keeps ~16 mantissa bits:
// a plain bf16 rounding of these flips far more quantization codes than the
// fp32 arithmetic of the definition would.  Quantized W and H are fed to the
// tensor cores as their codes (E4M3 values and INT8 integers are exact in
// bf16), with the fp32 scales applied in the epilogues.
// K and Q chunks are double-buffered with cp.async; V is prefetched once U
// has consumed it.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

struct FwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* beta;
  const float* g;
  const float* h0;
  float* o;
  float* ht;
  uint8_t* w_codes;
  float* w_scales;
  uint8_t* h_codes;
  float* h_scales;
  float* h_full;
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, G;
  int64_t nt_fixed;
  float scale;
};

template <int DK, int SM, int WM>
struct Smem {
  static constexpr int kTileK = kChunk * DK * 2;      // bf16 [64][DK]
  static constexpr int kTile64 = kChunk * 64 * 2;     // bf16 [64][64]
  static constexpr int kF32 = kF32Tile;                // f32  [64][kSA]
  static constexpr int K = 0;                          // 2 buffers
  static constexpr int Q = K + 2 * kTileK;             // 2 buffers
  static constexpr int V = Q + 2 * kTileK;
  static constexpr int BG = V + kTile64;               // 2 x (beta[64], g[64])
  static constexpr int VEC = BG + 2 * 2 * 64 * 4;      // gamma, e^g, beta e^g, beta, decay
  static constexpr int A = VEC + 5 * 64 * 4 + 256;
  static constexpr int TT = A + kF32;
  static constexpr int TW = TT + kF32;                 // Tw hi/lo -> (H code staging) -> Delta' hi/lo
  static constexpr int TU = TW + 2 * kTile64;          // Tu hi/lo -> Delta hi/lo
  static constexpr int P = TU + 2 * kTile64;           // P hi/lo
  static constexpr int WC = P + 2 * kTile64;           // W^ codes (or W hi [, lo])
  static constexpr int WC_N = (WM == GDN_QDQ_NONE) ? 2 : 1;
  static constexpr int HC = WC + WC_N * kTileK;        // H^ codes (or H hi [, lo]) [DK][64]
  static constexpr int HC_N = (SM == GDN_QDQ_NONE) ? 2 : 1;
  static constexpr int BYTES = HC + HC_N * DK * 64 * 2;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert((A % 128) == 0 && (TW % 128) == 0 && (WC % 128) == 0 && (HC % 128) == 0,
                "tile alignment");
};

// Issue the async loads of chunk rows [t0, t0 + 64) of one sequence
// (rows >= L zero-filled) into the K / Q buffers and the beta/g staging.
template <int DK>
__device__ __forceinline__ void load_kq(const FwdParams& p, unsigned char* sm, int kOff,
                                        int qOff, int bgOff, int64_t tok0, int L, int hk, int h) {
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm + kOff);
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(sm + qOff);
  constexpr int CPR = DK / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < kChunk * CPR; i += kThreads) {
    const int r = i / CPR, c = i % CPR;
    const bool ok = r < L;
    const int64_t tok = tok0 + (ok ? r : 0);
    const __nv_bfloat16* ks = p.k + (tok * p.Hk + hk) * DK + c * 8;
    const __nv_bfloat16* qs = p.q + (tok * p.Hk + hk) * DK + c * 8;
    cp_async16(smem_u32(Ks + swz<DK>(r, c * 8)), ks, ok ? 16 : 0);
    cp_async16(smem_u32(Qs + swz<DK>(r, c * 8)), qs, ok ? 16 : 0);
  }
  if (threadIdx.x < 2 * kChunk) {
    const int r = threadIdx.x & 63;
    const bool ok = r < L;
    const int64_t tok = tok0 + (ok ? r : 0);
    const float* src = (threadIdx.x < kChunk ? p.beta : p.g) + tok * p.Hv + h;
    const uint32_t dst = smem_u32(sm + bgOff + threadIdx.x * 4);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                 "r"(ok ? 4 : 0));
  }
}

__device__ __forceinline__ void load_v(const FwdParams& p, unsigned char* sm, int vOff,
                                       int64_t tok0, int L, int h, int vb) {
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(sm + vOff);
  for (int i = threadIdx.x; i < kChunk * 8; i += kThreads) {
    const int r = i >> 3, c = i & 7;
    const bool ok = r < L;
    const int64_t tok = tok0 + (ok ? r : 0);
    const __nv_bfloat16* src = p.v + (tok * p.Hv + h) * p.Dv + vb * 64 + c * 8;
    cp_async16(smem_u32(Vs + swz<64>(r, c * 8)), src, ok ? 16 : 0);
  }
}

template <int DK, int SM, int WM>
__global__ void __launch_bounds__(kThreads, 1) gdn_fwd_kernel(const FwdParams p) {
  using S = Smem<DK, SM, WM>;
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ float red[2][kWarps];

  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;

  int64_t tok0, slot0;
  int L;
  if (p.cu_seqlens) {
    const int64_t a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
    tok0 = a;
    L = (int)(b - a);
    slot0 = a / kChunk + n;
  } else {
    tok0 = (int64_t)n * p.T;
    L = (int)p.T;
    slot0 = (int64_t)n * p.nt_fixed;
  }
  const int nchunks = (L + kChunk - 1) / kChunk;

  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(sm + S::V);
  float* gam = reinterpret_cast<float*>(sm + S::VEC);
  float* eg = gam + 64;
  float* beg = gam + 128;
  float* bet = gam + 192;
  float* dec = gam + 256;
  float* As = reinterpret_cast<float*>(sm + S::A);
  float* Ts = reinterpret_cast<float*>(sm + S::TT);
  __nv_bfloat16* TwH = reinterpret_cast<__nv_bfloat16*>(sm + S::TW);
  __nv_bfloat16* TwL = TwH + kChunk * 64;
  __nv_bfloat16* TuH = reinterpret_cast<__nv_bfloat16*>(sm + S::TU);
  __nv_bfloat16* TuL = TuH + kChunk * 64;
  __nv_bfloat16* PH = reinterpret_cast<__nv_bfloat16*>(sm + S::P);
  __nv_bfloat16* PL = PH + kChunk * 64;
  __nv_bfloat16* WcH = reinterpret_cast<__nv_bfloat16*>(sm + S::WC);
  __nv_bfloat16* WcL = WcH + kChunk * DK;  // only with WM == NONE
  __nv_bfloat16* HcH = reinterpret_cast<__nv_bfloat16*>(sm + S::HC);
  __nv_bfloat16* HcL = HcH + DK * 64;      // only with SM == NONE
  __nv_bfloat16* DpH = TwH;                // Delta' = diag(e^{gL - gamma}) Delta
  __nv_bfloat16* DpL = TwL;
  __nv_bfloat16* DH = TuH;
  __nv_bfloat16* DL = TuL;
  uint8_t* Hstage = reinterpret_cast<uint8_t*>(sm + S::TW);  // [DK][64] codes
  uint8_t* Wstage = reinterpret_cast<uint8_t*>(sm + S::TT);  // [64][DK] codes
  float* Ostage = As;                                         // [64][kSA] f32
  constexpr int OSTR = kSA;

  // warp tiles: [64 x 64] outputs -> 16 x 16 per warp; [64 x DK] -> 16 x DK/4
  const int rt = warp & 3, cq = warp >> 2;
  const int row0 = rt * 16, col0 = cq * 16;
  constexpr int NTW = DK / 32;
  const int wcol0 = cq * (DK / 4);
  // state tile [DK x 64]
  constexpr int HM = DK / 16;            // row tiles
  constexpr int HN = kWarps / HM;        // warps per row tile
  constexpr int NTH = 8 / HN;            // 8-wide n tiles per warp
  const int h_row0 = (warp % HM) * 16;
  const int h_col0 = (warp / HM) * (64 / HN);
  float hreg[NTH][4];
  {
    const float* src = p.h0 ? p.h0 + (((int64_t)n * p.Hv + h) * DK) * p.Dv + vb * 64 : nullptr;
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int d = h_row0 + gq + 8 * e2, c = h_col0 + nt * 8 + 2 * tq;
        float2 v2 = make_float2(0.f, 0.f);
        if (src) v2 = *reinterpret_cast<const float2*>(src + (int64_t)d * p.Dv + c);
        hreg[nt][2 * e2] = v2.x;
        hreg[nt][2 * e2 + 1] = v2.y;
      }
  }

  // Prologue: chunk 0 (K, Q, beta/g, V) and chunk 1 (K, Q, beta/g).
  if (nchunks > 0) {
    load_kq<DK>(p, sm, S::K, S::Q, S::BG, tok0, min(L, kChunk), hk, h);
    load_v(p, sm, S::V, tok0, min(L, kChunk), h, vb);
  }
  cp_async_commit();
  if (nchunks > 1)
    load_kq<DK>(p, sm, S::K + S::kTileK, S::Q + S::kTileK, S::BG + 512, tok0 + kChunk,
                min(L - kChunk, kChunk), hk, h);
  cp_async_commit();

  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int Lc = min(L - c * kChunk, kChunk);
    const int64_t ctok = tok0 + (int64_t)c * kChunk;
    const int64_t slot = slot0 + c;
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm + S::K + buf * S::kTileK);
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(sm + S::Q + buf * S::kTileK);
    const float* bsrc = reinterpret_cast<const float*>(sm + S::BG + buf * 512);
    cp_async_wait<1>();
    __syncthreads();

    // ---- a1: in-chunk cumulative log decay (warp 0; padded rows have g = 0) ----
    if (warp == 0) {
      const float g0 = bsrc[64 + 2 * lane], g1 = bsrc[64 + 2 * lane + 1];
      float s = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      const float gam1 = s, gam0 = s - g1;
      const float gL = __shfl_sync(0xffffffffu, s, 31);
      const float b0 = bsrc[2 * lane], b1 = bsrc[2 * lane + 1];
      gam[2 * lane] = gam0;
      gam[2 * lane + 1] = gam1;
      const float e0 = expf(gam0), e1 = expf(gam1);
      eg[2 * lane] = e0;
      eg[2 * lane + 1] = e1;
      beg[2 * lane] = b0 * e0;
      beg[2 * lane + 1] = b1 * e1;
      bet[2 * lane] = b0;
      bet[2 * lane + 1] = b1;
      dec[2 * lane] = expf(gL - gam0);
      dec[2 * lane + 1] = expf(gL - gam1);
    }
    // state amax (a6), warp partials
    {
      float m = 0.f;
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(hreg[nt][e]));
      m = warp_max(m);
      if (lane == 0) red[0][warp] = m;
    }
    __syncthreads();

    // ---- a2 (+ QK^T for a8): A = strict-lower(beta_i Gamma_ij KK^T), P = lower-incl(Gamma QK^T) ----
    if (cq <= rt) {
      float akk[2][4], aqk[2][4];
      zero_acc(akk);
      zero_acc(aqk);
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        uint32_t ak[4], aq[4], b[4];
        ldsm_x4(ak, a_frag_addr<DK>(Ks, row0, ks * 16, lane));
        ldsm_x4(aq, a_frag_addr<DK>(Qs, row0, ks * 16, lane));
        ldsm_x4(b, bnk_frag_addr<DK>(Ks, col0, ks * 16, lane));
        mma_bf16(akk[0], ak, b[0], b[1]);
        mma_bf16(akk[1], ak, b[2], b[3]);
        mma_bf16(aqk[0], aq, b[0], b[1]);
        mma_bf16(aqk[1], aq, b[2], b[3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = row0 + gq + 8 * e2;
          const int j = col0 + nt * 8 + 2 * tq;
          const float gi = gam[i];
          const float x0 = (j <= i) ? expf(gi - gam[j]) : 0.f;
          const float x1 = (j + 1 <= i) ? expf(gi - gam[j + 1]) : 0.f;
          const float bi = bet[i];
          *reinterpret_cast<float2*>(As + i * kSA + j) =
              make_float2((j < i) ? bi * x0 * akk[nt][2 * e2] : 0.f,
                          (j + 1 < i) ? bi * x1 * akk[nt][2 * e2 + 1] : 0.f);
          const float p0 = x0 * aqk[nt][2 * e2], p1 = x1 * aqk[nt][2 * e2 + 1];
          float h0v, l0v, h1v, l1v;
          split_bf16(p0, h0v, l0v);
          split_bf16(p1, h1v, l1v);
          st_bf16x2(PH + swz<64>(i, j), h0v, h1v);
          st_bf16x2(PL + swz<64>(i, j), l0v, l1v);
        }
    }

    // ---- a6: state QDQ (every thread holds a piece of the state tile) ----
    float sH = 1.f;
    {
      float amax = red[0][0];
#pragma unroll
      for (int i = 1; i < kWarps; ++i) amax = fmaxf(amax, red[0][i]);
      if constexpr (SM != GDN_QDQ_NONE) {
        float rcp;
        qdq_scale<SM>(amax, sH, rcp);
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int d = h_row0 + gq + 8 * e2, col = h_col0 + nt * 8 + 2 * tq;
            float* hv = &hreg[nt][2 * e2];
            uint8_t c0, c1;
            float v0, v1;
            if (amax == 0.f) {
              c0 = qdq_zero_code<SM>(hv[0]);
              c1 = qdq_zero_code<SM>(hv[1]);
              v0 = 0.f;
              v1 = 0.f;
            } else {
              c0 = qdq_code<SM>(hv[0], rcp);
              c1 = qdq_code<SM>(hv[1], rcp);
              v0 = qdq_code_value<SM>(c0);
              v1 = qdq_code_value<SM>(c1);
              hv[0] = __fmul_rn(v0, sH);
              hv[1] = __fmul_rn(v1, sH);
            }
            st_bf16x2(HcH + swz<64>(d, col), v0, v1);
            *reinterpret_cast<uint16_t*>(Hstage + d * 64 + col) = (uint16_t)(c0 | (c1 << 8));
          }
        if (amax == 0.f) sH = 0.f;
      } else {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int d = h_row0 + gq + 8 * e2, col = h_col0 + nt * 8 + 2 * tq;
            float hi0, lo0, hi1, lo1;
            split_bf16(hreg[nt][2 * e2], hi0, lo0);
            split_bf16(hreg[nt][2 * e2 + 1], hi1, lo1);
            st_bf16x2(HcH + swz<64>(d, col), hi0, hi1);
            st_bf16x2(HcL + swz<64>(d, col), lo0, lo1);
            if (p.h_full) {
              float* dst = p.h_full + ((slot * p.Hv + h) * DK + d) * p.Dv + vb * 64 + col;
              *reinterpret_cast<float2*>(dst) = make_float2(hreg[nt][2 * e2], hreg[nt][2 * e2 + 1]);
            }
          }
      }
    }

    __syncthreads();  // A, P, H codes complete

    // saved context: state codes (coalesced 16-byte rows) and scale
    if constexpr (SM != GDN_QDQ_NONE) {
      if (p.h_codes) {
        for (int i = threadIdx.x; i < DK * 4; i += kThreads) {
          const int d = i >> 2, c16 = i & 3;
          const uint4 val = *reinterpret_cast<const uint4*>(Hstage + d * 64 + c16 * 16);
          *reinterpret_cast<uint4*>(p.h_codes + ((slot * p.Hv + h) * DK + d) * p.Dv + vb * 64 +
                                    c16 * 16) = val;
        }
        if (threadIdx.x == 0) p.h_scales[(slot * p.Hv + h) * (p.Dv / 64) + vb] = sH;
      }
    }

    // ---- a3: T = (I + A)^-1 ----
    solve_unit_lower64<kThreads>(As, Ts);

    // ---- a4 operands: Tw = T diag(beta e^gamma), Tu = T diag(beta), split hi/lo ----
    for (int e = threadIdx.x; e < 64 * 32; e += kThreads) {
      const int i = e >> 5, j = (e & 31) * 2;
      const float2 tt = *reinterpret_cast<const float2*>(Ts + i * kSA + j);
      const float t0 = (j <= i) ? tt.x : 0.f;
      const float t1 = (j + 1 <= i) ? tt.y : 0.f;
      float a0, a1, b0, b1;
      split_bf16(t0 * beg[j], a0, b0);
      split_bf16(t1 * beg[j + 1], a1, b1);
      st_bf16x2(TwH + swz<64>(i, j), a0, a1);
      st_bf16x2(TwL + swz<64>(i, j), b0, b1);
      split_bf16(t0 * bet[j], a0, b0);
      split_bf16(t1 * bet[j + 1], a1, b1);
      st_bf16x2(TuH + swz<64>(i, j), a0, a1);
      st_bf16x2(TuL + swz<64>(i, j), b0, b1);
    }
    __syncthreads();

    // ---- a4: W = Tw K  [64 x DK] and U = Tu V  [64 x 64] (hi and lo passes) ----
    float wacc[NTW][4];
    zero_acc(wacc);
    float uacc[2][4];
    zero_acc(uacc);
    wgemm<NTW, false, true, 64, DK>(wacc, TwH, row0, Ks, wcol0, 0, 64, lane);
    wgemm<2, false, true, 64, 64>(uacc, TuH, row0, Vs, col0, 0, 64, lane);
    wgemm<NTW, false, true, 64, DK>(wacc, TwL, row0, Ks, wcol0, 0, 64, lane);
    wgemm<2, false, true, 64, 64>(uacc, TuL, row0, Vs, col0, 0, 64, lane);
    {
      float m = 0.f;
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(wacc[nt][e]));
      m = warp_max(m);
      if (lane == 0) red[1][warp] = m;
    }
    __syncthreads();  // W amax partials; Tw/Tu/V reads done

    // V buffer is free: prefetch the next chunk's V.
    if (c + 1 < nchunks) load_v(p, sm, S::V, ctok + kChunk, min(L - (c + 1) * kChunk, kChunk), h, vb);
    cp_async_commit();

    // ---- a5: W QDQ over the whole [L, DK] tile ----
    float sW = 1.f;
    {
      float amax = red[1][0];
#pragma unroll
      for (int i = 1; i < kWarps; ++i) amax = fmaxf(amax, red[1][i]);
      if constexpr (WM != GDN_QDQ_NONE) {
        float rcp;
        qdq_scale<WM>(amax, sW, rcp);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, col = wcol0 + nt * 8 + 2 * tq;
            uint8_t c0, c1;
            float v0, v1;
            if (amax == 0.f) {
              c0 = qdq_zero_code<WM>(wacc[nt][2 * e2]);
              c1 = qdq_zero_code<WM>(wacc[nt][2 * e2 + 1]);
              v0 = v1 = 0.f;
            } else {
              c0 = qdq_code<WM>(wacc[nt][2 * e2], rcp);
              c1 = qdq_code<WM>(wacc[nt][2 * e2 + 1], rcp);
              v0 = qdq_code_value<WM>(c0);
              v1 = qdq_code_value<WM>(c1);
            }
            st_bf16x2(WcH + swz<DK>(i, col), v0, v1);
            *reinterpret_cast<uint16_t*>(Wstage + i * DK + col) = (uint16_t)(c0 | (c1 << 8));
          }
        if (amax == 0.f) sW = 0.f;
      } else {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, col = wcol0 + nt * 8 + 2 * tq;
            float hi0, lo0, hi1, lo1;
            split_bf16(wacc[nt][2 * e2], hi0, lo0);
            split_bf16(wacc[nt][2 * e2 + 1], hi1, lo1);
            st_bf16x2(WcH + swz<DK>(i, col), hi0, hi1);
            st_bf16x2(WcL + swz<DK>(i, col), lo0, lo1);
          }
      }
    }
    __syncthreads();  // W^ operand complete

    if constexpr (WM != GDN_QDQ_NONE) {
      if (p.w_codes && vb == 0) {
        constexpr int CPR = DK / 16;
        for (int i = threadIdx.x; i < Lc * CPR; i += kThreads) {
          const int r = i / CPR, c16 = i % CPR;
          const uint4 val = *reinterpret_cast<const uint4*>(Wstage + r * DK + c16 * 16);
          *reinterpret_cast<uint4*>(p.w_codes + ((ctok + r) * p.Hv + h) * DK + c16 * 16) = val;
        }
        if (threadIdx.x == 0) p.w_scales[slot * p.Hv + h] = sW;
      }
    }

    // ---- a7: Delta = U - W^ H^ ----
    {
      float dacc[2][4];
      zero_acc(dacc);
      wgemm<2, false, true, DK, 64>(dacc, WcH, row0, HcH, col0, 0, DK, lane);
      if constexpr (WM == GDN_QDQ_NONE) wgemm<2, false, true, DK, 64>(dacc, WcL, row0, HcH, col0, 0, DK, lane);
      if constexpr (SM == GDN_QDQ_NONE) wgemm<2, false, true, DK, 64>(dacc, WcH, row0, HcL, col0, 0, DK, lane);
      const float sWH = (WM != GDN_QDQ_NONE ? sW : 1.f) * (SM != GDN_QDQ_NONE ? sH : 1.f);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
          const float d0 = uacc[nt][2 * e2] - sWH * dacc[nt][2 * e2];
          const float d1 = uacc[nt][2 * e2 + 1] - sWH * dacc[nt][2 * e2 + 1];
          float h0v, l0v, h1v, l1v;
          split_bf16(d0, h0v, l0v);
          split_bf16(d1, h1v, l1v);
          st_bf16x2(DH + swz<64>(i, j), h0v, h1v);
          st_bf16x2(DL + swz<64>(i, j), l0v, l1v);
          const float di = dec[i];
          split_bf16(d0 * di, h0v, l0v);
          split_bf16(d1 * di, h1v, l1v);
          st_bf16x2(DpH + swz<64>(i, j), h0v, h1v);
          st_bf16x2(DpL + swz<64>(i, j), l0v, l1v);
        }
    }
    __syncthreads();  // Delta operands complete

    // ---- a8: O = scale (diag(e^gamma) Q H^ + P Delta) ----
    {
      float o1[2][4], o2[2][4];
      zero_acc(o1);
      zero_acc(o2);
      wgemm<2, false, true, DK, 64>(o1, Qs, row0, HcH, col0, 0, DK, lane);
      if constexpr (SM == GDN_QDQ_NONE) wgemm<2, false, true, DK, 64>(o1, Qs, row0, HcL, col0, 0, DK, lane);
      const int kend = row0 + 16;   // P is lower triangular: columns j <= i only
      wgemm<2, false, true, 64, 64>(o2, PH, row0, DH, col0, 0, kend, lane);
      wgemm<2, false, true, 64, 64>(o2, PH, row0, DL, col0, 0, kend, lane);
      wgemm<2, false, true, 64, 64>(o2, PL, row0, DH, col0, 0, kend, lane);
      const float sq = (SM != GDN_QDQ_NONE) ? sH : 1.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
          const float ei = eg[i] * sq;
          float2 r;
          r.x = p.scale * (ei * o1[nt][2 * e2] + o2[nt][2 * e2]);
          r.y = p.scale * (ei * o1[nt][2 * e2 + 1] + o2[nt][2 * e2 + 1]);
          *reinterpret_cast<float2*>(Ostage + i * OSTR + j) = r;
        }
    }

    // ---- a9: H <- e^{gamma_L} H^ + K^T Delta' ----
    {
      const float egL = eg[63];
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) hreg[nt][e] *= egL;
      wgemm<NTH, true, true, DK, 64>(hreg, Ks, h_row0, DpH, h_col0, 0, 64, lane);
      wgemm<NTH, true, true, DK, 64>(hreg, Ks, h_row0, DpL, h_col0, 0, 64, lane);
    }
    __syncthreads();  // O staged; all reads of K/Q(buf), Delta, P done

    // output rows of this chunk (coalesced 16-byte stores)
    for (int i = threadIdx.x; i < Lc * 16; i += kThreads) {
      const int r = i >> 4, c4 = i & 15;
      const float4 val = *reinterpret_cast<const float4*>(Ostage + r * OSTR + c4 * 4);
      *reinterpret_cast<float4*>(p.o + ((ctok + r) * p.Hv + h) * p.Dv + vb * 64 + c4 * 4) = val;
    }
    // prefetch chunk c + 2 into this buffer
    if (c + 2 < nchunks)
      load_kq<DK>(p, sm, S::K + buf * S::kTileK, S::Q + buf * S::kTileK, S::BG + buf * 512,
                  ctok + 2 * kChunk, min(L - (c + 2) * kChunk, kChunk), hk, h);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // final state (unquantized)
  if (p.ht) {
    float* dst = p.ht + (((int64_t)n * p.Hv + h) * DK) * p.Dv + vb * 64;
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int d = h_row0 + gq + 8 * e2, col = h_col0 + nt * 8 + 2 * tq;
        *reinterpret_cast<float2*>(dst + (int64_t)d * p.Dv + col) =
            make_float2(hreg[nt][2 * e2], hreg[nt][2 * e2 + 1]);
      }
  }
}

template <int DK, int SM, int WM>
gdn_status launch_t(const FwdParams& prm, const Dims& d, cudaStream_t st) {
  using S = Smem<DK, SM, WM>;
  auto kern = gdn_fwd_kernel<DK, SM, WM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  dim3 grid((unsigned)(d.Dv / 64), (unsigned)d.Hv, (unsigned)d.N);
  kern<<<grid, kThreads, S::BYTES, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int DK>
gdn_status dispatch_modes(const gdn_problem& p, const FwdParams& prm, const Dims& d,
                          cudaStream_t st) {
#define GDN_CASE(SMV, WMV) \
  if (p.state_mode == SMV && p.w_mode == WMV) return launch_t<DK, SMV, WMV>(prm, d, st);
  GDN_CASE(GDN_QDQ_E4M3, GDN_QDQ_E4M3)
  GDN_CASE(GDN_QDQ_INT8, GDN_QDQ_E4M3)
  GDN_CASE(GDN_QDQ_NONE, GDN_QDQ_NONE)
  GDN_CASE(GDN_QDQ_E4M3, GDN_QDQ_NONE)
  GDN_CASE(GDN_QDQ_NONE, GDN_QDQ_E4M3)
  GDN_CASE(GDN_QDQ_INT8, GDN_QDQ_NONE)
  GDN_CASE(GDN_QDQ_INT8, GDN_QDQ_INT8)
  GDN_CASE(GDN_QDQ_E4M3, GDN_QDQ_INT8)
  GDN_CASE(GDN_QDQ_NONE, GDN_QDQ_INT8)
#undef GDN_CASE
  return GDN_ERR_UNSUPPORTED_MODE;
}

}  // namespace

gdn_status launch_fwd(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const float* h0,
                      float* o, float* ht, void* ctx, cudaStream_t st) {
  FwdParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.h0 = h0;
  prm.o = o;
  prm.ht = ht;
  if (ctx) {
    const CtxLayout L = ctx_layout(p);
    unsigned char* base = static_cast<unsigned char*>(ctx);
    if (p.w_mode != GDN_QDQ_NONE) {
      prm.w_codes = base + L.w_codes;
      prm.w_scales = reinterpret_cast<float*>(base + L.w_scales);
    }
    if (p.state_mode != GDN_QDQ_NONE) {
      prm.h_codes = base + L.h_codes;
      prm.h_scales = reinterpret_cast<float*>(base + L.h_scales);
    } else {
      prm.h_full = reinterpret_cast<float*>(base + L.h_full);
    }
  }
  prm.cu_seqlens = p.cu_seqlens;
  prm.T = d.T;
  prm.Hk = d.Hk;
  prm.Hv = d.Hv;
  prm.Dv = d.Dv;
  prm.G = d.Hv / d.Hk;
  prm.nt_fixed = d.nt_fixed;
  prm.scale = p.scale;
  if (d.Dk == 128) return dispatch_modes<128>(p, prm, d, st);
  return dispatch_modes<64>(p, prm, d, st);
}

}  // namespace gdn
