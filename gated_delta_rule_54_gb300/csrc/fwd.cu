// Forward of the chunked gated delta rule with state / W fake QDQ.
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
// GB300 design: only H^ -> Delta -> H is a serial dependence between chunks,
// so the forward is three launches.
//   1. gdn_fwd_prep_kernel, one CTA per (chunk, value head), all chunks in
//      parallel: KK^T, the exact solve, W (quantized: codes and scale go to the
//      saved context) and U (fp32, parked in the output buffer o).
//   2. gdn_fwd_state_kernel, one CTA per (sequence, value head, 64-wide value
//      block) walks its chunks in order with the fp32 state tile in registers;
//      per chunk only the state QDQ (codes to the context), Delta = U - W^ H^
//      (stored over U in o) and the state update remain on the serial path,
//      with the next chunk's operands prefetched by TMA on an mbarrier.
//   3. gdn_fwd_output_kernel, one CTA per (chunk, value head), all in
//      parallel: QK^T once, then per value block O from H^ (the saved codes)
//      and Delta (read from o), written over Delta; it also saves P and Delta
//      as bf16 tile images for the backward.
// Contractions run on tensor cores (mma.sync bf16, fp32 accumulation).
// Operands that are not exactly bf16 (T diag(.), Delta, the decayed Delta, P,
// and unquantized W / H) are split into hi + lo bf16 halves so the state path
// keeps ~16 mantissa bits: a plain bf16 rounding of these flips far more
// quantization codes than the fp32 arithmetic of the definition would.
// Quantized W and H enter the tensor cores as their codes (E4M3 values and
// INT8 integers are exact in bf16) with the fp32 scales applied in epilogues.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include <cooperative_groups.h>

#include "common.cuh"
#include "fused.h"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

namespace {

// set by a kernel whose bounded wait for a TMA transfer gave up
__device__ int g_fwd_device_error;

struct FwdParams {
  // TMA descriptors (2-D): k, q [B*T, Hk*Dk] bf16, v [B*T, Hv*Dv] bf16, o/U [B*T, Hv*Dv] f32,
  // W codes [B*T, Hv*Dk] u8 (plain rows, and with the 128-byte swizzle when
  // Dk = 128), state codes [n_slots*Hv*Dk, Dv] u8
  CUtensorMap tm_k, tm_q, tm_v, tm_u, tm_wc, tm_wc_sw, tm_hc;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* beta;
  const float* g;
  const float* h0;
  float* o;  // also holds U between the prep and the output launches
  float* ht;
  uint8_t* w_codes;
  float* w_scales;
  float* w_full;
  uint8_t* h_codes;
  float* h_scales;
  float* h_full;
  float* cvec;  // [n_slots, Hv, kCvecFloats] chunk vectors
  __nv_bfloat16 *tb, *gkk, *pb;  // [n_slots, Hv] 8 KiB tile images for the backward (or null)
  __nv_bfloat16* db;             // [n_slots, Hv, Dv / 64] Delta tile images for the backward (or null)
  __nv_bfloat16* tu_img;         // [n_slots, Hv, 2, 4096] T diag(beta) hi, lo images (fused scan)
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, G, N;
  int block_v;  // state-scale tile width: 16, 32, 64, or 128 (two value blocks)
  int bv_log2;  // log2(block_v)
  int neumann;  // -1: exact solve; d >= 0: Neumann polynomial of degree d
  int64_t nt_fixed;
  int64_t n_slots;  // chunk slots of the call
  float scale;
};

// x[i] of a short register array without a local-memory copy (i < N)
template <int N>
__device__ __forceinline__ float pick(const float (&x)[N], int i) {
  float r = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) r = (i == j) ? x[j] : r;
  return r;
}

// The chunk stored at a chunk slot (see gdn_qdq.h); false for an unused
// packed slot.  Uniform across a CTA.
struct ChunkRef {
  int64_t tok;  // first token
  int L;        // valid rows (1..64)
};

__device__ __forceinline__ bool chunk_of_slot(const FwdParams& p, int64_t slot, ChunkRef& r) {
  if (!p.cu_seqlens) {
    const int64_t n = slot / p.nt_fixed, c = slot % p.nt_fixed;
    r.tok = n * p.T + c * kChunk;
    r.L = (int)min((int64_t)kChunk, p.T - c * kChunk);
    return r.L > 0;
  }
  // largest n with floor(cu[n] / 64) + n <= slot (strictly increasing in n)
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)p.cu_seqlens[mid] / kChunk + mid <= slot)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int64_t a = p.cu_seqlens[lo], b = p.cu_seqlens[lo + 1];
  const int64_t c = slot - (a / kChunk + lo);
  if (c < 0 || c * kChunk >= b - a) return false;
  r.tok = a + c * kChunk;
  r.L = (int)min((int64_t)kChunk, b - a - c * kChunk);
  return true;
}

// [64][DK] bf16 rows of q or k of one chunk (rows >= L zero-filled), swizzled.
template <int DK, int NTHREADS>
__device__ __forceinline__ void load_rows_bf16(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                               int64_t tok0, int L, int H, int hh) {
  constexpr int CPR = DK / 8;
  for (int i = threadIdx.x; i < kChunk * CPR; i += NTHREADS) {
    const int r = i / CPR, c = i % CPR;
    const bool ok = r < L;
    const int64_t tok = tok0 + (ok ? r : 0);
    cp_async16(smem_u32(dst + swz<DK>(r, c * 8)), src + (tok * H + hh) * DK + c * 8, ok ? 16 : 0);
  }
}

// 64 floats of beta or g of one chunk (rows >= L zero-filled).
__device__ __forceinline__ void load_vec64(float* dst, const float* src, int64_t tok0, int L,
                                           int Hv, int h, int t) {
  const bool ok = t < L;
  const int64_t tok = tok0 + (ok ? t : 0);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst + t)),
               "l"(src + tok * Hv + h), "r"(ok ? 4 : 0));
}

// gamma = in-chunk cumsum of g (padded rows have g = 0, so gamma stays at the
// last valid value there).  Warp-wide; lane l owns rows 2l, 2l+1.
__device__ __forceinline__ void chunk_cumsum(const float* g, int lane, float& gam0, float& gam1,
                                             float& gL) {
  const float g0 = g[2 * lane], g1 = g[2 * lane + 1];
  float s = g0 + g1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += y;
  }
  gam1 = s;
  gam0 = s - g1;
  gL = __shfl_sync(0xffffffffu, s, 31);
}

// T = sum_{i<=degree} X^i with X = -A ("[7/7] Experimental GDN/KDA
// approximate-inverse QAT", "What does this PR do?": the Neumann polynomial of
// an explicit degree, in fp32), by Horner's rule T <- I + X T from T = I.  A is
// the strictly lower fp32 [64][kSA] tile (zero elsewhere); T ping-pongs between
// Tmp and Ts and ends in Ts.  256 threads, each a 4 x 4 block of the product.
__device__ __forceinline__ void neumann_lower64(const float* As, float* Ts, float* Tmp, int degree) {
  const int tid = threadIdx.x;
  const int r0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
  float* cur = (degree % 2 == 0) ? Ts : Tmp;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(cur + (r0 + i) * kSA + c0) =
        make_float4(r0 + i == c0 ? 1.f : 0.f, r0 + i == c0 + 1 ? 1.f : 0.f,
                    r0 + i == c0 + 2 ? 1.f : 0.f, r0 + i == c0 + 3 ? 1.f : 0.f);
  __syncthreads();
  for (int step = 0; step < degree; ++step) {
    float* nxt = (cur == Ts) ? Tmp : Ts;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int k = 0; k < 64; ++k) {
      const float4 b = *reinterpret_cast<const float4*>(cur + k * kSA + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = -As[(r0 + i) * kSA + k];
        acc[i].x = fmaf(a, b.x, acc[i].x);
        acc[i].y = fmaf(a, b.y, acc[i].y);
        acc[i].z = fmaf(a, b.z, acc[i].z);
        acc[i].w = fmaf(a, b.w, acc[i].w);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + i;
      *reinterpret_cast<float4*>(nxt + r * kSA + c0) =
          make_float4(acc[i].x + (r == c0 ? 1.f : 0.f), acc[i].y + (r == c0 + 1 ? 1.f : 0.f),
                      acc[i].z + (r == c0 + 2 ? 1.f : 0.f), acc[i].w + (r == c0 + 3 ? 1.f : 0.f));
    }
    __syncthreads();
    cur = nxt;
  }
}

// ===========================================================================
// 1. Chunk-local prep: A, T, W (+ QDQ), U.
// ===========================================================================
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

template <int DK>
struct PrepSmem {
  static constexpr int K = 0;                            // bf16 [64][DK] (TMA)
  static constexpr int V = K + kChunk * DK * 2;          // bf16 Dv/64 x [64][64] (TMA)
  static constexpr int A = V + 2 * kChunk * 64 * 2;      // f32 [64][kSA]; later U staging (swz_f32)
  static constexpr int TT = A + kF32Tile;                // f32 [64][kSA]
  static constexpr int TW = TT + kF32Tile;               // Tw hi, lo
  static constexpr int TU = TW + 2 * kChunk * 64 * 2;    // Tu hi, lo
  static constexpr int WST = TU + 2 * kChunk * 64 * 2;   // u8 [64][DK] W codes
  static constexpr int BG = WST + kChunk * DK;           // beta[64], g[64]
  static constexpr int VEC = BG + 512;                   // gamma, e^gamma, beta e^gamma, beta
  static constexpr int BYTES = VEC + 4 * 64 * 4 + 1024;  // + alignment slack
  static_assert((V % 1024) == 0 && (A % 1024) == 0 && (TW % 128) == 0 && (WST % 128) == 0,
                "alignment");
  static_assert(WST - TW >= kF32Tile, "Tw, Tu hold a second fp32 tile for the Neumann products");
};

// Layout of the variant for the fused scan (exact solve, no V and no U): the
// W operand halves reuse A once the solve is done and the W code staging
// reuses T once T diag(.) is split, so three CTAs fit on an SM.
template <int DK>
struct PrepSmemT {
  static constexpr int K = 0;                            // bf16 [64][DK] (TMA)
  static constexpr int A = K + kChunk * DK * 2;          // f32 [64][kSA]; then Tw hi, lo
  static constexpr int TT = A + kF32Tile;                // f32 [64][kSA]; then W codes
  static constexpr int TU = TT + kF32Tile;               // Tu hi, lo (the images written out)
  static constexpr int TW = A;
  static constexpr int WST = TT;
  static constexpr int V = K;                            // (no V)
  static constexpr int BG = TU + 2 * kChunk * 64 * 2;    // beta[64], g[64]
  static constexpr int VEC = BG + 512;                   // gamma, e^gamma, beta e^gamma, beta
  static constexpr int BYTES = VEC + 4 * 64 * 4 + 1024;  // + alignment slack
  static_assert((A % 1024) == 0 && (TT % 1024) == 0 && (TU % 1024) == 0, "alignment");
  static_assert(2 * kChunk * 64 * 2 <= kF32Tile && kChunk * DK <= kF32Tile, "aliases fit");
  static_assert(3 * (BYTES + 2048) <= 233472, "three CTAs per SM");
};

// TOUT: the variant for the fused scan, which forms U itself: T diag(beta),
// split into hi and lo bf16 halves, is written as two tile images to
// p.tu_img, and U is not computed.
template <int DK, int WM, bool TOUT>
__global__ void __launch_bounds__(kPrepThreads, TOUT ? 3 : 2) gdn_fwd_prep_kernel(const __grid_constant__ FwdParams p) {
  using S = typename std::conditional<TOUT, PrepSmemT<DK>, PrepSmem<DK>>::type;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ float red[kPrepWarps];
  __shared__ __align__(8) uint64_t bar;
  // the fused path's variant runs K K^T and W = Tw K on tcgen05 (accumulators
  // in 128 TMEM columns, three CTAs per SM share the 512)
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ int tc_failed;

  // The fused path's variant is persistent: CTA b takes the chunk-heads b,
  // b + grid, ... and loads the next one's K, beta and g while it finishes the
  // current one (K is free once W = Tw K has run).  The other variant has one
  // CTA per chunk-head.
  const int64_t units = p.n_slots * p.Hv;
  // the fused scan that follows may take the SMs this CTA leaves (it waits for
  // the whole grid before reading any output of it)
  if constexpr (TOUT) grid_dep_launch();
  // the next chunk-head at or after u that holds tokens (units if none)
  auto next_unit = [&](int64_t u, ChunkRef& r) {
    for (; u < units; u += gridDim.x)
      if (chunk_of_slot(p, u / p.Hv, r)) return u;
    return units;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int nvb = p.Dv / 64;

  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm + S::K);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(sm + S::V);
  float* bsrc = reinterpret_cast<float*>(sm + S::BG);
  float* gam = reinterpret_cast<float*>(sm + S::VEC);
  float* eg = gam + 64;
  float* beg = gam + 128;
  float* bet = gam + 192;
  float* As = reinterpret_cast<float*>(sm + S::A);
  float* Ts = reinterpret_cast<float*>(sm + S::TT);
  __nv_bfloat16* TwH = reinterpret_cast<__nv_bfloat16*>(sm + S::TW);
  __nv_bfloat16* TwL = TwH + kChunk * 64;
  __nv_bfloat16* TuH = reinterpret_cast<__nv_bfloat16*>(sm + S::TU);
  __nv_bfloat16* TuL = TuH + kChunk * 64;
  uint8_t* Wst = sm + S::WST;
  float* Ust = As;

  // K and V as TMA boxes (rows >= L hold another sequence's tokens: they only
  // meet zero beta, so they reach neither A, W nor U); beta and g zero-filled
  auto issue_loads = [&](int64_t u, const ChunkRef& r) {
    const int hh = (int)(u % p.Hv);
    if (threadIdx.x == 0) {
      mbar_expect_tx(&bar, kChunk * DK * 2 + (TOUT ? 0 : nvb * kChunk * 64 * 2));
#pragma unroll
      for (int pn = 0; pn < DK / 64; ++pn)
        tma_load_2d(Ks + pn * kChunk * 64, &p.tm_k, (hh / p.G) * DK + pn * 64, (int)r.tok, &bar);
      for (int vb = 0; vb < (TOUT ? 0 : nvb); ++vb)
        tma_load_2d(Vs + vb * kChunk * 64, &p.tm_v, hh * p.Dv + vb * 64, (int)r.tok, &bar);
    }
    if (threadIdx.x < 2 * kChunk) {
      const int t = threadIdx.x & 63;
      load_vec64(bsrc + (threadIdx.x < kChunk ? 0 : 64), threadIdx.x < kChunk ? p.beta : p.g,
                 r.tok, r.L, p.Hv, hh, t);
    }
    cp_async_commit();
  };
  ChunkRef cr;
  int64_t u = next_unit(blockIdx.x, cr);
  if (u >= units) return;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();  // the mbarrier is initialised before the first copy signals it
  issue_loads(u, cr);
  if constexpr (TOUT) {
    if (warp == 0) tmem_alloc(&tmem_slot, 128);
    if (threadIdx.x == 0) {
      mbar_init(&bar_mma, 1);
      tc_failed = 0;
      fence_mbar_init();
    }
    tc_fence_before();
  }
  __syncthreads();  // the MMA barrier and the TMEM columns are set up
  uint32_t ld_phase = 0;
  for (; u < units;) {
  const int64_t slot = u / p.Hv;
  const int h = (int)(u % p.Hv);
  const int hk = h / p.G;
  const int L = cr.L;
  const int64_t tok0 = cr.tok;
  int64_t nu = units;  // the next chunk-head of this CTA
  ChunkRef ncr{};
  {
    const bool ok = mbar_wait(&bar, ld_phase);
    cp_async_wait<0>();
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        atomicOr(&g_fwd_device_error, 1);
        mbar_wait(&bar, ld_phase);  // once more, bounded, for the copies in flight
      }
      break;
    }
    ld_phase ^= 1u;
  }

  if (warp == 0) {
    float gam0, gam1, gL;
    chunk_cumsum(bsrc + 64, lane, gam0, gam1, gL);
    const float b0 = bsrc[2 * lane], b1 = bsrc[2 * lane + 1];
    const float e0 = expf(gam0), e1 = expf(gam1);
    gam[2 * lane] = gam0;
    gam[2 * lane + 1] = gam1;
    eg[2 * lane] = e0;
    eg[2 * lane + 1] = e1;
    beg[2 * lane] = b0 * e0;
    beg[2 * lane + 1] = b1 * e1;
    bet[2 * lane] = b0;
    bet[2 * lane + 1] = b1;
    // the chunk vectors the state scan, the output pass and the backward read
    float* cv = p.cvec + (slot * p.Hv + h) * kCvecFloats;
    *reinterpret_cast<float2*>(cv + kCvGam + 2 * lane) = make_float2(gam0, gam1);
    *reinterpret_cast<float2*>(cv + kCvEg + 2 * lane) = make_float2(e0, e1);
    *reinterpret_cast<float2*>(cv + kCvDec + 2 * lane) = make_float2(expf(gL - gam0), expf(gL - gam1));
    *reinterpret_cast<float2*>(cv + kCvBet + 2 * lane) = make_float2(b0, b1);
    *reinterpret_cast<float2*>(cv + kCvBeg + 2 * lane) = make_float2(b0 * e0, b1 * e1);
  }

  // warp tile: rows 16 rt .. +15, columns 32 ch .. +31 of a [64 x 64] product
  const int rt = warp & 3, ch = warp >> 2;
  const int row0 = rt * 16, col0 = ch * 32;

  // ---- a2: A = strict-lower(beta_i Gamma_ij k_i.k_j) (blocks above the diagonal skipped);
  //      KK^T needs no gamma, so it runs before the barrier that publishes gamma ----
  const bool a_tile = col0 <= row0 + 15;
  float acc[4][4];
  zero_acc(acc);
  uint32_t tmem = 0;
  if constexpr (TOUT) {
    // K K^T: M = 64, N = 64, K = DK (K-major panels), one commit; issued from
    // warp 1 so that it starts while warp 0 forms gamma
    tc_fence_after();
    tmem = tmem_slot;
    if (threadIdx.x == 32) {
      const uint64_t kd = sdesc(smem_u32(Ks), 16, 1024);
      constexpr uint32_t id = idesc(64, 64, 0, 0);
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks)
        umma(tmem, dadd(kd, (ks >> 2) * 8192 + (ks & 3) * 32), dadd(kd, (ks >> 2) * 8192 + (ks & 3) * 32),
             id, ks > 0);
      umma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 0)) tc_failed = 1;
    tc_fence_after();
    tmem_ld_frag<4>(tmem + ((uint32_t)(32 * rt) << 16) + col0, acc);
  } else {
    if (a_tile) wgemm<4, false, false, DK, DK>(acc, Ks, row0, Ks, col0, 0, DK, lane);
  }
  __syncthreads();
  {
    // Gamma o KK^T (strictly lower; rows >= L hold another sequence's keys: zero)
    // as the backward's tile image, and A = diag(beta) (Gamma o KK^T)
    __nv_bfloat16* gimg = p.gkk ? p.gkk + (slot * p.Hv + h) * (kTileImgBytes / 2) : nullptr;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
        float k0 = 0.f, k1 = 0.f;
        if (a_tile && i < L) {
          // e^{gamma_i - gamma_j} as 2^{(gamma_i - gamma_j) log2 e} by the hardware exp2
          // (about 2^-22 relative; the argument's rounding grows with the decay but the
          // factor then shrinks as fast, so the absolute error of A stays ~1e-7)
          const float gi = gam[i] * kLog2eF;
          k0 = (j < i) ? ex2_approx_f(gi - gam[j] * kLog2eF) * acc[nt][2 * e2] : 0.f;
          k1 = (j + 1 < i) ? ex2_approx_f(gi - gam[j + 1] * kLog2eF) * acc[nt][2 * e2 + 1] : 0.f;
        }
        if (gimg) st_bf16x2(gimg + swz<64>(i, j), k0, k1);
        // (tiles above the diagonal hold zeros: the Neumann products read all of A)
        *reinterpret_cast<float2*>(As + i * kSA + j) = make_float2(bet[i] * k0, bet[i] * k1);
      }
  }
  // the previous chunk-head's W-code and Tu image stores have read T and Tu
  if (threadIdx.x == 0) tma_store_wait_read();
  __syncthreads();

  // ---- a3: T = (I + A)^-1, or its Neumann polynomial ----
  if (TOUT || p.neumann < 0)
    solve_unit_lower64<kPrepThreads>(As, Ts);
  else if constexpr (!TOUT)
    neumann_lower64(As, Ts, reinterpret_cast<float*>(sm + S::TW), p.neumann);

  // ---- a4 operands: Tw = T diag(beta e^gamma), Tu = T diag(beta), split hi/lo;
  //      T itself as the backward's tile image ----
  __nv_bfloat16* timg = p.tb ? p.tb + (slot * p.Hv + h) * (kTileImgBytes / 2) : nullptr;
  // a thread keeps its column pair j, j + 1 (the row advances by 8 per pass):
  // its diagonal factors are read once
  static_assert(kPrepThreads % 32 == 0, "column pair fixed per thread");
  const int jc = (threadIdx.x & 31) * 2;
  const float bw0 = beg[jc], bw1 = beg[jc + 1], bu0 = bet[jc], bu1 = bet[jc + 1];
  for (int e = threadIdx.x; e < 64 * 32; e += kPrepThreads) {
    const int i = e >> 5, j = jc;
    const float2 tt = *reinterpret_cast<const float2*>(Ts + i * kSA + j);
    const float t0 = (j <= i) ? tt.x : 0.f;
    const float t1 = (j + 1 <= i) ? tt.y : 0.f;
    if (timg) st_bf16x2(timg + swz<64>(i, j), t0, t1);
    float a0, a1, b0, b1;
    split_bf16(t0 * bw0, a0, b0);
    split_bf16(t1 * bw1, a1, b1);
    st_bf16x2(TwH + swz<64>(i, j), a0, a1);
    st_bf16x2(TwL + swz<64>(i, j), b0, b1);
    split_bf16(t0 * bu0, a0, b0);
    split_bf16(t1 * bu1, a1, b1);
    st_bf16x2(TuH + swz<64>(i, j), a0, a1);
    st_bf16x2(TuL + swz<64>(i, j), b0, b1);
  }
  __syncthreads();

  // ---- a4: W = Tw K [64 x DK] (warp: 16 rows x DK/2 columns), hi and lo passes ----
  constexpr int NTW = DK / 16;
  const int wc0 = ch * (DK / 2);
  float wacc[NTW][4];
  zero_acc(wacc);
  if constexpr (TOUT) {
    // W = Tw_hi K + Tw_lo K: M = 64, N = DK, K = 64 (K read MN-major)
    static_assert(!TOUT || DK == 128, "the tensor-core prep is for Dk = 128");
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
      bulk_store_1d(p.tu_img + (slot * p.Hv + h) * (2 * kChunk * kChunk), TuH,
                    2 * kChunk * kChunk * 2);
      tma_store_commit();
      const uint64_t kd = sdesc(smem_u32(Ks), 8192, 1024);
      const uint64_t th = sdesc(smem_u32(TwH), 16, 1024), tl = sdesc(smem_u32(TwL), 16, 1024);
      constexpr uint32_t id = idesc(64, DK, 0, 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) umma(tmem, dadd(th, ks * 32), dadd(kd, ks * 2048), id, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) umma(tmem, dadd(tl, ks * 32), dadd(kd, ks * 2048), id, true);
      umma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 1)) tc_failed = 1;
    tc_fence_after();
    // K and beta, g are free: the next chunk-head's arrive during the rest of this one
    nu = next_unit(u + gridDim.x, ncr);
    if (nu < units) issue_loads(nu, ncr);
    const uint32_t tw = tmem + ((uint32_t)(32 * rt) << 16) + wc0;
    tmem_ld_frag_pair<4>(tw, *reinterpret_cast<float(*)[4][4]>(&wacc[0][0]), tw + 32,
                         *reinterpret_cast<float(*)[4][4]>(&wacc[4][0]));
  } else {
    wgemm_shared_b<NTW, false, true, 64, DK>(wacc, wacc, TwH, TwL, row0, Ks, wc0, 0, 64, lane);
  }

  // ---- a5: W QDQ over the whole [L, DK] tile ----
  if constexpr (WM != GDN_QDQ_NONE) {
    // Dk = 128: the codes are staged with the 128-byte swizzle (16-byte chunk
    // c of row i at c ^ (i % 8)), so a warp's eight rows fall in distinct banks,
    // and leave through the swizzled tensor map
    constexpr bool WSW = DK == 128;
    static_assert(!WSW || (S::WST % 1024) == 0, "swizzled W-code staging is 1024-byte aligned");
    auto wst_off = [&](int i, int col) {
      return WSW ? i * DK + (((col >> 4) ^ (i & 7)) << 4) + (col & 15) : i * DK + col;
    };
    float m = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(wacc[nt][e]));
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kPrepWarps; ++i) amax = fmaxf(amax, red[i]);
    float sW, rcp;
    qdq_scale<WM>(amax, sW, rcp);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, col = wc0 + nt * 8 + 2 * tq;
        uint16_t c2;
        if constexpr (WM == GDN_QDQ_E4M3) {
          // rcp == 0 (amax 0, or no usable scale) gives signed-zero codes
          float2 val;
          c2 = e4m3_code2(wacc[nt][2 * e2], wacc[nt][2 * e2 + 1], rcp, val);
        } else {
          uint8_t c0, c1;
          if (amax == 0.f) {
            c0 = qdq_zero_code<WM>(wacc[nt][2 * e2]);
            c1 = qdq_zero_code<WM>(wacc[nt][2 * e2 + 1]);
          } else {
            c0 = qdq_code<WM>(wacc[nt][2 * e2], rcp);
            c1 = qdq_code<WM>(wacc[nt][2 * e2 + 1], rcp);
          }
          c2 = (uint16_t)(c0 | (c1 << 8));
        }
        *reinterpret_cast<uint16_t*>(Wst + wst_off(i, col)) = c2;
      }
    if (L == kChunk) {
      fence_proxy_async();
      __syncthreads();
      if (threadIdx.x == 0) {
        tma_store_2d(WSW ? &p.tm_wc_sw : &p.tm_wc, h * DK, (int)tok0, Wst);
        tma_store_commit();
      }
    } else {
      __syncthreads();
      constexpr int CPR = DK / 16;
      for (int i = threadIdx.x; i < L * CPR; i += kPrepThreads) {
        const int r = i / CPR, c16 = i % CPR;
        *reinterpret_cast<uint4*>(p.w_codes + ((tok0 + r) * p.Hv + h) * DK + c16 * 16) =
            *reinterpret_cast<const uint4*>(Wst + wst_off(r, c16 * 16));
      }
    }
    if (threadIdx.x == 0) p.w_scales[slot * p.Hv + h] = sW;
  } else {
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, col = wc0 + nt * 8 + 2 * tq;
        if (i < L)
          *reinterpret_cast<float2*>(p.w_full + ((tok0 + i) * p.Hv + h) * DK + col) =
              make_float2(wacc[nt][2 * e2], wacc[nt][2 * e2 + 1]);
      }
  }

  // ---- a4: U = Tu V, one 64-column block at a time, parked in o ----
  for (int vb = 0; vb < (TOUT ? 0 : nvb); ++vb) {
    float uacc[4][4];
    zero_acc(uacc);
    const __nv_bfloat16* Vb = Vs + vb * kChunk * 64;
    wgemm_shared_b<4, false, true, 64, 64>(uacc, uacc, TuH, TuL, row0, Vb, col0, 0, 64, lane);
    if (vb > 0 && threadIdx.x == 0) tma_store_wait_read();  // previous block's U has left
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
        *reinterpret_cast<float2*>(Ust + swz_f32(i, j)) =
            make_float2(uacc[nt][2 * e2], uacc[nt][2 * e2 + 1]);
      }
    if (L == kChunk) {
      fence_proxy_async();
      __syncthreads();
      if (threadIdx.x == 0) {
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_store_2d(&p.tm_u, h * p.Dv + vb * 64 + pn * 32, (int)tok0, Ust + pn * kChunk * 32);
        tma_store_commit();
      }
    } else {
      __syncthreads();
      for (int i = threadIdx.x; i < L * 16; i += kPrepThreads) {
        const int r = i >> 4, c4 = i & 15;
        *reinterpret_cast<float4*>(p.o + ((tok0 + r) * p.Hv + h) * p.Dv + vb * 64 + c4 * 4) =
            *reinterpret_cast<const float4*>(Ust + swz_f32(r, c4 * 4));
      }
    }
  }
  if constexpr (TOUT) {
    tc_fence_before();  // this chunk-head's TMEM reads precede the next one's products
  } else {
    nu = next_unit(u + gridDim.x, ncr);  // (none: one CTA per chunk-head)
    if (nu < units) {
      __syncthreads();  // K and V have been read
      issue_loads(nu, ncr);
    }
  }
  u = nu;
  cr = ncr;
  }  // chunk-heads of this CTA

  if (threadIdx.x == 0) tma_store_wait_all();
  if constexpr (TOUT) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && tc_failed) {
      atomicOr(&g_fwd_device_error, 1);
      mbar_wait(&bar_mma, 1);  // once more, bounded, for the products in flight
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_slot, 128);
  }
}

// ===========================================================================
// 2. Serial state scan: H^ = Q_S(H), Delta = U - W^ H^, H <- e^{gL} H^ + K~^T Delta.
// ===========================================================================
constexpr int kStateThreads = 512;
constexpr int kStateWarps = kStateThreads / 32;

template <int DK, int SM, int WM>
struct StateSmem {
  static constexpr int WRAW = (WM == GDN_QDQ_NONE) ? kChunk * DK * 4 : kChunk * DK;
  static constexpr int K = 0;                                          // 2 x bf16 [64][DK] (TMA)
  static constexpr int U = K + 2 * kChunk * DK * 2;                    // 2 x f32 [64][64] (TMA, swz_f32)
  static constexpr int WR = U + 2 * kChunk * 64 * 4;                   // 2 x W codes (TMA) / f32
  static constexpr int CV = WR + 2 * WRAW;                             // 2 x chunk vectors (bulk copy)
  static constexpr int WC = CV + 2 * kCvecFloats * 4;                  // W^ bf16 [64][DK] (hi, lo)
  static constexpr int HC = WC + (WM == GDN_QDQ_NONE ? 2 : 1) * kChunk * DK * 2;  // H^ [DK][64]
  static constexpr int DP = HC + (SM == GDN_QDQ_NONE ? 2 : 1) * DK * 64 * 2;      // Delta' hi, lo
  static constexpr int HST = DP + 2 * kChunk * 64 * 2;                 // u8 [DK][64] codes (TMA store)
  static constexpr int BYTES = HST + DK * 64 + 1024;                   // + alignment slack
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert((U % 1024) == 0 && (WR % 1024) == 0 && (WC % 128) == 0 && (HC % 128) == 0 &&
                    (DP % 128) == 0 && (HST % 128) == 0,
                "alignment");
};

// TMA boxes of one chunk: K (two 64-column panels), U (two 32-column fp32
// panels), the chunk vectors and, for quantized W, its codes (an fp32 W by
// cp.async).
template <int DK, int WM>
__device__ __forceinline__ uint32_t state_chunk_tx_bytes() {
  return kChunk * DK * 2 + kChunk * 64 * 4 + kCvecFloats * 4 +
         (WM != GDN_QDQ_NONE ? kChunk * DK : 0);
}

template <int DK, int WM, bool F8>
__device__ __forceinline__ void issue_state_chunk(const FwdParams& p, __nv_bfloat16* Ks,
                                                  unsigned char* Wr, float* Us, float* Cv,
                                                  uint64_t* bar, int64_t tok0, int L, int hk,
                                                  int h, int vb, int64_t slot) {
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, state_chunk_tx_bytes<DK, WM>());
    bulk_load_1d(Cv, p.cvec + (slot * p.Hv + h) * kCvecFloats, kCvecFloats * 4, bar);
#pragma unroll
    for (int pn = 0; pn < DK / 64; ++pn)
      tma_load_2d(Ks + pn * kChunk * 64, &p.tm_k, hk * DK + pn * 64, (int)tok0, bar);
#pragma unroll
    for (int pn = 0; pn < 2; ++pn)
      tma_load_2d(Us + pn * kChunk * 32, &p.tm_u, h * p.Dv + vb * 64 + pn * 32, (int)tok0, bar);
    if constexpr (WM != GDN_QDQ_NONE)
      tma_load_2d(Wr, F8 ? &p.tm_wc_sw : &p.tm_wc, h * DK, (int)tok0, bar);
  }
  if constexpr (WM == GDN_QDQ_NONE) {
    constexpr int CPR = DK / 4;
    for (int i = threadIdx.x; i < kChunk * CPR; i += kStateThreads) {
      const int r = i / CPR, c = i % CPR;
      const bool ok = r < L;
      const int64_t tok = tok0 + (ok ? r : 0);
      cp_async16(smem_u32(Wr + (r * DK + c * 4) * 4), p.w_full + (tok * p.Hv + h) * DK + c * 4,
                 ok ? 16 : 0);
    }
  }
  cp_async_commit();
}

// BV is the state-scale tile width: 16 or 32 (two or four tiles in the 64-column
// block), 64 (the block), or 128 (two blocks: the pair of CTAs is a cluster
// that swaps its block amax every chunk).  The tile bookkeeping is resolved at
// compile time, so the common one-tile case carries none of it.
template <int DK, int SM, int WM, int BV>
__global__ void __launch_bounds__(kStateThreads, 1) gdn_fwd_state_kernel(const __grid_constant__ FwdParams p) {
  using S = StateSmem<DK, SM, WM>;
  // E4M3 W and state at Dk = 128: Delta = W^ H^ runs on E4M3 codes directly
  // (W codes as TMA wrote them, H^ codes written [v][dk] as the B operand)
  constexpr bool F8 = SM == GDN_QDQ_E4M3 && WM == GDN_QDQ_E4M3 && DK == 128;
  constexpr int NTL = BV < 64 ? 64 / BV : 1;  // state-scale tiles in this block
  constexpr bool PAIR = BV == 128;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ float red[kStateWarps][NTL];  // per-warp partial amax of each state-scale tile
  __shared__ float xchg[2][2];             // PAIR: (fail, amax) from the peer value block
  __shared__ __align__(8) uint64_t bars[2];

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

  __nv_bfloat16* WcH = reinterpret_cast<__nv_bfloat16*>(sm + S::WC);
  __nv_bfloat16* WcL = WcH + kChunk * DK;  // WM == NONE only
  __nv_bfloat16* HcH = reinterpret_cast<__nv_bfloat16*>(sm + S::HC);
  __nv_bfloat16* HcL = HcH + DK * 64;      // SM == NONE only
  __nv_bfloat16* DpH = reinterpret_cast<__nv_bfloat16*>(sm + S::DP);
  __nv_bfloat16* DpL = DpH + kChunk * 64;
  uint8_t* Hst = sm + S::HST;
  uint8_t* Hb = sm + S::HC;  // F8: H^ codes [64 v][DK dk], swizzled like a bf16 [64][64] tile
  auto Kbuf = [&](int b) { return reinterpret_cast<__nv_bfloat16*>(sm + S::K + b * kChunk * DK * 2); };
  auto Wbuf = [&](int b) { return sm + S::WR + b * S::WRAW; };
  auto Ubuf = [&](int b) { return reinterpret_cast<float*>(sm + S::U + b * kChunk * 64 * 4); };
  auto Cbuf = [&](int b) { return reinterpret_cast<float*>(sm + S::CV + b * kCvecFloats * 4); };

  // Delta tile: [64 x 64] -> 16 x 16 per warp; state tile [DK x 64]
  const int row0 = (warp & 3) * 16, col0 = (warp >> 2) * 16;
  constexpr int HM = DK / 16;
  constexpr int HN = kStateWarps / HM;
  constexpr int NTH = 8 / HN;
  const int h_row0 = (warp % HM) * 16;
  const int h_col0 = (warp / HM) * (64 / HN);
  float hreg[NTH][4];
  // Every warp's column range starts on a multiple of 16 and every tile is at
  // least 16 wide, so a thread's state columns fall in two tiles at most:
  // ta (n-tiles 0, 1) and tb (n-tiles 2, 3); its Delta columns in tile td.
  const int ta = NTL == 1 ? 0 : h_col0 / BV;
  const int tb = NTL == 1 ? 0 : (h_col0 + 16) / BV;
  const int td = NTL == 1 ? 0 : col0 / BV;
  // per-warp partial amax of every state-scale tile of the block -> red
  auto tile_partials = [&]() {
    float ma = 0.f, mb = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (nt < 2) ma = fmaxf(ma, fabsf(hreg[nt][e]));
        else mb = fmaxf(mb, fabsf(hreg[nt][e]));
      }
    if constexpr (NTL == 1) {
      const float m = warp_max(fmaxf(ma, mb));
      if (lane == 0) red[warp][0] = m;
    } else {
      ma = warp_max(ma);
      if constexpr (NTH > 2) mb = warp_max(mb);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NTL; ++i) red[warp][i] = fmaxf(i == ta ? ma : 0.f, i == tb ? mb : 0.f);
      }
    }
  };
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
    tile_partials();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  float sW_next = 1.f;
  if (nchunks > 0) {
    issue_state_chunk<DK, WM, F8>(p, Kbuf(0), Wbuf(0), Ubuf(0), Cbuf(0), &bars[0], tok0,
                              min(L, kChunk), hk, h, vb, slot0);
    if constexpr (WM != GDN_QDQ_NONE) sW_next = p.w_scales[slot0 * p.Hv + h];
  }

  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int Lc = min(L - c * kChunk, kChunk);
    const int64_t slot = slot0 + c;
    const float sW = sW_next;
    const bool ok = mbar_wait(&bars[buf], (uint32_t)(c >> 1) & 1u);
    cp_async_wait<0>();
    if (threadIdx.x == 0) tma_store_wait_read();  // the codes store of chunk c - 1 has read Hst
    // chunk c landed; amax partials of H visible; buffer buf ^ 1 free
    bool fail = __syncthreads_or(!ok);
    // amax of each state-scale tile of the state entering chunk c
    float amx[NTL];
#pragma unroll
    for (int i = 0; i < NTL; ++i) {
      float a = red[0][i];
#pragma unroll
      for (int w = 1; w < kStateWarps; ++w) a = fmaxf(a, red[w][i]);
      amx[i] = a;
    }
    if constexpr (PAIR) {
      // one scale across both value blocks: the pair of CTAs (a cluster) swaps
      // its block amax, and its failure flag so that both leave together
      namespace cg = cooperative_groups;
      cg::cluster_group cl = cg::this_cluster();
      if (threadIdx.x == 0) {
        float* peer = cl.map_shared_rank(&xchg[c & 1][0], (int)(cl.block_rank() ^ 1));
        peer[0] = fail ? 1.f : 0.f;
        peer[1] = amx[0];
      }
      cl.sync();
      fail = fail || xchg[c & 1][0] != 0.f;
      amx[0] = fmaxf(amx[0], xchg[c & 1][1]);
    }
    if (fail) {
      if (threadIdx.x == 0) {
        atomicOr(&g_fwd_device_error, 1);
        mbar_wait(&bars[buf], (uint32_t)(c >> 1) & 1u);  // once more, bounded, for the copies in flight
        tma_store_wait_all();
      }
      return;
    }

    const float* dec = Cbuf(buf) + kCvDec;  // e^{gamma_L - gamma_i}
    const float egL = Cbuf(buf)[kCvEg + 63];  // e^{gamma_L} (gamma is flat past the last row)

    // W^ operand: codes -> bf16 values (exact), or the fp32 W split hi/lo; rows >= Lc are zero
    // (F8 reads the codes as they landed; rows >= Lc of Delta' are zeroed below)
    if constexpr (F8) {
    } else if constexpr (WM != GDN_QDQ_NONE) {
      const uint8_t* Wr = Wbuf(buf);
      constexpr int C4 = DK / 4;
      for (int i = threadIdx.x; i < kChunk * C4; i += kStateThreads) {
        const int r = i / C4, c4 = i % C4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < Lc) v = qdq_code4_values<WM>(*reinterpret_cast<const uint32_t*>(Wr + r * DK + c4 * 4));
        *reinterpret_cast<uint2*>(WcH + swz<DK>(r, c4 * 4)) =
            make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
      }
    } else {
      const float* Wr = reinterpret_cast<const float*>(Wbuf(buf));
      constexpr int C4 = DK / 4;
      for (int i = threadIdx.x; i < kChunk * C4; i += kStateThreads) {
        const int r = i / C4, c4 = i % C4;
        const float4 v = *reinterpret_cast<const float4*>(Wr + r * DK + c4 * 4);
        float h0v, l0v, h1v, l1v, h2v, l2v, h3v, l3v;
        split_bf16(v.x, h0v, l0v);
        split_bf16(v.y, h1v, l1v);
        split_bf16(v.z, h2v, l2v);
        split_bf16(v.w, h3v, l3v);
        const int e = swz<DK>(r, c4 * 4);
        *reinterpret_cast<uint2*>(WcH + e) = make_uint2(pack_bf16(h0v, h1v), pack_bf16(h2v, h3v));
        *reinterpret_cast<uint2*>(WcL + e) = make_uint2(pack_bf16(l0v, l1v), pack_bf16(l2v, l3v));
      }
    }

    // ---- a6: state QDQ per [DK x BV] tile ----
    // scale and reciprocal of each tile (the scale of an all-zero tile is 0)
    float sHt[NTL], rct[NTL];
#pragma unroll
    for (int i = 0; i < NTL; ++i) {
      sHt[i] = 1.f;
      rct[i] = 0.f;
      if constexpr (SM != GDN_QDQ_NONE) {
        qdq_scale<SM>(amx[i], sHt[i], rct[i]);
      }
    }
    const float sHa = pick(sHt, ta), rca = pick(rct, ta), ama = pick(amx, ta);
    const float sHb = pick(sHt, tb), rcb = pick(rct, tb), amb = pick(amx, tb);
    {
      if constexpr (F8) {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          const float sH = nt < 2 ? sHa : sHb, rcp = nt < 2 ? rca : rcb;
          const bool zero = (nt < 2 ? ama : amb) == 0.f;
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int d = h_row0 + gq + 8 * e2, col = h_col0 + nt * 8 + 2 * tq;
            float* hv = &hreg[nt][2 * e2];
            float2 val;
            // no usable scale (rcp == 0): signed-zero codes; with amax == 0 the values
            // (all zeros) stay, and a tiny amax turns them into zeros of their sign
            const uint16_t c2 = e4m3_code2(hv[0], hv[1], rcp, val);
            if (!zero) {
              hv[0] = __fmul_rn(val.x, sH);
              hv[1] = __fmul_rn(val.y, sH);
            }
            *reinterpret_cast<uint16_t*>(Hst + d * 64 + col) = c2;
            uint8_t* hb = Hb + 2 * swz<64>(col, d >> 1) + (d & 1);
            hb[0] = (uint8_t)(c2 & 0xff);
            hb[2 * swz<64>(col + 1, d >> 1) - 2 * swz<64>(col, d >> 1)] = (uint8_t)(c2 >> 8);
          }
        }
        fence_proxy_async();  // Hst is read by the TMA store below
      } else if constexpr (SM != GDN_QDQ_NONE) {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          const float sH = nt < 2 ? sHa : sHb, rcp = nt < 2 ? rca : rcb;
          const float amax = nt < 2 ? ama : amb;
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int d = h_row0 + gq + 8 * e2, col = h_col0 + nt * 8 + 2 * tq;
            float* hv = &hreg[nt][2 * e2];
            uint8_t c0, c1;
            float v0 = 0.f, v1 = 0.f;
            if (amax == 0.f) {
              c0 = qdq_zero_code<SM>(hv[0]);
              c1 = qdq_zero_code<SM>(hv[1]);
            } else {
              c0 = qdq_code<SM>(hv[0], rcp);
              c1 = qdq_code<SM>(hv[1], rcp);
              v0 = qdq_code_value<SM>(c0);
              v1 = qdq_code_value<SM>(c1);
              hv[0] = __fmul_rn(v0, sH);
              hv[1] = __fmul_rn(v1, sH);
            }
            st_bf16x2(HcH + swz<64>(d, col), v0, v1);
            *reinterpret_cast<uint16_t*>(Hst + d * 64 + col) = (uint16_t)(c0 | (c1 << 8));
          }
        }
        fence_proxy_async();  // Hst is read by the TMA store below
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
            *reinterpret_cast<float2*>(p.h_full + ((slot * p.Hv + h) * DK + d) * p.Dv + vb * 64 +
                                       col) = make_float2(hreg[nt][2 * e2], hreg[nt][2 * e2 + 1]);
          }
      }
    }
    __syncthreads();  // W^, H^ operands ready

    if (threadIdx.x == 0) {
      if constexpr (SM != GDN_QDQ_NONE) {
        tma_store_2d(&p.tm_hc, vb * 64, (int)((slot * p.Hv + h) * DK), Hst);
        tma_store_commit();
        // scales [slot, Hv, Dv / BV]
        if constexpr (PAIR) {
          if (vb == 0) p.h_scales[slot * p.Hv + h] = sHt[0];
        } else {
#pragma unroll
          for (int i = 0; i < NTL; ++i) p.h_scales[(slot * p.Hv + h) * (p.Dv / (64 / NTL)) + vb * NTL + i] = sHt[i];
        }
      }
    }
    // prefetch chunk c + 1 (buffer buf ^ 1 was last read before this iteration's first barrier)
    if (c + 1 < nchunks) {
      issue_state_chunk<DK, WM, F8>(p, Kbuf(buf ^ 1), Wbuf(buf ^ 1), Ubuf(buf ^ 1), Cbuf(buf ^ 1),
                                &bars[buf ^ 1], tok0 + (int64_t)(c + 1) * kChunk,
                                min(L - (c + 1) * kChunk, kChunk), hk, h, vb, slot + 1);
      if constexpr (WM != GDN_QDQ_NONE) sW_next = p.w_scales[(slot + 1) * p.Hv + h];
    }

    // ---- a7: Delta = U - W^ H^ (stored over U in o, for the output pass);
    //      Delta' = diag(e^{gamma_L - gamma}) Delta (rows >= Lc zero) ----
    {
      float dacc[2][4];
      zero_acc(dacc);
      if constexpr (F8) {
        const __nv_bfloat16* Wb = reinterpret_cast<const __nv_bfloat16*>(Wbuf(buf));
        const __nv_bfloat16* Hbb = reinterpret_cast<const __nv_bfloat16*>(Hb);
#pragma unroll
        for (int k2 = 0; k2 < DK / 2; k2 += 16) {  // 32 codes per step
          uint32_t a[4], b[4];
          ldsm_x4(a, a_frag_addr<64>(Wb, row0, k2, lane));
          ldsm_x4(b, bnk_frag_addr<64>(Hbb, col0, k2, lane));
          mma_e4m3(dacc[0], a, b[0], b[1]);
          mma_e4m3(dacc[1], a, b[2], b[3]);
        }
      } else {
        wgemm<2, false, true, DK, 64>(dacc, WcH, row0, HcH, col0, 0, DK, lane);
        if constexpr (WM == GDN_QDQ_NONE) wgemm<2, false, true, DK, 64>(dacc, WcL, row0, HcH, col0, 0, DK, lane);
        if constexpr (SM == GDN_QDQ_NONE) wgemm<2, false, true, DK, 64>(dacc, WcH, row0, HcL, col0, 0, DK, lane);
      }
      const float* Us = Ubuf(buf);
      const float sWH = (WM != GDN_QDQ_NONE ? sW : 1.f) * (SM != GDN_QDQ_NONE ? pick(sHt, td) : 1.f);
      float* dst = p.o + ((tok0 + (int64_t)c * kChunk) * p.Hv + h) * p.Dv + vb * 64;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
          const float2 u = *reinterpret_cast<const float2*>(Us + swz_f32(i, j));
          const float2 dl = make_float2(u.x - sWH * dacc[nt][2 * e2], u.y - sWH * dacc[nt][2 * e2 + 1]);
          // Delta replaces U in o (this sequence's rows only)
          if (i < Lc) *reinterpret_cast<float2*>(dst + (int64_t)i * p.Hv * p.Dv + j) = dl;
          const float di = i < Lc ? dec[i] : 0.f;  // rows past the chunk end contribute nothing
          float h0v, l0v, h1v, l1v;
          split_bf16(dl.x * di, h0v, l0v);
          split_bf16(dl.y * di, h1v, l1v);
          st_bf16x2(DpH + swz<64>(i, j), h0v, h1v);
          st_bf16x2(DpL + swz<64>(i, j), l0v, l1v);
        }
      }
    }
    __syncthreads();  // Delta' ready

    // ---- a9: H <- e^{gamma_L} H^ + K^T Delta' (K rows >= Lc meet zero rows of Delta') ----
    {
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) hreg[nt][e] *= egL;
      const __nv_bfloat16* Ks = Kbuf(buf);
      wgemm_shared_a<NTH, NTH, true, true, true, DK, 64, 64>(hreg, hreg, Ks, h_row0, DpH, h_col0, DpL,
                                                              h_col0, 0, 64, lane);
      tile_partials();
    }
  }
  cp_async_wait<0>();
  if (threadIdx.x == 0) tma_store_wait_all();

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

// ===========================================================================
// 3. Output: O = scale (diag(e^gamma) Q H^ + P Delta); Delta = U - W^ H^ as the
//    state scan left it in o.  One CTA per (chunk, value head): P = QK^T once,
//    then the value blocks in turn, the next block's Delta arriving by TMA
//    while the current one is multiplied.
// ===========================================================================
constexpr int kOutThreads = 256;

template <int DK, int SM, int WM>
struct OutSmem {
  static constexpr bool QUANT = SM != GDN_QDQ_NONE;
  static constexpr int Q = 0;                                  // bf16 [64][DK] (TMA)
  static constexpr int K = Q + kChunk * DK * 2;                // bf16 [64][DK] (TMA); later Delta hi, lo
  static constexpr int U = K + kChunk * DK * 2;                // f32 Delta [64][64] swz_f32 (TMA), per block
  static constexpr int P = U + kChunk * 64 * 4;                // P hi, lo
  static constexpr int HC = P + 2 * kChunk * 64 * 2;           // H^ of one block [DK][64] (hi, lo)
  static constexpr int HR = HC + (QUANT ? 1 : 2) * DK * 64 * 2;  // u8 H codes, both blocks (TMA)
  static constexpr int CV = HR + (QUANT ? 2 * DK * 64 : 0);    // chunk vectors
  // Delta hi, lo [64][64]: in the dead K tile when it is large enough
  static constexpr bool D_IN_K = 2 * kChunk * 64 * 2 <= kChunk * DK * 2;
  static constexpr int D = D_IN_K ? K : CV + kCvecFloats * 4;
  static constexpr int END = D_IN_K ? CV + kCvecFloats * 4 : D + 2 * kChunk * 64 * 2;
  static constexpr int BYTES = END + 1024;  // + alignment slack
  static_assert((K % 1024) == 0 && (U % 1024) == 0 && (P % 1024) == 0 &&
                    (HC % 128) == 0 && (HR % 128) == 0 && (CV % 16) == 0 && (D % 128) == 0,
                "alignment");
  static_assert(2 * (BYTES + 2048) <= 233472, "two CTAs per SM (with static and reserved shared memory)");
};

template <int DK, int SM, int WM>
__global__ void __launch_bounds__(kOutThreads, 2) gdn_fwd_output_kernel(const __grid_constant__ FwdParams p) {
  using S = OutSmem<DK, SM, WM>;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar;

  const int nvb = p.Dv / 64;
  const int64_t slot = blockIdx.x / p.Hv;
  const int h = (int)(blockIdx.x % p.Hv);
  ChunkRef cr;
  if (!chunk_of_slot(p, slot, cr)) return;
  const int hk = h / p.G;
  const int L = cr.L;
  const int64_t tok0 = cr.tok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;

  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(sm + S::Q);
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm + S::K);
  __nv_bfloat16* HcH = reinterpret_cast<__nv_bfloat16*>(sm + S::HC);
  __nv_bfloat16* HcL = HcH + DK * 64;
  float* Us = reinterpret_cast<float*>(sm + S::U);
  __nv_bfloat16* PH = reinterpret_cast<__nv_bfloat16*>(sm + S::P);
  __nv_bfloat16* PL = PH + kChunk * 64;
  __nv_bfloat16* DH = reinterpret_cast<__nv_bfloat16*>(sm + S::D);
  __nv_bfloat16* DL = DH + kChunk * 64;
  uint8_t* Hraw = sm + S::HR;  // [nvb][DK][64] state codes
  float* Cv = reinterpret_cast<float*>(sm + S::CV);
  const float* gam = Cv + kCvGam;
  const float* eg = Cv + kCvEg;

  auto load_u = [&](int vb) {  // by thread 0
#pragma unroll
    for (int pn = 0; pn < 2; ++pn)
      tma_load_2d(Us + pn * kChunk * 32, &p.tm_u, h * p.Dv + vb * 64 + pn * 32, (int)tok0, &bar);
  };
  // fp32 H of one block (state site off) -> hi, lo bf16 halves
  auto split_h_full = [&](int vb) {
    const float* src = p.h_full + ((slot * p.Hv + h) * DK) * p.Dv + vb * 64;
    for (int i = threadIdx.x; i < DK * 16; i += kOutThreads) {
      const int d = i >> 4, c4 = i & 15;
      const float4 v = *reinterpret_cast<const float4*>(src + (int64_t)d * p.Dv + c4 * 4);
      float h0v, l0v, h1v, l1v, h2v, l2v, h3v, l3v;
      split_bf16(v.x, h0v, l0v);
      split_bf16(v.y, h1v, l1v);
      split_bf16(v.z, h2v, l2v);
      split_bf16(v.w, h3v, l3v);
      const int e = swz<64>(d, c4 * 4);
      *reinterpret_cast<uint2*>(HcH + e) = make_uint2(pack_bf16(h0v, h1v), pack_bf16(h2v, h3v));
      *reinterpret_cast<uint2*>(HcL + e) = make_uint2(pack_bf16(l0v, l1v), pack_bf16(l2v, l3v));
    }
  };

  // ---- loads: TMA boxes on one mbarrier (phase 0: everything but the later
  //      blocks' Delta; phase vb: block vb's Delta) ----
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t bytes = 2 * kChunk * DK * 2 + kChunk * 64 * 4 + kCvecFloats * 4 +
                           (S::QUANT ? nvb * DK * 64 : 0);
    mbar_expect_tx(&bar, bytes);
    bulk_load_1d(Cv, p.cvec + (slot * p.Hv + h) * kCvecFloats, kCvecFloats * 4, &bar);
#pragma unroll
    for (int pn = 0; pn < DK / 64; ++pn) {
      tma_load_2d(Qs + pn * kChunk * 64, &p.tm_q, hk * DK + pn * 64, (int)tok0, &bar);
      tma_load_2d(Ks + pn * kChunk * 64, &p.tm_k, hk * DK + pn * 64, (int)tok0, &bar);
    }
    load_u(0);
    if constexpr (S::QUANT)
      for (int b = 0; b < nvb; ++b)
        tma_load_2d(Hraw + b * DK * 64, &p.tm_hc, b * 64, (int)((slot * p.Hv + h) * DK), &bar);
  }
  if constexpr (!S::QUANT) split_h_full(0);
  __syncthreads();  // the mbarrier is initialised before anyone waits on it
  const bool ok = mbar_wait(&bar, 0);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) {
      atomicOr(&g_fwd_device_error, 1);
      mbar_wait(&bar, 0);  // once more, bounded, for the copies in flight
    }
    return;
  }

  // warp tile: rows 16 rt .. +15, columns 32 ch .. +31.  Rows >= L of Q and K
  // hold another sequence's tokens: they only reach P entries outside the
  // causal mask or output rows that are not stored.
  const int rt = warp & 3, ch = warp >> 2;
  const int row0 = rt * 16, col0 = ch * 32;
  const bool p_tile = col0 <= row0 + 15;
  float pacc[4][4];
  zero_acc(pacc);
  if (p_tile) wgemm<4, false, false, DK, DK>(pacc, Qs, row0, Ks, col0, 0, DK, lane);

  for (int vb = 0; vb < nvb; ++vb) {
    if (vb > 0) {
      const bool okb = mbar_wait(&bar, (uint32_t)vb & 1u);
      if (__syncthreads_or(!okb)) {
        if (threadIdx.x == 0) {
          atomicOr(&g_fwd_device_error, 1);
          mbar_wait(&bar, (uint32_t)vb & 1u);
        }
        return;
      }
    }
    // codes -> bf16 values (exact); fp32 H split (state site off)
    if constexpr (S::QUANT) {
      const uint8_t* hr = Hraw + vb * DK * 64;
      for (int i = threadIdx.x; i < DK * 16; i += kOutThreads) {
        const int d = i >> 4, c4 = i & 15;
        const float4 v = qdq_code4_values<SM>(*reinterpret_cast<const uint32_t*>(hr + d * 64 + c4 * 4));
        *reinterpret_cast<uint2*>(HcH + swz<64>(d, c4 * 4)) =
            make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
      }
    } else if (vb > 0) {
      split_h_full(vb);
    }
    __syncthreads();  // H^ operand ready; the P product has read K (its tile becomes Delta)

    // state scales of this warp's two 16-column groups (each inside one
    // state-scale tile: tiles are 16-aligned and at least 16 wide); scales are
    // [slot, Hv, Dv / block_v]
    float sHa = 1.f, sHb = 1.f;
    if constexpr (S::QUANT) {
      const int64_t sb = (slot * p.Hv + h) * (p.Dv >> p.bv_log2);
      const int c = vb * 64 + col0;
      sHa = p.h_scales[sb + (c >> p.bv_log2)];
      sHb = p.h_scales[sb + ((c + 16) >> p.bv_log2)];
    }
    float qacc[4][4];
    zero_acc(qacc);
    wgemm<4, false, true, DK, 64>(qacc, Qs, row0, HcH, col0, 0, DK, lane);
    if constexpr (!S::QUANT) wgemm<4, false, true, DK, 64>(qacc, Qs, row0, HcL, col0, 0, DK, lane);

    // block 0 saves P (bf16; rows >= L zero) as the backward's tile image, and
    // every block its Delta (the hi half: Delta rounded to bf16)
    __nv_bfloat16* pimg = (vb == 0 && p.pb) ? p.pb + (slot * p.Hv + h) * (kTileImgBytes / 2) : nullptr;
    __nv_bfloat16* dimg = p.db ? p.db + ((slot * p.Hv + h) * nvb + vb) * (kTileImgBytes / 2) : nullptr;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
        float h0v, l0v, h1v, l1v;
        if (vb == 0) {
          if (p_tile) {
            const float gi = gam[i];
            const float p0 = (j <= i) ? expf(gi - gam[j]) * pacc[nt][2 * e2] : 0.f;
            const float p1 = (j + 1 <= i) ? expf(gi - gam[j + 1]) * pacc[nt][2 * e2 + 1] : 0.f;
            split_bf16(p0, h0v, l0v);
            split_bf16(p1, h1v, l1v);
            st_bf16x2(PH + swz<64>(i, j), h0v, h1v);
            st_bf16x2(PL + swz<64>(i, j), l0v, l1v);
            if (pimg) st_bf16x2(pimg + swz<64>(i, j), i < L ? p0 : 0.f, i < L ? p1 : 0.f);
          } else if (pimg) {
            st_bf16x2(pimg + swz<64>(i, j), 0.f, 0.f);
          }
        }
        float2 dl = *reinterpret_cast<const float2*>(Us + swz_f32(i, j));
        if (i >= L) dl = make_float2(0.f, 0.f);  // rows of another sequence
        split_bf16(dl.x, h0v, l0v);
        split_bf16(dl.y, h1v, l1v);
        st_bf16x2(DH + swz<64>(i, j), h0v, h1v);
        st_bf16x2(DL + swz<64>(i, j), l0v, l1v);
        if (dimg) st_bf16x2(dimg + swz<64>(i, j), h0v, h1v);
      }
    }
    // P, Delta ready; this block's Delta tile and H^ are read: the next block's
    // Delta may land in the Delta tile (reads by the generic proxy, then TMA)
    fence_proxy_async();
    __syncthreads();
    if (threadIdx.x == 0 && vb + 1 < nvb) {
      mbar_expect_tx(&bar, kChunk * 64 * 4);
      load_u(vb + 1);
    }

    float o2[4][4];
    zero_acc(o2);
    const int kend = row0 + 16;  // P is lower triangular: columns j <= i only
    wgemm_split3<4, false, true, 64, 64>(o2, PH, PL, row0, DH, DL, col0, 0, kend, lane);
    // O straight from the accumulators: each lane quad covers 32 contiguous bytes of a row
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = row0 + gq + 8 * e2, j = col0 + nt * 8 + 2 * tq;
        const float sq = nt < 2 ? sHa : sHb;
        const float ei = eg[i] * sq;
        if (i < L)
          *reinterpret_cast<float2*>(p.o + ((tok0 + i) * p.Hv + h) * p.Dv + vb * 64 + j) =
              make_float2(p.scale * (ei * qacc[nt][2 * e2] + o2[nt][2 * e2]),
                          p.scale * (ei * qacc[nt][2 * e2 + 1] + o2[nt][2 * e2 + 1]));
      }
    // the next block's H^ conversion and Delta split wait at its first barrier
    // for every warp to finish this block's products (they read H^, Delta hi/lo)
  }
}

// ===========================================================================
// launch
// ===========================================================================
template <typename Kern>
gdn_status set_smem(Kern kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
                 cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

template <int DK, int SM, int WM, int BV>
gdn_status launch_state(const FwdParams& prm, dim3 grid, cudaStream_t st) {
  // the none-state kernel is built for BV 64 only
  constexpr int B = SM == GDN_QDQ_NONE ? 64 : BV;
  auto k2 = gdn_fwd_state_kernel<DK, SM, WM, B>;
  if (set_smem(k2, StateSmem<DK, SM, WM>::BYTES) != GDN_OK) return GDN_ERR_CUDA;
  if constexpr (B == 128) {
    // the two value blocks of a (sequence, head) share a state scale: a 2-CTA cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = StateSmem<DK, SM, WM>::BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k2, prm) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  } else {
    k2<<<grid, kStateThreads, StateSmem<DK, SM, WM>::BYTES, st>>>(prm);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
}

template <int DK, int SM, int WM>
gdn_status launch_t(const FwdParams& prm, const Dims& d, cudaStream_t st) {
  const int nvb = d.Dv / 64;
  if (d.B * d.T > 0 && d.n_slots > 0) {
    auto k1 = gdn_fwd_prep_kernel<DK, WM, false>;
    if (set_smem(k1, PrepSmem<DK>::BYTES) != GDN_OK) return GDN_ERR_CUDA;
    k1<<<(unsigned)(d.n_slots * d.Hv), kPrepThreads, PrepSmem<DK>::BYTES, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  }
  {
    const dim3 grid((unsigned)nvb, (unsigned)d.Hv, (unsigned)d.N);
    const int bv = SM == GDN_QDQ_NONE ? 64 : prm.block_v;  // no state scales without a state QDQ
    const gdn_status s = bv == 16    ? launch_state<DK, SM, WM, 16>(prm, grid, st)
                         : bv == 32  ? launch_state<DK, SM, WM, 32>(prm, grid, st)
                         : bv == 128 ? launch_state<DK, SM, WM, 128>(prm, grid, st)
                                     : launch_state<DK, SM, WM, 64>(prm, grid, st);
    if (s != GDN_OK) return s;
  }
  if (d.B * d.T > 0 && d.n_slots > 0) {
    auto k3 = gdn_fwd_output_kernel<DK, SM, WM>;
    if (set_smem(k3, OutSmem<DK, SM, WM>::BYTES) != GDN_OK) return GDN_ERR_CUDA;
    k3<<<(unsigned)(d.n_slots * d.Hv), kOutThreads, OutSmem<DK, SM, WM>::BYTES, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  }
  return GDN_OK;
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

// Dk = Dv = 128, both sites quantized, block_v 64, exact solve: the chunk
// prep (T kept in fp32, no U) and the fused scan + outputs.
gdn_status launch_fused(const gdn_problem& p, const FwdParams& prm, const Dims& d,
                        cudaStream_t st) {
  const bool prep = d.B * d.T > 0 && d.n_slots > 0;
  if (prep) {
    gdn_status s = GDN_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return GDN_ERR_CUDA;
    // persistent: three CTAs per SM walk the chunk-heads
    const int64_t units = d.n_slots * d.Hv;
    const unsigned grid = (unsigned)std::min<int64_t>(units, 3 * (int64_t)sms);
    auto prep = [&](auto kern) {
      if (set_smem(kern, PrepSmemT<128>::BYTES) != GDN_OK) return GDN_ERR_CUDA;
      kern<<<grid, kPrepThreads, PrepSmemT<128>::BYTES, st>>>(prm);
      return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    };
    s = p.w_mode == GDN_QDQ_E4M3 ? prep(gdn_fwd_prep_kernel<128, GDN_QDQ_E4M3, true>)
                                 : prep(gdn_fwd_prep_kernel<128, GDN_QDQ_INT8, true>);
    if (s != GDN_OK) return s;
  }
  FusedParams f{};
  f.tm_k = prm.tm_k;
  f.tm_q = prm.tm_q;
  f.tm_v = prm.tm_v;
  f.tm_wc = prm.tm_wc;
  f.tu_img = prm.tu_img;
  f.cvec = prm.cvec;
  f.w_scales = prm.w_scales;
  f.h0 = prm.h0;
  f.o = prm.o;
  f.ht = prm.ht;
  f.h_codes = prm.h_codes;
  f.h_scales = prm.h_scales;
  f.pb = prm.pb;
  f.db = prm.db;
  f.cu_seqlens = prm.cu_seqlens;
  f.T = prm.T;
  f.nt_fixed = prm.nt_fixed;
  f.Hv = prm.Hv;
  f.G = prm.G;
  f.N = prm.N;
  f.scale = prm.scale;
  return launch_fused_scan(f, p.state_mode, p.w_mode, st, prep);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D row-major map: `cols` elements per row (contiguous), `rows` rows of
// `row_bytes` bytes; boxes of box_cols x box_rows elements.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols,
              uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle sw) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fwd_device_error(bool reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (reset && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_fwd_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

gdn_status launch_fwd(const gdn_problem& p, const Dims& d, const void* q, const void* k,
                      const void* v, const float* beta, const float* g, const float* h0,
                      float* o, float* ht, void* ctx, cudaStream_t st) {
  // 32-bit grid limits of the two per-chunk launches
  if (d.n_slots * d.Hv * (d.Dv / 64) > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED_SHAPE;
  FwdParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.h0 = h0;
  prm.o = o;
  prm.ht = ht;
  const CtxLayout L = ctx_layout(p);
  unsigned char* base = static_cast<unsigned char*>(ctx);
  // segments absent from this problem's layout stay null (nothing writes them)
  auto at = [&](int64_t off) -> unsigned char* { return off < 0 ? nullptr : base + off; };
  prm.w_codes = at(L.w_codes);
  prm.w_scales = reinterpret_cast<float*>(at(L.w_scales));
  prm.w_full = reinterpret_cast<float*>(at(L.w_full));
  prm.cvec = reinterpret_cast<float*>(at(L.cvec));
  prm.tb = reinterpret_cast<__nv_bfloat16*>(at(L.tb));
  prm.gkk = reinterpret_cast<__nv_bfloat16*>(at(L.gkk));
  prm.pb = reinterpret_cast<__nv_bfloat16*>(at(L.pb));
  prm.db = reinterpret_cast<__nv_bfloat16*>(at(L.db));
  prm.tu_img = reinterpret_cast<__nv_bfloat16*>(at(L.tu_img));
  prm.h_codes = at(L.h_codes);
  prm.h_scales = reinterpret_cast<float*>(at(L.h_scales));
  prm.h_full = reinterpret_cast<float*>(at(L.h_full));
  prm.cu_seqlens = p.cu_seqlens;
  prm.T = d.T;
  prm.Hk = d.Hk;
  prm.Hv = d.Hv;
  prm.Dv = d.Dv;
  prm.G = d.Hv / d.Hk;
  prm.N = (int)d.N;
  prm.nt_fixed = d.nt_fixed;
  prm.n_slots = d.n_slots;
  prm.scale = p.scale;
  prm.block_v = p.block_v;
  prm.bv_log2 = p.block_v == 16 ? 4 : (p.block_v == 32 ? 5 : (p.block_v == 64 ? 6 : 7));
  prm.neumann = p.solve == GDN_SOLVE_NEUMANN ? p.solve_degree : -1;
  if (p.block_v == 128 && d.Dv != 128) return GDN_ERR_UNSUPPORTED_MODE;
  const uint64_t tok = (uint64_t)(d.B * d.T);
  if (tok > 0) {
    // 32-bit TMA coordinates: state-code rows of all slots must fit
    if ((uint64_t)d.n_slots * d.Hv * d.Dk > 0x7fffffffULL) return GDN_ERR_UNSUPPORTED_SHAPE;
    const int DK = d.Dk;
    bool ok = make_map(&prm.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, (uint64_t)d.Hk * DK, tok,
                       (uint64_t)d.Hk * DK * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, (uint64_t)d.Hk * DK, tok,
                       (uint64_t)d.Hk * DK * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&prm.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, (uint64_t)d.Hv * d.Dv, tok,
                       (uint64_t)d.Hv * d.Dv * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&prm.tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, o, (uint64_t)d.Hv * d.Dv, tok,
                       (uint64_t)d.Hv * d.Dv * 4, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && p.w_mode != GDN_QDQ_NONE)
      ok = make_map(&prm.tm_wc, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.w_codes, (uint64_t)d.Hv * DK,
                    tok, (uint64_t)d.Hv * DK, DK, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && p.w_mode != GDN_QDQ_NONE && DK == 128)
      ok = make_map(&prm.tm_wc_sw, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.w_codes, (uint64_t)d.Hv * DK,
                    tok, (uint64_t)d.Hv * DK, DK, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && p.state_mode != GDN_QDQ_NONE)
      ok = make_map(&prm.tm_hc, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.h_codes, (uint64_t)d.Dv,
                    (uint64_t)d.n_slots * d.Hv * DK, (uint64_t)d.Dv, 64, DK,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return GDN_ERR_CUDA;
  }
  if (fused_fwd(p)) return launch_fused(p, prm, d, st);
  if (d.Dk == 128) return dispatch_modes<128>(p, prm, d, st);
  return dispatch_modes<64>(p, prm, d, st);
}

}  // namespace gdn
