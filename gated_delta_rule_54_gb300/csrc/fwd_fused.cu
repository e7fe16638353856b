// Fused state scan + outputs of the chunked gated delta rule forward with
// state / W fake QDQ, on the Blackwell tensor cores (tcgen05.mma, fp32
// accumulators in tensor memory, operands in shared memory read through
// matrix descriptors, inputs by TMA).
//
// Method ("[1/4] GDN state/W QAT foundation", "What does this PR do?": chunk
// 64, dynamic E4M3 fake QDQ at the state and W sites, exact solve; "Usage":
// state tiles [Dk, block_v = 64]; "[2/4] GDN/KDA decode QAT with INT8
// recurrent state": INT8 variant).  Per chunk of L <= 64 tokens, with the
// state H (Dk x Dv, H = S^T) entering it and T, W^ from the chunk prep:
//   U = T diag(beta) V;  H^ = Q_S(H);  Delta = U - W^ H^;
//   O = scale (diag(e^gamma) Q H^ + (lower-incl(e^{gamma_i-gamma_j} q_i.k_j)) Delta);
//   H <- e^{gamma_L} H^ + (diag(e^{gamma_L - gamma}) K)^T Delta.
//
// One CTA (8 warps) per (sequence, value head, 64-column value block) walks
// its chunks.  Everything is M = 128 tcgen05 products of bf16 operands:
//   D3 = [Tu_hi ; *] V + [Tu_lo ; *] V            rows 0-63: U
//   D4 = [W^ ; Q] K^T                             rows 64-127: QK^T -> P
//   D1 = [W^ ; Q] H^                              rows 0-63: W^ H^, rows 64-127: Q H^
//   D2 = K^T Delta'_hi + K^T Delta'_lo            the state update (M = Dk)
//   D5 = [* ; P_hi] Delta_hi + [* ; P_hi] Delta_lo + [* ; P_lo] Delta_hi
//                                                 rows 64-127: P Delta
// (a "*" half reads whatever lies next to the operand in shared memory: those
// accumulator rows are never read).  Quantized W and H enter as their codes
// (E4M3 values and INT8 integers are exact in bf16) with the scales applied in
// the epilogues; operands that are not bf16-exact (T diag(beta), P, Delta,
// the decayed Delta) are split into hi + lo bf16 halves, so the products keep
// about 16 mantissa bits.  Thread r (TMEM lane r) of each warp pair holds 32
// columns of accumulator row r; the fp32 state row dk of this value block
// lives in the registers of the two threads of lane dk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "fused.h"
#include "launch.h"

namespace gdn {

namespace {

__device__ int g_fused_device_error;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// shared memory (bytes from a 1024-aligned base)
struct FSmem {
  static constexpr int AQW = 0;                    // 2 buffers x [W^ ; Q]: 2 dk panels x 128 rows x 128 B
  static constexpr int KT = AQW + 2 * 32768;       // 2 buffers x K (2 panels x 64 rows x 128 B)
  static constexpr int VT = KT + 2 * 16384;        // V block [64 tok][64 v] bf16 (TMA, swizzled)
  static constexpr int WC = VT + 8192;             // W codes [64][128] u8 (TMA)
  static constexpr int ATU = WC + 8192;            // Tu hi, Tu lo images (bulk copy) ...
  static constexpr int AP = ATU + 16384;           // ... then P lo, P hi, P lo
  static constexpr int HB = AP + 24576;            // H^ codes as bf16 [128 dk][64 v]
  static constexpr int DP = HB + 16384;            // decayed Delta hi, lo [64 tok][64 v]
  static constexpr int DD = DP + 16384;            // Delta hi, lo
  static constexpr int CV = DD + 16384;            // 2 buffers x chunk vectors (1280 B)
  static constexpr int BYTES = CV + 2 * kCvecFloats * 4 + 1024;  // + alignment slack
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(AP == ATU + 16384, "[Tu_lo ; P_lo] read contiguously by the U product");
};

// TMEM accumulator columns
constexpr uint32_t kD1 = 0, kD2 = 64, kD3 = 128, kD4 = 192, kD5 = 256, kTmemCols = 512;

// bytes of one chunk's inputs: K, Q (2 boxes each), V, W codes, Tu images, chunk vectors
constexpr uint32_t kChunkTx = 2 * 8192 + 2 * 8192 + 8192 + 8192 + 16384 + kCvecFloats * 4;

// ---------------------------------------------------------------------------
// tcgen05 helpers
// ---------------------------------------------------------------------------
// shared-memory matrix descriptor: 128-byte swizzle, 8-row groups SBO apart,
// LBO = distance between 64-element blocks along M/N (MN-major operands)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor, kind::f16: bf16 x bf16 -> f32, M x N, operand majors
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdKK = idesc(128, 64, 0, 0);  // A K-major, B K-major
constexpr uint32_t kIdKM = idesc(128, 64, 0, 1);  // A K-major, B MN-major
constexpr uint32_t kIdMM = idesc(128, 64, 1, 1);  // A MN-major, B MN-major

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the hardware approximation (relative error about 2^-22; subnormal
// results flush to zero)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// (hi, lo) bf16 pairs of (x0, x1): hi = bf16(x), lo = bf16(x - hi), packed
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
  lo = pack_bf16(x0 - h0, x1 - h1);
}

// byte offset of element (row, col) in a tile of 128-byte rows (64 bf16),
// 16-byte chunks swizzled by the row within its 8-row group
__device__ __forceinline__ uint32_t sw_off(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2);
}
// eight bf16 values at (row, 8c .. 8c+7) of a swizzled tile: one 16-byte store
__device__ __forceinline__ void st8_bf16(unsigned char* tile, int row, int c8, const float* x) {
  uint4 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  u.z = pack_bf16(x[4], x[5]);
  u.w = pack_bf16(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + sw_off(row, 8 * c8)) = u;
}
// sixteen values at (row, 16 c16 ..) split into hi and lo tiles
__device__ __forceinline__ void st16_split(unsigned char* hi_tile, unsigned char* lo_tile, int row,
                                           int col, const float* x) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) split2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  *reinterpret_cast<uint4*>(hi_tile + sw_off(row, col)) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(hi_tile + sw_off(row, col + 8)) = make_uint4(h[4], h[5], h[6], h[7]);
  *reinterpret_cast<uint4*>(lo_tile + sw_off(row, col)) = make_uint4(l[0], l[1], l[2], l[3]);
  *reinterpret_cast<uint4*>(lo_tile + sw_off(row, col + 8)) = make_uint4(l[4], l[5], l[6], l[7]);
}

// Sixteen state values quantized with scale reciprocal rcp: codes (packed
// little-endian in c4), dequantized values x <- code * s, and the codes' values
// (exact in bf16) in v.  zero: the tile's amax is 0 (signed-zero codes, values
// kept, which are zeros).
template <int SM>
__device__ __forceinline__ void quant16(float (&x)[16], float rcp, float s, bool zero,
                                        float (&v)[16], uint32_t (&c4)[4]) {
  if constexpr (SM == GDN_QDQ_E4M3) {
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float2 val;
      const uint16_t c2 = e4m3_code2(x[j], x[j + 1], rcp, val);
      v[j] = val.x;
      v[j + 1] = val.y;
      if (!zero) {
        x[j] = __fmul_rn(val.x, s);
        x[j + 1] = __fmul_rn(val.y, s);
      }
      if (j % 4 == 0)
        c4[j / 4] = c2;
      else
        c4[j / 4] |= (uint32_t)c2 << 16;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint8_t cd = zero ? qdq_zero_code<SM>(x[j]) : qdq_code<SM>(x[j], rcp);
      v[j] = zero ? 0.f : qdq_code_value<SM>(cd);
      if (!zero) x[j] = __fmul_rn(v[j], s);
      if (j % 4 == 0)
        c4[j / 4] = cd;
      else
        c4[j / 4] |= (uint32_t)cd << (8 * (j % 4));
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int SM, int WM>
__global__ void __launch_bounds__(kThreads, 1) gdn_fwd_fused_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar_in[2];  // a chunk's inputs (per input buffer)
  __shared__ __align__(8) uint64_t bar_u, bar_a, bar_s, bar_o, bar_end;  // MMA completions
  __shared__ uint32_t tmem_slot;
  __shared__ float red[kWarps];

  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;         // TMEM lane quadrant of this warp
  const int row = 32 * quad + lane;  // accumulator row (TMEM lane)
  const int col0 = 16 * (warp >> 2); // this thread's 16 columns of the 64
  const bool lo_rows = quad < 2;     // rows 0-63 (tokens of the W^ / U / Delta products)
  const int t_row = row & 63;        // token of this row in the chunk

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
  const int nch = (L + kChunk - 1) / kChunk;

  unsigned char* VT = sm + FSmem::VT;
  const uint8_t* WCs = sm + FSmem::WC;
  unsigned char* ATU = sm + FSmem::ATU;
  unsigned char* AP = sm + FSmem::AP;
  unsigned char* HB = sm + FSmem::HB;
  unsigned char* DP = sm + FSmem::DP;
  unsigned char* DD = sm + FSmem::DD;
  auto AQWb = [&](int b) { return sm + FSmem::AQW + b * 32768; };
  auto KTb = [&](int b) { return sm + FSmem::KT + b * 16384; };
  auto CVb = [&](int b) { return reinterpret_cast<float*>(sm + FSmem::CV + b * kCvecFloats * 4); };

  // ---- set-up: TMEM, barriers ----
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  if (tid == 0) {
    mbar_init(&bar_in[0], 1);
    mbar_init(&bar_in[1], 1);
    mbar_init(&bar_u, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_end, 1);
    fence_mbar_init();
  }

  // TMA of chunk c's inputs, each issued once the buffer it fills is free
  auto load_kqc = [&](int c) {  // K, Q, chunk vectors (double buffered); opens the chunk's tx
    const int b = c & 1;
    const int64_t tok = tok0 + (int64_t)c * kChunk;
    mbar_expect_tx(&bar_in[b], kChunkTx);
    bulk_load_1d(CVb(b), p.cvec + ((slot0 + c) * p.Hv + h) * kCvecFloats, kCvecFloats * 4,
                 &bar_in[b]);
#pragma unroll
    for (int pn = 0; pn < 2; ++pn) {
      tma_load_2d(KTb(b) + pn * 8192, &p.tm_k, hk * 128 + pn * 64, (int)tok, &bar_in[b]);
      tma_load_2d(AQWb(b) + pn * 16384 + 8192, &p.tm_q, hk * 128 + pn * 64, (int)tok, &bar_in[b]);
    }
  };
  auto load_w = [&](int c) {  // W codes
    const int64_t tok = tok0 + (int64_t)c * kChunk;
    tma_load_2d(sm + FSmem::WC, &p.tm_wc, h * 128, (int)tok, &bar_in[c & 1]);
  };
  auto load_vt = [&](int c) {  // V block and the Tu images
    const int b = c & 1;
    const int64_t tok = tok0 + (int64_t)c * kChunk;
    tma_load_2d(VT, &p.tm_v, h * 128 + vb * 64, (int)tok, &bar_in[b]);
    bulk_load_1d(ATU,
                 reinterpret_cast<const unsigned char*>(p.tu_img) + ((slot0 + c) * p.Hv + h) * 16384,
                 16384, &bar_in[b]);
  };

  // ---- the state: thread (row dk, col0) holds H[dk][col0 .. col0 + 15] ----
  float hv[16];
  {
    const float* src = p.h0 ? p.h0 + (((int64_t)n * p.Hv + h) * 128 + row) * 128 + vb * 64 + col0
                            : nullptr;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (src) x = *reinterpret_cast<const float4*>(src + j);
      hv[j] = x.x;
      hv[j + 1] = x.y;
      hv[j + 2] = x.z;
      hv[j + 3] = x.w;
    }
  }
  auto amax_partial = [&]() {
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(hv[j]));
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
  };
  amax_partial();

  tc_fence_before();
  __syncthreads();  // TMEM address, barriers, red[] visible
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)col0;  // this thread's lane

  if (tid == 0 && nch > 0) {
    load_kqc(0);
    load_w(0);
    load_vt(0);
  }

  bool bad = false;
  int c = 0;
  for (; c < nch; ++c) {
    const int b = c & 1;
    const int64_t slot = slot0 + c;
    const int64_t tok = tok0 + (int64_t)c * kChunk;
    const int Lc = min(L - c * kChunk, kChunk);
    const uint32_t ph = (uint32_t)c & 1u;
    const float sW = p.w_scales[slot * p.Hv + h];
    unsigned char* AQW = AQWb(b);

    // ---- a6: state QDQ of the state entering chunk c ----
    bad |= !mbar_wait(&bar_in[b], (uint32_t)(c >> 1) & 1u);
    if (__syncthreads_or(bad)) break;  // inputs landed; red[] complete; the last chunk's reads done
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, red[w]);
    float sH, rcp;
    qdq_scale<SM>(amax, sH, rcp);
    {
      float vals[16];
      uint32_t c4[4];
      quant16<SM>(hv, rcp, sH, amax == 0.f, vals, c4);
      // H^ codes as bf16 values: the MN-major B operand [dk][v]
      st8_bf16(HB, row, col0 >> 3, vals);
      st8_bf16(HB, row, (col0 >> 3) + 1, vals + 8);
      if (p.h_codes) {
        uint8_t* dst = p.h_codes + ((slot * p.Hv + h) * 128 + row) * 128 + vb * 64 + col0;
        *reinterpret_cast<uint4*>(dst) = make_uint4(c4[0], c4[1], c4[2], c4[3]);
        if (tid == 0) p.h_scales[(slot * p.Hv + h) * 2 + vb] = sH;
      }
    }
    if (tid == 0 && c + 1 < nch) load_kqc(c + 1);  // buffers of chunk c - 1: free

    // ---- W^ codes -> bf16 values in rows 0-63 of [W^ ; Q] ----
    const float* cv = CVb(b);
    {
      const int r = tid >> 3, d0 = (tid & 7) * 16;  // row, first of 16 codes
      const uint4 cw = *reinterpret_cast<const uint4*>(WCs + r * 128 + d0);
      const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a = qdq_code4_values<WM>(w4[i]);
        x[4 * i] = a.x;
        x[4 * i + 1] = a.y;
        x[4 * i + 2] = a.z;
        x[4 * i + 3] = a.w;
      }
      unsigned char* panel = AQW + (d0 >> 6) * 16384;
      st8_bf16(panel, r, (d0 & 63) >> 3, x);
      st8_bf16(panel, r, ((d0 & 63) >> 3) + 1, x + 8);
    }
    fence_proxy_async();  // generic-proxy writes of HB and AQW before the MMAs read them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- the chunk's first products ----
    if (tid == 0) {
      if (c + 1 < nch) load_w(c + 1);  // W codes of this chunk are converted
      const uint32_t aq = smem_u32(AQW), atu = smem_u32(ATU), vt = smem_u32(VT);
      const uint32_t kt = smem_u32(KTb(b)), hb = smem_u32(HB);
      // D3 = [Tu_hi ; *] V + [Tu_lo ; *] V  (U in rows 0-63)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD3, sdesc(atu + ks * 32, 16, 1024), sdesc(vt + ks * 2048, 8192, 1024), kIdKM,
             ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD3, sdesc(atu + 8192 + ks * 32, 16, 1024), sdesc(vt + ks * 2048, 8192, 1024),
             kIdKM, true);
      // D4 = [W^ ; Q] K^T  (QK^T in rows 64-127)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma(tmem + kD4, sdesc(aq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
             sdesc(kt + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), kIdKK, ks > 0);
      umma_commit(&bar_u);
      // D1 = [W^ ; Q] H^  (W^ H^ in rows 0-63, Q H^ in rows 64-127)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma(tmem + kD1, sdesc(aq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
             sdesc(hb + ks * 2048, 8192, 1024), kIdKM, ks > 0);
      umma_commit(&bar_a);
    }

    // ---- U (rows 0-63) and P (rows 64-127) ----
    bad |= !mbar_wait(&bar_u, ph);
    tc_fence_after();
    if (tid == 0 && c + 1 < nch) load_vt(c + 1);  // D3 has read V and Tu
    float u[16];
    if (lo_rows) {
      tmem_ld16(tl + kD3, u);
    } else {
      // P_ij = 2^{(gamma_i - gamma_j) log2 e} q_i.k_j for j <= i (i = t_row, j = col0 + jj)
      float x[16];
      tmem_ld16(tl + kD4, x);
      constexpr float kLog2e = 1.4426950408889634f;
      const float gi = cv[kCvGam + t_row];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = col0 + jj;
        x[jj] = (j <= t_row) ? ex2_approx((gi - cv[kCvGam + j]) * kLog2e) * x[jj] : 0.f;
      }
      // [P_lo | P_hi | P_lo]: hi at +8 KB, lo at 0 and +16 KB
      st16_split(AP + 8192, AP, t_row, col0, x);
      *reinterpret_cast<uint4*>(AP + 16384 + sw_off(t_row, col0)) =
          *reinterpret_cast<const uint4*>(AP + sw_off(t_row, col0));
      *reinterpret_cast<uint4*>(AP + 16384 + sw_off(t_row, col0 + 8)) =
          *reinterpret_cast<const uint4*>(AP + sw_off(t_row, col0 + 8));
      if (p.pb && vb == 0) {
        unsigned char* pimg = reinterpret_cast<unsigned char*>(p.pb) + (slot * p.Hv + h) * 8192;
        float z[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) z[jj] = t_row < Lc ? x[jj] : 0.f;
        st8_bf16(pimg, t_row, col0 >> 3, z);
        st8_bf16(pimg, t_row, (col0 >> 3) + 1, z + 8);
      }
    }

    // ---- a7: Delta = U - sW sH W^ H^ (rows 0-63); decayed Delta' for the state update ----
    bad |= !mbar_wait(&bar_a, ph);
    tc_fence_after();
    if (lo_rows) {
      float y[16];
      tmem_ld16(tl + kD1, y);
      const float sWH = sW * sH;
      const bool valid = t_row < Lc;
      const float di = valid ? cv[kCvDec + t_row] : 0.f;
      float dl[16], dd[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        dl[j] = valid ? u[j] - sWH * y[j] : 0.f;
        dd[j] = dl[j] * di;
      }
      st16_split(DD, DD + 8192, t_row, col0, dl);
      st16_split(DP, DP + 8192, t_row, col0, dd);
      if (p.db) {
        // the Delta image: the hi half (Delta rounded to bf16), as stored in DD
        unsigned char* dimg = reinterpret_cast<unsigned char*>(p.db) + ((slot * p.Hv + h) * 2 + vb) * 8192;
        *reinterpret_cast<uint4*>(dimg + sw_off(t_row, col0)) =
            *reinterpret_cast<const uint4*>(DD + sw_off(t_row, col0));
        *reinterpret_cast<uint4*>(dimg + sw_off(t_row, col0 + 8)) =
            *reinterpret_cast<const uint4*>(DD + sw_off(t_row, col0 + 8));
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- a9 state update and the P Delta product ----
    if (tid == 0) {
      const uint32_t kt = smem_u32(KTb(b)), dp = smem_u32(DP), dd = smem_u32(DD);
      const uint32_t ap = smem_u32(AP);
      // D2 = K^T Delta'_hi + K^T Delta'_lo (A: K tile read MN-major, M = dk)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD2, sdesc(kt + ks * 2048, 8192, 1024), sdesc(dp + ks * 2048, 8192, 1024), kIdMM,
             ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD2, sdesc(kt + ks * 2048, 8192, 1024), sdesc(dp + 8192 + ks * 2048, 8192, 1024),
             kIdMM, true);
      umma_commit(&bar_s);
      // D5 = [P_lo ; P_hi] Delta_hi + [P_lo ; P_hi] Delta_lo + [P_hi ; P_lo] Delta_hi
      //      (rows 64-127: P Delta to ~16 bits)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD5, sdesc(ap + ks * 32, 16, 1024), sdesc(dd + ks * 2048, 8192, 1024), kIdKM,
             ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD5, sdesc(ap + ks * 32, 16, 1024), sdesc(dd + 8192 + ks * 2048, 8192, 1024),
             kIdKM, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma(tmem + kD5, sdesc(ap + 8192 + ks * 32, 16, 1024), sdesc(dd + ks * 2048, 8192, 1024),
             kIdKM, true);
      umma_commit(&bar_o);
    }

    // ---- H <- e^{gamma_L} H^ + K~^T Delta ----
    bad |= !mbar_wait(&bar_s, ph);
    tc_fence_after();
    {
      float z[16];
      tmem_ld16(tl + kD2, z);
      const float egL = cv[kCvEg + 63];  // gamma is flat past the last valid row
#pragma unroll
      for (int j = 0; j < 16; ++j) hv[j] = hv[j] * egL + z[j];
      amax_partial();
    }

    // ---- a8: O = scale (e^gamma sH Q H^ + P Delta) (rows 64-127) ----
    if (!lo_rows) {
      bad |= !mbar_wait(&bar_o, ph);
      tc_fence_after();
      float qh[16], pd[16];
      tmem_ld16(tl + kD1, qh);
      tmem_ld16(tl + kD5, pd);
      if (t_row < Lc) {
        const float ei = cv[kCvEg + t_row] * sH;
        float* dst = p.o + ((tok + t_row) * p.Hv + h) * 128 + vb * 64 + col0;
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(dst + j) =
              make_float4(p.scale * (ei * qh[j] + pd[j]), p.scale * (ei * qh[j + 1] + pd[j + 1]),
                          p.scale * (ei * qh[j + 2] + pd[j + 2]), p.scale * (ei * qh[j + 3] + pd[j + 3]));
      }
    }
    tc_fence_before();  // the next chunk's products overwrite the accumulators read here
  }

  // ---- final state (unquantized) ----
  if (!bad && p.ht) {
    float* dst = p.ht + (((int64_t)n * p.Hv + h) * 128 + row) * 128 + vb * 64 + col0;
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      *reinterpret_cast<float4*>(dst + j) = make_float4(hv[j], hv[j + 1], hv[j + 2], hv[j + 3]);
  }

  // ---- tear-down: no product or copy may be in flight when TMEM is freed ----
  if (tid == 0) {
    if (bad) {
      atomicOr(&g_fused_device_error, 1);
      // the copies of the chunk the loop stopped at (bounded waits, as above)
      if (c < nch) mbar_wait(&bar_in[c & 1], (uint32_t)(c >> 1) & 1u);
      if (c + 1 < nch) mbar_wait(&bar_in[(c + 1) & 1], (uint32_t)((c + 1) >> 1) & 1u);
    }
    umma_commit(&bar_end);  // completes once every product issued so far is done
    mbar_wait(&bar_end, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols));
}

}  // namespace

gdn_status launch_fused_scan(const FusedParams& p, int state_mode, int w_mode, cudaStream_t st) {
  const dim3 grid(2, (unsigned)p.Hv, (unsigned)p.N);
  auto run = [&](auto kern) -> gdn_status {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FSmem::BYTES) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
    kern<<<grid, kThreads, FSmem::BYTES, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  };
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_E4M3)
    return run(gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_E4M3>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_E4M3)
    return run(gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_E4M3>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_INT8)
    return run(gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_INT8>);
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_INT8)
    return run(gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_INT8>);
  return GDN_ERR_UNSUPPORTED_MODE;
}

int fused_device_error(bool reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fused_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (reset && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_fused_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
