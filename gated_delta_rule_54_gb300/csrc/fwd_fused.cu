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
// One CTA (16 epilogue warps + 1 producer warp) per (sequence, value head,
// 64-column value block) walks its chunks.  Everything is M = 128 tcgen05
// products of bf16 operands:
//   D3 = [Tu_hi ; Tu_lo] V                        rows 0-63: Tu_hi V, rows 64-127: Tu_lo V;
//                                                 U = their sum (the second half crosses
//                                                 to the rows-0-63 warps in shared memory)
//   D4 = [W^ ; Q] K^T                             rows 64-127: QK^T -> P
//   D1 = [W^ ; Q] H^                              rows 0-63: W^ H^, rows 64-127: Q H^
//   D2 = K^T [Delta'_hi | Delta'_lo]              N = 128; the state update (M = Dk)
//                                                 is the sum of its two column halves
//   D5 = [* ; P_hi] [Delta_hi | Delta_lo] + [* ; P_lo] Delta_hi (into columns 0-63)
//                                                 rows 64-127: P Delta, again the sum
//                                                 of the two column halves
// (a "*" half reads whatever lies next to the operand in shared memory: those
// accumulator rows are never read).  A [hi | lo] operand is one N = 128 B
// operand: its halves lie a panel stride apart, so one product reads the A
// tile once for both.  Quantized W and H enter as their codes
// (E4M3 values and INT8 integers are exact in bf16) with the scales applied in
// the epilogues; operands that are not bf16-exact (T diag(beta), P, Delta,
// the decayed Delta) are split into hi + lo bf16 halves, so the products keep
// about 16 mantissa bits.  The four warps of TMEM lane quadrant q each read 16
// columns of accumulator rows 32q .. 32q + 31 (one row per thread); the fp32
// state row dk of this value block lives in the registers of the four threads
// of lane dk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "fused.h"
#include "tc.cuh"
#include "launch.h"

namespace gdn {

namespace {

__device__ int g_fused_device_error;

constexpr int kEpiThreads = 512;               // 16 epilogue warps
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kThreads = kEpiThreads + 32;     // + the producer warp (TMA and MMA issue)

// shared memory (bytes from a 1024-aligned base)
struct FSmem {
  static constexpr int AQW = 0;                    // [W^ ; Q]: 2 dk panels x 128 rows x 128 B
  static constexpr int KT = AQW + 32768;           // 2 buffers x K (2 panels x 64 rows x 128 B)
  static constexpr int VT = KT + 2 * 16384;        // 2 buffers x V block [64 tok][64 v] bf16
  static constexpr int WC = VT + 2 * 8192;         // 2 buffers x W codes [64][128] u8
  static constexpr int ATU = WC + 2 * 8192;        // 2 buffers x Tu hi, Tu lo images; buffer 1 ...
  static constexpr int AP = ATU + 2 * 16384;       // ... then P lo, P hi
  static constexpr int HB = AP + 16384;            // H^ codes as bf16 [128 dk][64 v]
  static constexpr int DP = HB + 16384;            // decayed Delta hi, lo [64 tok][64 v]
  static constexpr int DD = DP + 16384;            // Delta hi, lo
  static constexpr int ULO = DD + 16384;           // Tu_lo V, fp32 [64 tok][64 v] (16-byte chunks swizzled by row)
  static constexpr int CV = ULO + 16384;           // 2 buffers x chunk vectors (1280 B)
  static constexpr int BYTES = CV + 2 * kCvecFloats * 4 + 1024;  // + alignment slack
  static_assert(BYTES <= 232448, "shared memory budget");
};

// TMEM accumulator columns: D1 double buffered (chunk parity); D2 and D5 are
// N = 128 products
constexpr uint32_t kD1 = 0, kD2 = 128, kD3 = 256, kD4 = 320, kD5 = 384, kTmemCols = 512;

// bytes of the copy groups of one chunk
constexpr uint32_t kVtTx = 8192 + 16384 + 8192;  // V block, Tu images, W codes
constexpr uint32_t kKwTx = 2 * 8192;             // K (2 boxes)
constexpr uint32_t kCvTx = kCvecFloats * 4;   // chunk vectors
constexpr uint32_t kQTx = 2 * 8192;           // Q (2 boxes)

constexpr uint32_t kIdKK = idesc(128, 64, 0, 0);  // A K-major, B K-major
constexpr uint32_t kIdKM = idesc(128, 64, 0, 1);  // A K-major, B MN-major
// N = 128: a B operand of two 64-column panels 8 KB apart ([hi | lo] halves)
constexpr uint32_t kIdKM2 = idesc(128, 128, 0, 1);
constexpr uint32_t kIdMM2 = idesc(128, 128, 1, 1);

// barrier among the epilogue warps only (the producer warp does not take part),
// returning whether any of them passed v = true
__device__ __forceinline__ bool epi_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kEpiThreads)
      : "memory");
  return r != 0;
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
// Warp 16 is the producer: one lane issues the TMA copies and the tensor-core
// products.  Warps 0-15 run the epilogues; warp w reads TMEM lanes
// 32 (w % 4) .. +31 (accumulator rows) and columns 16 (w / 4) .. +15.
// Per chunk c the products and epilogues are ordered so that only the state
// chain waits: QDQ(c) -> D1(c) = [W^ ; Q] H^ -> Delta(c) -> D2(c) = K^T Delta'
// -> H_{c+1}; D4(c) (QK^T), D5(c) (P Delta) and D3(c+1) (U of the next chunk)
// fill the tensor pipe in between, the next chunk's W^ conversion runs while
// D2(c) executes, and the outputs of chunk c are stored after QDQ(c+1).
// CTX: the backward's context (state codes and scales, P images) is saved.
template <int SM, int WM, bool CTX>
__global__ void __launch_bounds__(kThreads, 1) gdn_fwd_fused_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  // copies of buffer b: in_vt (V, Tu, W codes), in_kw (K), in_cv (chunk vectors); in_q (Q)
  __shared__ __align__(8) uint64_t in_vt[2], in_kw[2], in_cv[2], in_q;
  // products done: u (D3), a (D1), d4 (D4), s (D2), o (D5), end (everything)
  __shared__ __align__(8) uint64_t b_u, b_a, b_d4, b_s, b_o, b_end;
  // epilogue signals: H^ and W^ ready, P ready, Delta ready, outputs stored
  __shared__ __align__(8) uint64_t e_hb, e_p, e_dl, e_out, e_ulo;
  __shared__ uint32_t tmem_slot;
  __shared__ float red[kEpiWarps];
  __shared__ int abort_flag;

  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == kEpiWarps;
  const int quad = warp & 3;         // TMEM lane quadrant of this warp
  const int row = 32 * quad + lane;  // accumulator row (TMEM lane)
  const int col0 = 16 * ((warp >> 2) & 3);  // this thread's 16 columns of the 64
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

  unsigned char* AQW = sm + FSmem::AQW;
  unsigned char* AP = sm + FSmem::AP;
  unsigned char* HB = sm + FSmem::HB;
  unsigned char* DP = sm + FSmem::DP;
  unsigned char* DD = sm + FSmem::DD;
  auto KTb = [&](int b) { return sm + FSmem::KT + b * 16384; };
  auto VTb = [&](int b) { return sm + FSmem::VT + b * 8192; };
  auto WCb = [&](int b) { return sm + FSmem::WC + b * 8192; };
  auto ATUb = [&](int b) { return sm + FSmem::ATU + b * 16384; };
  auto CVb = [&](int b) { return reinterpret_cast<float*>(sm + FSmem::CV + b * kCvecFloats * 4); };

  // ---- set-up: TMEM, barriers ----
  if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(&in_vt[bb], 1);
      mbar_init(&in_kw[bb], 1);
      mbar_init(&in_cv[bb], 1);
    }
    mbar_init(&in_q, 1);
    mbar_init(&b_u, 1);
    mbar_init(&b_a, 1);
    mbar_init(&b_d4, 1);
    mbar_init(&b_s, 1);
    mbar_init(&b_o, 1);
    mbar_init(&b_end, 1);
    mbar_init(&e_hb, kEpiWarps);
    mbar_init(&e_p, kEpiWarps / 2);
    mbar_init(&e_dl, kEpiWarps / 2);
    mbar_init(&e_out, kEpiWarps / 2);
    mbar_init(&e_ulo, kEpiWarps / 2);
    abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();  // TMEM address, barriers visible
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool bad = false;

  if (producer) {
    // ======================= producer warp =======================
    if (lane == 0 && nch > 0) {
      auto tok_of = [&](int c) { return (int)(tok0 + (int64_t)c * kChunk); };
      auto sh_of = [&](int c) { return (slot0 + c) * p.Hv + h; };
      auto load_vt = [&](int c) {  // V block, Tu images and W codes of chunk c
        const int b = c & 1;
        mbar_expect_tx(&in_vt[b], kVtTx);
        tma_load_2d(VTb(b), &p.tm_v, h * 128 + vb * 64, tok_of(c), &in_vt[b]);
        bulk_load_1d(ATUb(b), reinterpret_cast<const unsigned char*>(p.tu_img) + sh_of(c) * 16384,
                     16384, &in_vt[b]);
        tma_load_2d(WCb(b), &p.tm_wc, h * 128, tok_of(c), &in_vt[b]);
      };
      auto load_kw = [&](int c) {  // K of chunk c
        const int b = c & 1;
        mbar_expect_tx(&in_kw[b], kKwTx);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_2d(KTb(b) + pn * 8192, &p.tm_k, hk * 128 + pn * 64, tok_of(c), &in_kw[b]);
      };
      auto load_cv = [&](int c) {  // chunk vectors of chunk c
        const int b = c & 1;
        mbar_expect_tx(&in_cv[b], kCvTx);
        bulk_load_1d(CVb(b), p.cvec + sh_of(c) * kCvecFloats, kCvecFloats * 4, &in_cv[b]);
      };
      auto load_q = [&](int c) {  // Q into rows 64-127 of both panels of [W^ ; Q]
        mbar_expect_tx(&in_q, kQTx);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_2d(AQW + pn * 16384 + 8192, &p.tm_q, hk * 128 + pn * 64, tok_of(c), &in_q);
      };
      // D3 = [Tu_hi ; Tu_lo] V  (Tu_hi V in rows 0-63, Tu_lo V in rows 64-127)
      auto issue_u = [&](int c) {
        const int b = c & 1;
        const uint64_t atu = sdesc(smem_u32(ATUb(b)), 16, 1024), vt = sdesc(smem_u32(VTb(b)), 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma(tmem + kD3, dadd(atu, ks * 32), dadd(vt, ks * 2048), kIdKM, ks > 0);
        umma_commit(&b_u);
      };
      load_kw(0);
      load_q(0);
      // the chunk prep's outputs (Tu images, W codes, chunk vectors) are complete
      grid_dep_wait();
      load_vt(0);
      load_cv(0);
      bad |= !mbar_wait(&in_vt[0], 0);
      tc_fence_after();
      if (!bad) issue_u(0);
      for (int c = 0; c < nch && !bad; ++c) {
        const int b = c & 1;
        const uint32_t ph = (uint32_t)c & 1u, phb = (uint32_t)(c >> 1) & 1u;
        const bool more = c + 1 < nch;
        // V, Tu and W codes of the next chunk: their buffer's last readers, D3(c - 1)
        // and the W^ conversion of chunk c - 1, finished before the epilogues of
        // chunk c - 1 signalled
        if (more) load_vt(c + 1);
        // D1 = [W^ ; Q] H^ once H^(c) and W^(c) are written and K(c), Q(c) have landed
        bad |= !mbar_wait(&e_hb, ph);
        bad |= !mbar_wait(&in_q, ph);
        bad |= !mbar_wait(&in_kw[b], phb);
        if (bad) break;
        tc_fence_after();
        const uint64_t aq = sdesc(smem_u32(AQW), 16, 1024), hb = sdesc(smem_u32(HB), 8192, 1024);
        const uint64_t ktk = sdesc(smem_u32(KTb(b)), 16, 1024);
        const uint32_t d1 = tmem + kD1 + 64 * (c & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma(d1, dadd(aq, (ks >> 2) * 16384 + (ks & 3) * 32), dadd(hb, ks * 2048), kIdKM, ks > 0);
        umma_commit(&b_a);
        // D4 = [W^ ; Q] K^T (QK^T in rows 64-127)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma(tmem + kD4, dadd(aq, (ks >> 2) * 16384 + (ks & 3) * 32),
               dadd(ktk, (ks >> 2) * 8192 + (ks & 3) * 32), kIdKK, ks > 0);
        umma_commit(&b_d4);
        // K of the next chunk: H^(c) being ready means the state update of chunk
        // c - 1 ran, so D2(c - 1), the last reader of that K buffer, is done
        if (more) load_kw(c + 1);
        // Q of the next chunk once D1(c) and D4(c) have read this one
        if (more) {
          bad |= !mbar_wait(&b_d4, ph);
          if (!bad) load_q(c + 1);
        }
        // D2 = K^T [Delta'_hi | Delta'_lo] (A: K tile read MN-major, M = dk)
        bad |= !mbar_wait(&e_dl, ph);
        if (bad) break;
        tc_fence_after();
        const uint64_t dp = sdesc(smem_u32(DP), 8192, 1024), dd = sdesc(smem_u32(DD), 8192, 1024);
        const uint64_t ap = sdesc(smem_u32(AP), 16, 1024), ktm = sdesc(smem_u32(KTb(b)), 8192, 1024);
        // one N = 128 product: K^T Delta'_hi in columns 0-63, K^T Delta'_lo in 64-127
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma(tmem + kD2, dadd(ktm, ks * 2048), dadd(dp, ks * 2048), kIdMM2, ks > 0);
        umma_commit(&b_s);
        // chunk vectors of the next chunk once the outputs of chunk c - 1 are stored
        if (more) {
          if (c >= 1) bad |= !mbar_wait(&e_out, ph ^ 1u);
          if (!bad) load_cv(c + 1);
        }
        // D5 = [P_lo ; P_hi] [Delta_hi | Delta_lo] + [* ; P_lo] Delta_hi
        bad |= !mbar_wait(&e_p, ph);
        if (bad) break;
        tc_fence_after();
        // [P_lo ; P_hi] [Delta_hi | Delta_lo] as one N = 128 product, then
        // [* ; P_lo] Delta_hi into columns 0-63 (the A tile starts one panel
        // below P_lo, in the second Tu buffer, so its rows 64-127 are P_lo).  The P epilogue of chunk c + 1
        // reads D5(c) before it signals, so one buffer serves.
        const uint32_t d5 = tmem + kD5;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma(d5, dadd(ap, ks * 32), dadd(dd, ks * 2048), kIdKM2, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma(d5, dadd(ap, ks * 32) - (8192 >> 4), dadd(dd, ks * 2048), kIdKM, true);
        umma_commit(&b_o);
        // U of the next chunk (the Delta epilogue of chunk c has read D3(c))
        if (more) {
          bad |= !mbar_wait(&in_vt[b ^ 1], (uint32_t)((c + 1) >> 1) & 1u);
          if (bad) break;
          tc_fence_after();
          issue_u(c + 1);
        }
      }
      if (bad) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ======================= epilogue warps =======================
    const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)col0;  // this thread's lane
    float hv[16];  // thread (row dk, col0) holds H[dk][col0 .. col0 + 15]
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
    grid_dep_wait();  // the W scales below are the chunk prep's
    auto amax_partial = [&]() {
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(hv[j]));
      m = warp_max(m);
      if (lane == 0) red[warp] = m;
    };
    // W^ codes of chunk c -> bf16 values in rows 0-63 of [W^ ; Q]; nthr threads
    // (index i) share the 64 x 128 codes, 16 at a time
    auto convert_w = [&](int c, int i, int nthr) {
      for (int e = i; e < 64 * 8; e += nthr) {
        const int r = e >> 3, d0 = (e & 7) * 16;  // row, first of 16 codes
        const uint4 cw = *reinterpret_cast<const uint4*>(WCb(c & 1) + r * 128 + d0);
        const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
        float x[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 a = qdq_code4_values<WM>(w4[k]);
          x[4 * k] = a.x;
          x[4 * k + 1] = a.y;
          x[4 * k + 2] = a.z;
          x[4 * k + 3] = a.w;
        }
        unsigned char* panel = AQW + (d0 >> 6) * 16384;
        st8_bf16(panel, r, (d0 & 63) >> 3, x);
        st8_bf16(panel, r, ((d0 & 63) >> 3) + 1, x + 8);
      }
    };
    // outputs of chunk c: O = scale (e^gamma sH Q H^ + P Delta), rows 64-127
    auto store_out = [&](int c, float sH) {
      bad |= !mbar_wait(&b_o, (uint32_t)c & 1u);
      tc_fence_after();
      const int Lc = min(L - c * kChunk, kChunk);
      const float* cv = CVb(c & 1);
      float qh[16], pd[16];
      {
        float pl[16];
        tmem_ld16_pair(tl + kD5, pd, tl + kD5 + 64, pl);
#pragma unroll
        for (int j = 0; j < 16; ++j) pd[j] += pl[j];
      }
      tmem_ld16(tl + kD1 + 64 * (c & 1), qh);
      if (t_row < Lc) {
        const float ei = cv[kCvEg + t_row] * sH;
        float* dst = p.o + ((tok0 + (int64_t)c * kChunk + t_row) * p.Hv + h) * 128 + vb * 64 + col0;
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(dst + j) =
              make_float4(p.scale * (ei * qh[j] + pd[j]), p.scale * (ei * qh[j + 1] + pd[j + 1]),
                          p.scale * (ei * qh[j + 2] + pd[j + 2]),
                          p.scale * (ei * qh[j + 3] + pd[j + 3]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&e_out);
    };

    amax_partial();
    if (nch > 0) {
      bad |= !mbar_wait(&in_vt[0], 0);
      convert_w(0, tid, kEpiThreads);
    }
    constexpr bool all_convert = CTX;
    float sH_prev = 1.f;
    int c = 0;
    for (; c < nch; ++c) {
      const int b = c & 1;
      const int64_t slot = slot0 + c;
      const int Lc = min(L - c * kChunk, kChunk);
      const uint32_t ph = (uint32_t)c & 1u;
      const float sW = p.w_scales[slot * p.Hv + h];

      // ---- a6: state QDQ of the state entering chunk c (red[]: H_c's partial amax) ----
      // (uniform decision: every epilogue thread leaves the loop together)
      if (epi_sync_or(bad || *reinterpret_cast<volatile int*>(&abort_flag) != 0)) {
        bad = true;
        break;
      }
      float amax = red[0];
#pragma unroll
      for (int w = 1; w < kEpiWarps; ++w) amax = fmaxf(amax, red[w]);
      float sH, rcp;
      qdq_scale<SM>(amax, sH, rcp);
      uint32_t c4[4];
      {
        float vals[16];
        quant16<SM>(hv, rcp, sH, amax == 0.f, vals, c4);
        st8_bf16(HB, row, col0 >> 3, vals);
        st8_bf16(HB, row, (col0 >> 3) + 1, vals + 8);
      }
      fence_proxy_async();  // H^ (and the W^ converted earlier) before D1 reads them
      __syncwarp();
      if (lane == 0) mbar_arrive(&e_hb);
      // the backward's copy of the state codes, after the signal (the arrival
      // orders this thread's earlier writes, so a global store before it would
      // hold it back)
      if (CTX && p.h_codes) {
        uint8_t* dst = p.h_codes + ((slot * p.Hv + h) * 128 + row) * 128 + vb * 64 + col0;
        *reinterpret_cast<uint4*>(dst) = make_uint4(c4[0], c4[1], c4[2], c4[3]);
        if (tid == 0) p.h_scales[(slot * p.Hv + h) * 2 + vb] = sH;
      }

      // ---- Tu_lo V (D3 rows 64-127) to the warps of rows 0-63 ----
      float* ulo = reinterpret_cast<float*>(sm + FSmem::ULO) + t_row * 64;
      auto ulo_chunk = [&](int j) { return ((col0 >> 2) + j) ^ (t_row & 7); };
      if (!lo_rows) {
        bad |= !mbar_wait(&b_u, ph);
        tc_fence_after();
        float x[16];
        tmem_ld16(tl + kD3, x);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<float4*>(ulo + 4 * ulo_chunk(j)) =
              make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&e_ulo);
      }

      // ---- outputs of the previous chunk (its D1 and D5 buffers) ----
      if (!lo_rows && c > 0) store_out(c - 1, sH_prev);


      bad |= !mbar_wait(&in_cv[b], (uint32_t)(c >> 1) & 1u);  // this chunk's vectors
      const float* cv = CVb(b);
      float u[16];
      if (lo_rows) {
        // U (rows 0-63) = Tu_hi V (D3 rows 0-63) + Tu_lo V (from the other warps)
        bad |= !mbar_wait(&b_u, ph);
        tc_fence_after();
        tmem_ld16(tl + kD3, u);
        bad |= !mbar_wait(&e_ulo, ph);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 a = *reinterpret_cast<const float4*>(ulo + 4 * ulo_chunk(j));
          u[4 * j] += a.x;
          u[4 * j + 1] += a.y;
          u[4 * j + 2] += a.z;
          u[4 * j + 3] += a.w;
        }
      } else {
        // P_ij = 2^{(gamma_i - gamma_j) log2 e} q_i.k_j for j <= i (i = t_row, j = col0 + jj)
        bad |= !mbar_wait(&b_d4, ph);
        tc_fence_after();
        float x[16];
        tmem_ld16(tl + kD4, x);
        constexpr float kLog2e = 1.4426950408889634f;
        const float gi = cv[kCvGam + t_row];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = col0 + jj;
          x[jj] = (j <= t_row) ? ex2_approx((gi - cv[kCvGam + j]) * kLog2e) * x[jj] : 0.f;
        }
        // [P_lo | P_hi]: lo at 0, hi at +8 KB
        st16_split(AP + 8192, AP, t_row, col0, x);
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&e_p);
        // the P image the backward reads: P_hi (the bf16 rounding of P) in the
        // tile's swizzled layout, rows past the chunk end zero, after the signal
        if (CTX && p.pb && vb == 0) {
          unsigned char* pimg = reinterpret_cast<unsigned char*>(p.pb) + (slot * p.Hv + h) * 8192;
          float z[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) z[jj] = t_row < Lc ? x[jj] : 0.f;
          st8_bf16(pimg, t_row, col0 >> 3, z);
          st8_bf16(pimg, t_row, (col0 >> 3) + 1, z + 8);
        }
      }

      // ---- a7: Delta = U - sW sH W^ H^ (rows 0-63); decayed Delta' for the state update ----
      if (lo_rows) {
        bad |= !mbar_wait(&b_a, ph);
        tc_fence_after();
        float y[16];
        tmem_ld16(tl + kD1 + 64 * (c & 1), y);
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
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&e_dl);
        if (CTX && p.db) {
          // the Delta image: the hi half (Delta rounded to bf16, as in DD), after the signal
          unsigned char* dimg =
              reinterpret_cast<unsigned char*>(p.db) + ((slot * p.Hv + h) * 2 + vb) * 8192;
          st8_bf16(dimg, t_row, col0 >> 3, dl);
          st8_bf16(dimg, t_row, (col0 >> 3) + 1, dl + 8);
        }
      }

      // ---- the next chunk's W^, while D2 runs: [W^ ; Q] is free once D1 and D4 are done.
      // Without the backward's context the warps of rows 64-127 convert it (the
      // others carry the chain Delta -> D2 -> state); with it, those warps also
      // store the P image, and all warps share the conversion ----
      if (c + 1 < nch && (all_convert || !lo_rows)) {
        bad |= !mbar_wait(&b_d4, ph);
        bad |= !mbar_wait(&in_vt[b ^ 1], (uint32_t)((c + 1) >> 1) & 1u);
        if (all_convert)
          convert_w(c + 1, tid, kEpiThreads);
        else
          convert_w(c + 1, ((warp >> 2) * 2 + (warp & 1)) * 32 + lane, kEpiThreads / 2);
      }

      // ---- a9: H <- e^{gamma_L} H^ + K~^T Delta ----
      bad |= !mbar_wait(&b_s, ph);
      tc_fence_after();
      {
        float z[16], zl[16];
        tmem_ld16_pair(tl + kD2, z, tl + kD2 + 64, zl);
        const float egL = cv[kCvEg + 63];  // gamma is flat past the last valid row
#pragma unroll
        for (int j = 0; j < 16; ++j) hv[j] = hv[j] * egL + (z[j] + zl[j]);
        amax_partial();
      }
      tc_fence_before();
      sH_prev = sH;
    }
    // the last chunk's outputs
    if (!bad && !lo_rows && c == nch && nch > 0) store_out(nch - 1, sH_prev);
    // ---- final state (unquantized) ----
    if (!bad && c == nch && p.ht) {
      float* dst = p.ht + (((int64_t)n * p.Hv + h) * 128 + row) * 128 + vb * 64 + col0;
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(hv[j], hv[j + 1], hv[j + 2], hv[j + 3]);
    }
    if (bad) abort_flag = 1;
  }

  // ---- tear-down: no product or copy may be in flight when TMEM is freed ----
  __syncthreads();
  if (tid == 0 && abort_flag) atomicOr(&g_fused_device_error, 1);
  if (producer && lane == 0) {
    if (abort_flag) {
      // copies still in flight land within the bounded waits
      mbar_wait(&in_q, 0);
      mbar_wait(&in_q, 1);
      for (int bb = 0; bb < 2; ++bb) {
        mbar_wait(&in_vt[bb], 0);
        mbar_wait(&in_kw[bb], 0);
        mbar_wait(&in_cv[bb], 0);
      }
    }
    umma_commit(&b_end);  // completes once every product issued so far is done
    mbar_wait(&b_end, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

gdn_status launch_fused_scan(const FusedParams& p, int state_mode, int w_mode, cudaStream_t st,
                             bool after_prep) {
  const dim3 grid(2, (unsigned)p.Hv, (unsigned)p.N);
  auto run = [&](auto kern) -> gdn_status {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FSmem::BYTES) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
    // programmatic stream serialization: CTAs take the SMs the chunk prep
    // leaves, set up and load their first K and Q, then wait for the prep.
    // Only behind the prep: the inputs read before that wait were written by
    // work that completed before the prep started.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = FSmem::BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prep ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  };
  // the context (P images, state codes) is saved or not: one variant each
  const bool ctx = p.pb != nullptr;
  auto pick = [&](auto with_ctx, auto without) { return ctx ? run(with_ctx) : run(without); };
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_E4M3)
    return pick(gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_E4M3, true>,
                gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_E4M3, false>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_E4M3)
    return pick(gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_E4M3, true>,
                gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_E4M3, false>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_INT8)
    return pick(gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_INT8, true>,
                gdn_fwd_fused_kernel<GDN_QDQ_INT8, GDN_QDQ_INT8, false>);
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_INT8)
    return pick(gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_INT8, true>,
                gdn_fwd_fused_kernel<GDN_QDQ_E4M3, GDN_QDQ_INT8, false>);
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
