// Chunk-parallel gradients of the identity-STE backward (Dk = Dv = 128, both
// QDQ sites on, exact solve) on the Blackwell tensor cores.
//
// Method ("[1/4] GDN state/W QAT foundation", "What does this PR do?": the
// gradient passes through both quantizers unchanged, and the quantized W the
// forward saved is reused).  Per chunk, with the state gradient dH' that the
// reverse scan carried into it (notation as in the reverse scan):
//   P = lower-incl(e^{g_i-g_j} q_i.k_j),  A = diag(beta) strict-lower(e^{g_i-g_j} k_i.k_j)
//   Delta = T diag(beta) V - W^ H^
//   dDelta = scale P^T dO + diag(dec) K dH'
//   dP = lower-incl(scale dO Delta^T);  Gm = dP o Gamma
//   dQ = scale diag(e^g) dO H^T + Gm K
//   dW = -dDelta H^T;   dV = diag(beta) T^T dDelta
//   dT = (dDelta V^T) diag(beta) + (dW K^T) diag(beta e^g);  dA = -T^T dT T^T (strict lower)
//   dK = diag(dec) Delta dH'^T + diag(beta e^g) T^T dW + Gm^T Q + (dKK + dKK^T) K,
//        dKK = diag(beta) dA o Gamma
// and dbeta, dg from the row sums of the chain rule through A, P, W, U and the
// cumulative log decay (dg = reverse cumsum of dgamma).
//
// One CTA of 16 warps per (chunk slot, value head).  P, Gamma o KK^T and Delta
// are recomputed from Q, K, V, the saved T diag(beta) hi / lo images and the W
// and state codes (Delta with the codes' products exact in fp32), so the
// forward saves no P, Gamma o KK^T or Delta tiles.  Every product is an M = 64
// tcgen05 MMA issued by one thread; the seven rounds of products and epilogues
// follow the dependencies of the formulas above:
//   1  S = QK^T, G = KK^T, U = Tu_hi V + Tu_lo V, WH = Wc Hc, KdH = K dH'
//   2  P^T dO, dO Delta^T, Delta dH'^T
//   3  dO H^T, dDelta H^T, dDelta V^T, T^T dDelta
//   4  dW K^T, T^T dW, Gm^T Q
//   5  X = T^T dT;   6  X T^T;   7  Gm K, dKK K, dKK^T K
// Warp w reads accumulator rows 16 (w % 4) .. +15 (its TMEM lane quadrant) and a
// quarter of the columns, in the warp-level mma fragment layout.
#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "bwd_tc.h"
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

namespace {

__device__ int g_bwdtc_device_error;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kTmemCols = 512;

// shared memory (bytes from a 1024-aligned base); tiles are 64-column panels
struct BSmem {
  static constexpr int QS = 0;               // Q [64 tok][128 d]
  static constexpr int KS = QS + 16384;      // K [64 tok][128 d]
  static constexpr int VS = KS + 16384;      // V [64 tok][128 n]
  static constexpr int DOS = VS + 16384;     // dO [64 tok][128 n]
  static constexpr int HB = DOS + 16384;     // H^ [128 d][128 n]: codes, then values
  static constexpr int DH = HB + 32768;      // dH' [128 d][128 n]; then dDelta, Gm
  static constexpr int TU = DH + 32768;      // T diag(beta) hi, lo; then dW [64 tok][128 d]
  static constexpr int WB = TU + 16384;      // W codes [64 tok][128 d]; then dT, X
  static constexpr int DB = WB + 16384;      // Delta [64 tok][128 n]; then dT, X / dKK
  static constexpr int PB = DB + 16384;      // P [64][64]; then Gm
  static constexpr int GK = PB + 8192;       // Gamma o KK^T (strictly lower)
  static constexpr int TB = GK + 8192;       // T
  static constexpr int CV = TB + 8192;       // 2 x chunk vectors (this tile's, the next one's)
  static constexpr int RACC = CV + 2 * kCvecFloats * 4;  // row partial sums [kSlots][64] + scalars
  static constexpr int kSlots = 36;
  static constexpr int BYTES = RACC + kSlots * 256 + 4 * (kWarps + 2) + 1024;
  // aliases (live ranges do not overlap).  The next tile's inputs land in
  // their buffers as these die: W codes after round 1; V, dO, state codes and
  // dH' after round 3; T diag(beta) and Q after round 4; T after round 6; K
  // after round 7.
  static constexpr int DDB = DH;             // dDelta [64 tok][128 n]  (rounds 2-3)
  static constexpr int GMB = PB;             // Gm [64][64]              (rounds 2-7, over P)
  static constexpr int DWB = TU;             // dW [64 tok][128 d]       (rounds 3-4)
  static constexpr int DTB = DB;             // dT [64][64]              (rounds 4-5)
  static constexpr int XB = DB + 8192;       // X = T^T dT               (rounds 5-6)
  static constexpr int DKKB = DB + 8192;     // dKK + dKK^T              (rounds 6-7, over X)
  static constexpr int WC8 = WB + 8192;      // W codes u8 [64][128]     (upper half of W^)
  static constexpr int HC8 = HB + 16384;     // state codes u8 [128][128] (upper half of H^)
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(PB == DB + 16384 && GK == PB + 8192, "the final stores stage 32 KiB from DB");
};

// a tile: one (chunk slot, value head)
struct Tile {
  int64_t ctok, sh;  // first token of the chunk, slot * Hv + h
  int h, hk, Lc;     // value head, key head, valid rows
};

// bytes of the input copies of one chunk
constexpr uint32_t kInTx = 4 * 16384 + 8192 + 16384 + 8192 + 16384 + 32768 + kCvecFloats * 4;

// racc slot indices: four slots per kind (one per column quarter for row sums,
// one per row quarter for column sums); each entry has one writer per round
enum : int {
  R_PPR = 0,   // row sums of dP * P
  R_PPC = 4,   // column sums of dP * P
  R_AAR = 8,   // row sums of dA * A
  R_AAC = 12,  // column sums of dA * A
  R_OH = 16,   // sum_d q_id dQinter_id
  R_TT = 20,   // sum_d k_id dec_i (Delta dH'^T)_id
  R_KW = 24,   // sum_d k_id (T^T dW)_id
  R_BU = 28,   // sum_n v_in (T^T dDelta)_in
  R_BA = 32,   // sum_j dA_ij Gamma_ij KK_ij
};

// row sums of a warp's [16 x 8 NT] fragment tile, added to racc slot `slot`
// (rows r0 = row0 + gq, r0 + 8) by the lanes with tq == 0
template <int NT>
__device__ __forceinline__ void add_row_sums(const float (&x)[NT][4], float* racc, int slot, int row0,
                                             int gq, int tq) {
  float r0 = 0.f, r1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    r0 += x[nt][0] + x[nt][1];
    r1 += x[nt][2] + x[nt][3];
  }
  r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
  r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
  r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
  r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
  if (tq == 0) {
    racc[slot * 64 + row0 + gq] += r0;
    racc[slot * 64 + row0 + gq + 8] += r1;
  }
}
// column sums of a warp's fragment tile (its 16 rows), added to racc slot
// `slot` (columns col0 + 8 nt + 2 tq + e) by the lanes with gq == 0
template <int NT>
__device__ __forceinline__ void add_col_sums(const float (&x)[NT][4], float* racc, int slot, int col0,
                                             int gq, int tq) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float c = x[nt][e] + x[nt][2 + e];
      c += __shfl_xor_sync(0xffffffffu, c, 4);
      c += __shfl_xor_sync(0xffffffffu, c, 8);
      c += __shfl_xor_sync(0xffffffffu, c, 16);
      if (gq == 0) racc[slot * 64 + col0 + 8 * nt + 2 * tq + e] += c;
    }
}

// two bf16 values at a fragment's byte address in a panel tile
__device__ __forceinline__ void st2o(unsigned char* at, float a, float b) {
  *reinterpret_cast<uint32_t*>(at) = pack_bf16(a, b);
}
__device__ __forceinline__ float2 ld2o(const unsigned char* at) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(at));
}

// Stores a warp's [16 x 32] fp32 fragment tile (warp rows gq, gq + 8 and
// columns 8 nt + 2 tq, + 1 of its 32) as whole 128-byte row segments: the
// fragments pass through the warp's 2 KiB of shared memory `stage` (16-byte
// chunks permuted by the row) and leave four rows per instruction.  dst(r) is
// warp row r's first float; rows r >= nrows are not written.
template <typename RowPtr>
__device__ __forceinline__ void store_rows32(float* stage, const float (&v)[4][4], int gq, int tq,
                                             int lane, int nrows, RowPtr dst) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const int r = gq + 8 * e2;
      const int ch = 2 * nt + (tq >> 1);
      *reinterpret_cast<float2*>(stage + r * 32 + ((ch ^ (r & 7)) << 2) + 2 * (tq & 1)) =
          make_float2(v[nt][2 * e2], v[nt][2 * e2 + 1]);
    }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 4 * k + (lane >> 3), ch = lane & 7;
    const float4 x = *reinterpret_cast<const float4*>(stage + r * 32 + ((ch ^ (r & 7)) << 2));
    if (r < nrows) *reinterpret_cast<float4*>(dst(r) + 4 * ch) = x;
  }
  __syncwarp();
}

// D (+)= A B over nk K steps of 16.  K-major operands: `panel` bytes between
// 64-wide K panels (a step moves 32 bytes); MN-major operands: a step moves
// 16 rows (2048 bytes).
__device__ __forceinline__ void mma_steps(uint32_t d, uint64_t a, bool a_mn, uint32_t a_panel,
                                          uint64_t b, bool b_mn, uint32_t b_panel, int nk,
                                          uint32_t id, bool acc) {
  for (int ks = 0; ks < nk; ++ks) {
    const uint32_t ao = a_mn ? ks * 2048u : (ks >> 2) * a_panel + (ks & 3) * 32u;
    const uint32_t bo = b_mn ? ks * 2048u : (ks >> 2) * b_panel + (ks & 3) * 32u;
    umma(d, dadd(a, ao), dadd(b, bo), id, acc || ks > 0);
  }
}

template <int SM, int WM>
__global__ void __launch_bounds__(kThreads, 1) gdn_bwd_chunk_tc_kernel(const __grid_constant__ BwdTcParams p) {
  using S = BSmem;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar_in, bar_mma, bar_end;
  __shared__ uint32_t tmem_slot;
  __shared__ float scl[9];  // the tile's state scales (one per block_v columns), then sW
  __shared__ Tile s_next;   // the next tile (decoded by thread 0 during this one)
  __shared__ long long s_tnext;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, cq = warp >> 2;  // row quadrant (TMEM lanes), column quarter
  const int gq = lane >> 2, tq = lane & 3;
  const int row0 = 16 * q4;                 // this warp's accumulator rows row0 .. row0 + 15
  float* racc = reinterpret_cast<float*>(sm + S::RACC);
  float* hd_part = racc + S::kSlots * 64;  // [kWarps] <H^, dH'> partials, then [2] sums of t_i

  if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
  if (tid == 0) {
    mbar_init(&bar_in, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_end, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tq_base = tmem + ((uint32_t)(32 * q4) << 16);  // this warp's lane quadrant
  const uint32_t sb = smem_u32(sm);
  // byte offsets of this thread's fragment pairs (row row0 + gq, n tile nt) in
  // 64-row panel tiles, for N = 64 (columns 16 cq ..) and N = 128 (32 cq ..)
  // accumulators; row + 8 is 1024 bytes further
  uint32_t fo64[2], fo128[4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) fo64[nt] = pan_off(row0 + gq, 16 * cq + 8 * nt + 2 * tq, 64);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) fo128[nt] = pan_off(row0 + gq, 32 * cq + 8 * nt + 2 * tq, 64);

  // bounded wait on a barrier; on a timeout the error flag is set and the
  // copies / products in flight are waited for once more before teardown
  // (a thread whose wait gave up carries on with garbage; the CTA barrier that
  // ends the round makes the decision uniform, and every thread then leaves)
  bool failed = false;
  auto wait_all = [&](uint64_t* bar, uint32_t parity) {
    if (!mbar_wait(bar, parity)) failed = true;
    tc_fence_after();
  };
  // the round's shared-memory operands are written: make them visible to the
  // tensor cores and order the previous TMEM reads before the next products
  auto publish = [&]() {
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(failed)) failed = true;
    tc_fence_after();
  };

  // ---- tiles: (chunk slot, value head), tile = slot * Hv + h, every gridDim.x-th ----
  const int64_t n_tiles = p.n_slots * p.Hv;
  auto decode = [&](int64_t t, Tile& ti) -> bool {
    const int t32 = (int)t;  // tiles < 2^31 (the launcher checks)
    const int slot = t32 / p.Hv;
    int n, c;
    if (p.cu_seqlens) {
      int lo = 0, hi = p.N - 1;
      while (lo < hi) {  // last n with floor(cu[n] / 64) + n <= slot
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_seqlens[mid] / kChunk + mid <= slot) lo = mid; else hi = mid - 1;
      }
      n = lo;
      c = slot - (p.cu_seqlens[n] / kChunk + n);
    } else {
      n = slot / (int)p.nt_fixed;
      c = slot - n * (int)p.nt_fixed;
    }
    const int64_t tok0 = p.cu_seqlens ? (int64_t)p.cu_seqlens[n] : (int64_t)n * p.T;
    const int L = p.cu_seqlens ? (int)(p.cu_seqlens[n + 1] - tok0) : (int)p.T;
    if (c < 0 || c * kChunk >= L) return false;  // an unused slot
    ti.h = t32 - slot * p.Hv;
    ti.hk = ti.h / p.G;
    ti.Lc = min(L - c * kChunk, kChunk);
    ti.ctok = tok0 + (int64_t)c * kChunk;
    ti.sh = t;
    return true;
  };
  auto next_tile = [&](int64_t from, Tile& ti) -> int64_t {
    for (int64_t t = from; t < n_tiles; t += gridDim.x)
      if (decode(t, ti)) return t;
    return -1;
  };
  // the input copies of tile ti in five groups, each issued (by thread 0) once
  // the current tile no longer reads the buffers it fills; cb: the chunk-vector
  // buffer.  Group 0 opens the barrier's next phase with the whole byte count.
  auto load_group = [&](int g, const Tile& ti, int cb) {
    if (tid != 0) return;
    const int y = (int)ti.ctok;
    const int64_t sh = ti.sh;
    if (g == 0) {
      mbar_expect_tx(&bar_in, kInTx);
      tma_load_2d(sm + S::WC8, &p.tm_wc, ti.h * 128, y, &bar_in);
      bulk_load_1d(sm + S::CV + cb * kCvecFloats * 4, p.cvec + sh * kCvecFloats, kCvecFloats * 4,
                   &bar_in);
    } else if (g == 1) {
#pragma unroll
      for (int pn = 0; pn < 2; ++pn) {
        tma_load_2d(sm + S::VS + pn * 8192, &p.tm_v, ti.h * 128 + pn * 64, y, &bar_in);
        tma_load_2d(sm + S::DOS + pn * 8192, &p.tm_do, ti.h * 128 + pn * 64, y, &bar_in);
      }
      bulk_load_1d(sm + S::HC8, p.h_codes + sh * 16384, 16384, &bar_in);
      bulk_load_1d(sm + S::DH, static_cast<const unsigned char*>(p.ws_dh) + sh * 32768, 32768, &bar_in);
    } else if (g == 2) {
      bulk_load_1d(sm + S::TU, static_cast<const unsigned char*>(p.tu_img) + sh * 16384, 16384, &bar_in);
#pragma unroll
      for (int pn = 0; pn < 2; ++pn)
        tma_load_2d(sm + S::QS + pn * 8192, &p.tm_q, ti.hk * 128 + pn * 64, y, &bar_in);
    } else if (g == 3) {
      bulk_load_1d(sm + S::TB, static_cast<const unsigned char*>(p.tb) + sh * 8192, 8192, &bar_in);
    } else {
#pragma unroll
      for (int pn = 0; pn < 2; ++pn)
        tma_load_2d(sm + S::KS + pn * 8192, &p.tm_k, ti.hk * 128 + pn * 64, y, &bar_in);
    }
  };

  const uint32_t kId64 = idesc(64, 64, 0, 0), kId128KK = idesc(64, 128, 0, 0);
  const uint32_t kId128KM = idesc(64, 128, 0, 1), kId128MM = idesc(64, 128, 1, 1);
  const uint32_t kId64MM = idesc(64, 64, 1, 1);
  auto dsc = [&](int region, uint32_t lbo) { return sdesc(sb + (uint32_t)region, lbo, 1024); };
  uint32_t parity = 0, in_parity = 0;
  auto round_end = [&]() {
    if (tid == 0) umma_commit(&bar_mma);
    wait_all(&bar_mma, parity);
    parity ^= 1u;
  };

  // the scales of tile ti into registers of thread 0 (stored at the tile's start)
  const int nbv = 128 >> p.bv_log2;
  float nscl[9];
  auto load_scales = [&](const Tile& ti) {
    for (int j = 0; j < 8; ++j) nscl[j] = j < nbv ? p.h_scales[ti.sh * nbv + j] : 0.f;
    nscl[8] = p.w_scales[ti.sh];
  };
  Tile cur;
  int64_t t_cur = next_tile(blockIdx.x, cur);
  if (t_cur >= 0 && tid == 0) {
    for (int g = 0; g < 5; ++g) load_group(g, cur, 0);
    load_scales(cur);
  }
  for (int it = 0; t_cur >= 0; ++it) {
    Tile nxt{};
    bool more = false;  // thread 0: there is a next tile (nxt)
    const int cb = it & 1;
    const int h = cur.h, hk = cur.hk, Lc = cur.Lc;
    const int64_t ctok = cur.ctok;
    const float* cvs = reinterpret_cast<const float*>(sm + S::CV + cb * kCvecFloats * 4);
    const float* gam = cvs + kCvGam;
    const float* eg = cvs + kCvEg;
    const float* dec = cvs + kCvDec;
    const float* bet = cvs + kCvBet;
    const float* beg = cvs + kCvBeg;
    (void)hk;
    for (int i = tid; i < S::kSlots * 64 + kWarps + 2; i += kThreads) racc[i] = 0.f;
    if (tid == 0)
      for (int j = 0; j < 9; ++j) scl[j] = nscl[j];

    wait_all(&bar_in, in_parity);
    in_parity ^= 1u;

    // ---- prologue: rows past the chunk end zeroed; W and state codes -> bf16
    //      (the u8 codes sit in the upper halves of their bf16 tiles: all are
    //      read into registers before any is written) ----
    if (Lc < kChunk) {
      for (int i = tid; i < (kChunk - Lc) * 8 * 2; i += kThreads) {
        const int r = Lc + (i >> 4), ch = i & 15;  // 16-byte chunk ch of row r (two panels)
        const uint32_t off = (uint32_t)((ch >> 3) * 8192 + r * 128 + (ch & 7) * 16);
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + S::QS + off) = z;
        *reinterpret_cast<uint4*>(sm + S::KS + off) = z;
        *reinterpret_cast<uint4*>(sm + S::VS + off) = z;
        *reinterpret_cast<uint4*>(sm + S::DOS + off) = z;
      }
    }
    {
      // W codes: thread tid holds row tid / 8, codes 16 (tid % 8) ..; state codes:
      // row tid / 4, codes 32 (tid % 4) ..
      const uint4 wc = *reinterpret_cast<const uint4*>(sm + S::WC8 + 16 * tid);
      const uint4 hc0 = *reinterpret_cast<const uint4*>(sm + S::HC8 + 32 * tid);
      const uint4 hc1 = *reinterpret_cast<const uint4*>(sm + S::HC8 + 32 * tid + 16);
      __syncthreads();
      const int wr = tid >> 3, wcol = (tid & 7) * 16;
      const bool wz = wr >= Lc;  // W codes of rows past the chunk end belong to other tokens
      auto put8 = [&](unsigned char* tile, int rows, int r, int col, uint32_t a, uint32_t b, bool zero,
                      auto mode) {
        constexpr int MODE = decltype(mode)::value;
        const float4 x = qdq_code4_values<MODE>(a), y = qdq_code4_values<MODE>(b);
        *reinterpret_cast<uint4*>(tile + pan_off(r, col, rows)) =
            zero ? make_uint4(0, 0, 0, 0)
                 : make_uint4(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w), pack_bf16(y.x, y.y),
                              pack_bf16(y.z, y.w));
      };
      using WMc = std::integral_constant<int, WM>;
      using SMc = std::integral_constant<int, SM>;
      put8(sm + S::WB, 64, wr, wcol, wc.x, wc.y, wz, WMc{});
      put8(sm + S::WB, 64, wr, wcol + 8, wc.z, wc.w, wz, WMc{});
      const int hr = tid >> 2, hcol = (tid & 3) * 32;
      put8(sm + S::HB, 128, hr, hcol, hc0.x, hc0.y, false, SMc{});
      put8(sm + S::HB, 128, hr, hcol + 8, hc0.z, hc0.w, false, SMc{});
      put8(sm + S::HB, 128, hr, hcol + 16, hc1.x, hc1.y, false, SMc{});
      put8(sm + S::HB, 128, hr, hcol + 24, hc1.z, hc1.w, false, SMc{});
    }
    publish();
    if (failed) goto teardown;

    {
      // =============== round 1: S, G, U, WH, K dH' ===============
      if (tid == 0) {
        mma_steps(tmem + 256, dsc(S::WB, 16), false, 8192, dsc(S::HB, 16384), true, 0, 8, kId128KM, false);
        mma_steps(tmem + 0, dsc(S::QS, 16), false, 8192, dsc(S::KS, 16), false, 8192, 8, kId64, false);
        mma_steps(tmem + 64, dsc(S::KS, 16), false, 8192, dsc(S::KS, 16), false, 8192, 8, kId64, false);
        mma_steps(tmem + 128, dsc(S::TU, 16), false, 0, dsc(S::VS, 8192), true, 0, 4, kId128KM, false);
        mma_steps(tmem + 128, dsc(S::TU + 8192, 16), false, 0, dsc(S::VS, 8192), true, 0, 4, kId128KM,
                  true);
        mma_steps(tmem + 384, dsc(S::KS, 16), false, 8192, dsc(S::DH, 16384), true, 0, 8, kId128KM, false);
        // the next tile (its latency overlaps the products): decode, scales
        const int64_t t_nxt = next_tile(t_cur + gridDim.x, nxt);
        more = t_nxt >= 0;
        s_next = nxt;
        s_tnext = t_nxt;
        if (more) load_scales(nxt);
      }
      round_end();
      if (more) load_group(0, nxt, cb ^ 1);  // W codes, chunk vectors
      {
        // P and Gamma o KK^T (N = 64: columns 16 cq ..)
        float s[2][4], g[2][4];
        tmem_ld_frag_pair<2>(tq_base + 0 + 16 * cq, s, tq_base + 64 + 16 * cq, g);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, j = 16 * cq + 8 * nt + 2 * tq;
            const float gi = gam[i];
            const float x0 = __expf(gi - gam[j]), x1 = __expf(gi - gam[j + 1]);
            st2o(sm + S::PB + fo64[nt] + 1024 * e2, j <= i ? x0 * s[nt][2 * e2] : 0.f,
                j + 1 <= i ? x1 * s[nt][2 * e2 + 1] : 0.f);
            st2o(sm + S::GK + fo64[nt] + 1024 * e2, j < i ? x0 * g[nt][2 * e2] : 0.f,
                j + 1 < i ? x1 * g[nt][2 * e2 + 1] : 0.f);
          }
      }
      {
        // Delta = U - sW sH(n) WH (N = 128: columns 32 cq ..)
        float u[4][4], wh[4][4];
        tmem_ld_frag_pair<4>(tq_base + 128 + 32 * cq, u, tq_base + 256 + 32 * cq, wh);
        const float sW = scl[8];
        const float* hs = scl;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int col = 32 * cq + 8 * nt + 2 * tq;
          const float s0 = sW * hs[col >> p.bv_log2], s1 = sW * hs[(col + 1) >> p.bv_log2];
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            st2o(sm + S::DB + fo128[nt] + 1024 * e2, u[nt][2 * e2] - s0 * wh[nt][2 * e2],
                u[nt][2 * e2 + 1] - s1 * wh[nt][2 * e2 + 1]);
          }
        }
      }
      {
        // state codes -> values (bf16 of code x scale), in place; <H^, dH'>
        float hd = 0.f;
        const float* hs = scl;
        for (int i = tid; i < 2 * 128 * 8; i += kThreads) {
          const int pn = i >> 10, d = (i >> 3) & 127, pc = i & 7;  // panel, row, physical chunk
          const int col = pn * 64 + ((pc ^ (d & 7)) << 3);         // first logical column
          const float sH = hs[col >> p.bv_log2];
          const uint32_t off = (uint32_t)(pn * 16384 + d * 128 + pc * 16);
          uint4 hv = *reinterpret_cast<const uint4*>(sm + S::HB + off);
          const uint4 dv4 = *reinterpret_cast<const uint4*>(sm + S::DH + off);
          uint32_t* hw = &hv.x;
          const uint32_t* dw = &dv4.x;
#pragma unroll
          for (int w2 = 0; w2 < 4; ++w2) {
            const float2 cv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[w2]));
            const float2 dd = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[w2]));
            const float v0 = cv.x * sH, v1 = cv.y * sH;
            hw[w2] = pack_bf16(v0, v1);
            hd += v0 * dd.x + v1 * dd.y;
          }
          *reinterpret_cast<uint4*>(sm + S::HB + off) = hv;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, o);
        if (lane == 0) hd_part[warp] = hd;
      }
      publish();
      if (failed) goto teardown;

      // =============== round 2: P^T dO, dO Delta^T, Delta dH'^T ===============
      if (tid == 0) {
        mma_steps(tmem + 0, dsc(S::PB, 8192), true, 0, dsc(S::DOS, 8192), true, 0, 4, kId128MM, false);
        mma_steps(tmem + 128, dsc(S::DOS, 16), false, 8192, dsc(S::DB, 16), false, 8192, 8, kId64, false);
        mma_steps(tmem + 192, dsc(S::DB, 16), false, 8192, dsc(S::DH, 16), false, 16384, 8, kId128KK,
                  false);
      }
      round_end();
      float dQ[4][4], dK[4][4];
      {
        // dDelta = scale P^T dO + dec K dH'  -> bf16 (dH' is no longer read)
        float a[4][4], b[4][4];
        tmem_ld_frag_pair<4>(tq_base + 0 + 32 * cq, a, tq_base + 384 + 32 * cq, b);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2;
            const float di = dec[i];
            st2o(sm + S::DDB + fo128[nt] + 1024 * e2, p.scale * a[nt][2 * e2] + di * b[nt][2 * e2],
                p.scale * a[nt][2 * e2 + 1] + di * b[nt][2 * e2 + 1]);
          }
      }
      {
        // dP = lower-incl(scale dO Delta^T); Gm = dP o Gamma; sums of dP * P
        float x[2][4], pp[2][4];
        tmem_ld_frag<2>(tq_base + 128 + 16 * cq, x);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, j = 16 * cq + 8 * nt + 2 * tq;
            const float2 pv = ld2o(sm + S::PB + fo64[nt] + 1024 * e2);
            const float gi = gam[i];
            const float d0 = j <= i ? p.scale * x[nt][2 * e2] : 0.f;
            const float d1 = j + 1 <= i ? p.scale * x[nt][2 * e2 + 1] : 0.f;
            st2o(sm + S::GMB + fo64[nt] + 1024 * e2, j <= i ? d0 * __expf(gi - gam[j]) : 0.f,
                j + 1 <= i ? d1 * __expf(gi - gam[j + 1]) : 0.f);
            pp[nt][2 * e2] = d0 * pv.x;
            pp[nt][2 * e2 + 1] = d1 * pv.y;
          }
        add_row_sums<2>(pp, racc, R_PPR + cq, row0, gq, tq);
        add_col_sums<2>(pp, racc, R_PPC + q4, 16 * cq, gq, tq);
      }
      {
        // dK = dec (Delta dH'^T); t_i = sum_d k_id dK_id
        float a[4][4], kd[4][4];
        tmem_ld_frag<4>(tq_base + 192 + 32 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2;
            const float2 kv = ld2o(sm + S::KS + fo128[nt] + 1024 * e2);
            const float di = dec[i];
            dK[nt][2 * e2] = di * a[nt][2 * e2];
            dK[nt][2 * e2 + 1] = di * a[nt][2 * e2 + 1];
            kd[nt][2 * e2] = dK[nt][2 * e2] * kv.x;
            kd[nt][2 * e2 + 1] = dK[nt][2 * e2 + 1] * kv.y;
          }
        add_row_sums<4>(kd, racc, R_TT + cq, row0, gq, tq);
      }
      publish();
      if (failed) goto teardown;

      // =============== round 3: dO H^T, dDelta H^T, dDelta V^T, T^T dDelta ===============
      if (tid == 0) {
        mma_steps(tmem + 0, dsc(S::DOS, 16), false, 8192, dsc(S::HB, 16), false, 16384, 8, kId128KK,
                  false);
        mma_steps(tmem + 128, dsc(S::DDB, 16), false, 8192, dsc(S::HB, 16), false, 16384, 8, kId128KK,
                  false);
        mma_steps(tmem + 256, dsc(S::DDB, 16), false, 8192, dsc(S::VS, 16), false, 8192, 8, kId64, false);
        mma_steps(tmem + 320, dsc(S::TB, 8192), true, 0, dsc(S::DDB, 8192), true, 0, 4, kId128MM, false);
      }
      round_end();
      {
        // dQ = scale e^g (dO H^T); sum_d q_id dQ_id
        float a[4][4], qd[4][4];
        tmem_ld_frag<4>(tq_base + 0 + 32 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2;
            const float2 qv = ld2o(sm + S::QS + fo128[nt] + 1024 * e2);
            const float si = p.scale * eg[i];
            dQ[nt][2 * e2] = si * a[nt][2 * e2];
            dQ[nt][2 * e2 + 1] = si * a[nt][2 * e2 + 1];
            qd[nt][2 * e2] = dQ[nt][2 * e2] * qv.x;
            qd[nt][2 * e2 + 1] = dQ[nt][2 * e2 + 1] * qv.y;
          }
        add_row_sums<4>(qd, racc, R_OH + cq, row0, gq, tq);
      }
      {
        // dW = -dDelta H^T -> bf16 (T diag(beta) is no longer read)
        float a[4][4];
        tmem_ld_frag<4>(tq_base + 128 + 32 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            st2o(sm + S::DWB + fo128[nt] + 1024 * e2, -a[nt][2 * e2], -a[nt][2 * e2 + 1]);
          }
      }
      {
        // dV = beta (T^T dDelta); sum_n v_jn (T^T dDelta)_jn
        float a[4][4], bv[4][4];
        tmem_ld_frag<4>(tq_base + 320 + 32 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int j = row0 + gq + 8 * e2;
            const float2 vv = ld2o(sm + S::VS + fo128[nt] + 1024 * e2);
            bv[nt][2 * e2] = a[nt][2 * e2] * vv.x;
            bv[nt][2 * e2 + 1] = a[nt][2 * e2 + 1] * vv.y;
            a[nt][2 * e2] *= bet[j];
            a[nt][2 * e2 + 1] *= bet[j];
          }
        add_row_sums<4>(bv, racc, R_BU + cq, row0, gq, tq);
        // staging: Delta's tile and the dead half of dH' (8 warps each)
        float* stage = reinterpret_cast<float*>(
            sm + (warp < 8 ? S::DB + 2048 * warp : S::DH + 16384 + 2048 * (warp - 8)));
        store_rows32(stage, a, gq, tq, lane, Lc - row0, [&](int r) {
          return p.dv + ((ctok + row0 + r) * p.Hv + h) * 128 + 32 * cq;
        });
      }
      publish();
      if (failed) goto teardown;

      // =============== round 4: dW K^T, T^T dW, Gm^T Q ===============
      if (more) load_group(1, nxt, cb ^ 1);  // V, dO, state codes, dH'
      if (tid == 0) {
        mma_steps(tmem + 0, dsc(S::DWB, 16), false, 8192, dsc(S::KS, 16), false, 8192, 8, kId64, false);
        mma_steps(tmem + 64, dsc(S::TB, 8192), true, 0, dsc(S::DWB, 8192), true, 0, 4, kId128MM, false);
        mma_steps(tmem + 384, dsc(S::GMB, 8192), true, 0, dsc(S::QS, 8192), true, 0, 4, kId128MM, false);
      }
      round_end();
      if (more) load_group(2, nxt, cb ^ 1);  // T diag(beta), Q
      {
        // dT = (dDelta V^T) diag(beta) + (dW K^T) diag(beta e^g) -> bf16
        float a[2][4], b[2][4];
        tmem_ld_frag_pair<2>(tq_base + 256 + 16 * cq, a, tq_base + 0 + 16 * cq, b);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int j = 16 * cq + 8 * nt + 2 * tq;
            st2o(sm + S::DTB + fo64[nt] + 1024 * e2, a[nt][2 * e2] * bet[j] + b[nt][2 * e2] * beg[j],
                a[nt][2 * e2 + 1] * bet[j + 1] + b[nt][2 * e2 + 1] * beg[j + 1]);
          }
      }
      {
        // dK += beta e^g (T^T dW); sum_d k_id (T^T dW)_id
        float a[4][4], kw[4][4];
        tmem_ld_frag<4>(tq_base + 64 + 32 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2;
            const float2 kv = ld2o(sm + S::KS + fo128[nt] + 1024 * e2);
            dK[nt][2 * e2] += beg[i] * a[nt][2 * e2];
            dK[nt][2 * e2 + 1] += beg[i] * a[nt][2 * e2 + 1];
            kw[nt][2 * e2] = a[nt][2 * e2] * kv.x;
            kw[nt][2 * e2 + 1] = a[nt][2 * e2 + 1] * kv.y;
          }
        add_row_sums<4>(kw, racc, R_KW + cq, row0, gq, tq);
      }
      publish();
      if (failed) goto teardown;

      // =============== round 5: X = T^T dT ===============
      if (tid == 0)
        mma_steps(tmem + 0, dsc(S::TB, 8192), true, 0, dsc(S::DTB, 8192), true, 0, 4, kId64MM, false);
      round_end();
      {
        float a[2][4];
        tmem_ld_frag<2>(tq_base + 0 + 16 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            st2o(sm + S::XB + fo64[nt] + 1024 * e2, a[nt][2 * e2], a[nt][2 * e2 + 1]);
          }
      }
      publish();
      if (failed) goto teardown;

      // =============== round 6: X T^T ===============
      if (tid == 0)
        mma_steps(tmem + 64, dsc(S::XB, 16), false, 0, dsc(S::TB, 16), false, 0, 4, kId64, false);
      round_end();
      if (more) load_group(3, nxt, cb ^ 1);  // T
      {
        // dA = -(X T^T) strictly lower; dKK = dA beta_i Gamma_ij (strictly lower;
        // round 7 reads it and its transpose); sums of dA * Gamma o KK^T and of dA * A
        float a[2][4], ba[2][4], aa[2][4];
        tmem_ld_frag<2>(tq_base + 64 + 16 * cq, a);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, j = 16 * cq + 8 * nt + 2 * tq;
            const float2 gv = ld2o(sm + S::GK + fo64[nt] + 1024 * e2);
            const float gi = gam[i], bi = bet[i];
            float kk[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = j + e;
              const float da = jj < i ? -a[nt][2 * e2 + e] : 0.f;
              const float gkk = e == 0 ? gv.x : gv.y;
              ba[nt][2 * e2 + e] = da * gkk;
              aa[nt][2 * e2 + e] = da * bi * gkk;
              kk[e] = jj < i ? da * bi * __expf(gi - gam[jj]) : 0.f;
            }
            st2o(sm + S::DKKB + fo64[nt] + 1024 * e2, kk[0], kk[1]);
          }
        add_row_sums<2>(ba, racc, R_BA + cq, row0, gq, tq);
        add_row_sums<2>(aa, racc, R_AAR + cq, row0, gq, tq);
        add_col_sums<2>(aa, racc, R_AAC + q4, 16 * cq, gq, tq);
      }
      publish();
      if (failed) goto teardown;

      // =============== round 7: Gm K, (dKK + dKK^T) K ===============
      if (tid == 0) {
        mma_steps(tmem + 128, dsc(S::GMB, 16), false, 0, dsc(S::KS, 8192), true, 0, 4, kId128KM, false);
        mma_steps(tmem + 384, dsc(S::DKKB, 16), false, 0, dsc(S::KS, 8192), true, 0, 4, kId128KM, true);
        mma_steps(tmem + 384, dsc(S::DKKB, 8192), true, 0, dsc(S::KS, 8192), true, 0, 4, kId128MM, true);
      }
      round_end();
      if (more) load_group(4, nxt, cb ^ 1);  // K
      {
        float a[4][4], b[4][4];
        tmem_ld_frag_pair<4>(tq_base + 128 + 32 * cq, a, tq_base + 384 + 32 * cq, b);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dQ[nt][e] += a[nt][e];
            dK[nt][e] += b[nt][e];
          }
        // whole rows through the warp's staging area (Delta / X / dKK, Gm and
        // Gamma o KK^T tiles, all dead now): dq, then dk
        float* stage = reinterpret_cast<float*>(sm + S::DB + 2048 * warp);
        const int head = p.G > 1 ? h : hk;
        store_rows32(stage, dQ, gq, tq, lane, Lc - row0, [&](int r) {
          return p.dq + ((ctok + row0 + r) * p.HH + head) * 128 + 32 * cq;
        });
        store_rows32(stage, dK, gq, tq, lane, Lc - row0, [&](int r) {
          return p.dk + ((ctok + row0 + r) * p.HH + head) * 128 + 32 * cq;
        });
      }
    }

    // ---- dgamma -> dg (reverse cumsum), dbeta (warps 0-1, fixed-order sums) ----
    if (__syncthreads_or(failed)) failed = true;
    if (failed) goto teardown;
    if (warp < 2) {
      const int i = tid;  // row 0..63
      auto sum4 = [&](int s0) {
        return (racc[s0 * 64 + i] + racc[(s0 + 1) * 64 + i]) +
               (racc[(s0 + 2) * 64 + i] + racc[(s0 + 3) * 64 + i]);
      };
      const float rr = sum4(R_PPR), cc = sum4(R_PPC), ar = sum4(R_AAR), ac = sum4(R_AAC);
      const float oh = sum4(R_OH), tt = sum4(R_TT), kw = sum4(R_KW), bu = sum4(R_BU);
      const float ba = sum4(R_BA);
      const float dgam = (rr - cc) + (ar - ac) + oh - tt + beg[i] * kw;
      const float dbeta = bu + eg[i] * kw + ba;
      // gamma_L (row 63) collects e^{gL} <H^, dH'> + sum_i t_i
      float tsum = tt;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
      __syncwarp();
      racc[i] = dgam;  // slot 0 row i: read above by this thread only
      racc[64 + i] = dbeta;
      if (lane == 0) hd_part[kWarps + warp] = tsum;
    }
    __syncthreads();
    if (warp == 0) {
      float hd = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) hd += hd_part[w];
      const float extra = eg[63] * hd + hd_part[kWarps] + hd_part[kWarps + 1];
      const float x1 = racc[2 * lane + 1] + (lane == 31 ? extra : 0.f);
      const float x0 = racc[2 * lane];
      float s = x0 + x1;  // pair sum, then suffix scan over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, s, o);
        if (lane + o < 32) s += y;
      }
      const float dg1 = s - x0, dg0 = s;
      const int64_t base = (ctok + 2 * lane) * p.Hv + h;
      if (2 * lane < Lc) {
        p.dg[base] = dg0;
        p.dbeta[base] = racc[64 + 2 * lane];
      }
      if (2 * lane + 1 < Lc) {
        p.dg[base + p.Hv] = dg1;
        p.dbeta[base + p.Hv] = racc[64 + 2 * lane + 1];
      }
    }
    __syncthreads();
    t_cur = s_tnext;
    cur = s_next;
  }

teardown:
  // after a bounded wait gave up, the next tile's copies may still be in flight;
  // no product may be in flight when TMEM is freed
  if (tid == 0) {
    if (failed) {
      atomicOr(&g_bwdtc_device_error, 1);
      mbar_wait(&bar_in, in_parity ^ 1u);
      mbar_wait(&bar_in, in_parity);
    }
    umma_commit(&bar_end);
    mbar_wait(&bar_end, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

gdn_status launch_bwd_chunk_tc(const BwdTcParams& p, int state_mode, int w_mode, int64_t n_slots,
                               cudaStream_t st) {
  if (n_slots <= 0) return GDN_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return GDN_ERR_CUDA;
  const int64_t tiles = n_slots * p.Hv;
  if (tiles >= ((int64_t)1 << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;  // 32-bit tile indices
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);  // persistent: one CTA per SM
  BwdTcParams q = p;
  q.n_slots = n_slots;
  auto go = [&](auto kern) -> gdn_status {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BSmem::BYTES) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
    kern<<<grid, kThreads, BSmem::BYTES, st>>>(q);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  };
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_E4M3)
    return go(gdn_bwd_chunk_tc_kernel<GDN_QDQ_E4M3, GDN_QDQ_E4M3>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_E4M3)
    return go(gdn_bwd_chunk_tc_kernel<GDN_QDQ_INT8, GDN_QDQ_E4M3>);
  if (state_mode == GDN_QDQ_INT8 && w_mode == GDN_QDQ_INT8)
    return go(gdn_bwd_chunk_tc_kernel<GDN_QDQ_INT8, GDN_QDQ_INT8>);
  if (state_mode == GDN_QDQ_E4M3 && w_mode == GDN_QDQ_INT8)
    return go(gdn_bwd_chunk_tc_kernel<GDN_QDQ_E4M3, GDN_QDQ_INT8>);
  return GDN_ERR_UNSUPPORTED_MODE;
}

int bwd_tc_device_error(bool reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwdtc_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (reset && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_bwdtc_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
