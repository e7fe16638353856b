// Reverse scan of the state gradient of the identity-STE backward on the
// Blackwell tensor cores (Dk = Dv = 128, W site quantized).
//
// Method ("[1/4] GDN state/W QAT foundation", "What does this PR do?": the
// gradient passes through the quantizers unchanged and reuses the saved
// quantized W).  With dH the gradient w.r.t. the state after chunk c (H = S^T,
// dH' of chunk c), the state entering chunk c gets
//   dDelta = scale P^T dO + diag(dec) K dH
//   dH    <- e^{gamma_L} dH + scale Q^T (diag(e^gamma) dO) - sW Wc^T dDelta
// (Wc the saved W codes, sW their scale; rows past the chunk end contribute
// nothing).  No solve is needed: only P, K, Q, dO and the codes.
//
// One CTA per (sequence, value head) covers both 64-column value blocks (N =
// 128), or, when twice as many CTAs still fit on the SMs at once, one per
// value block (the blocks' chains are independent); it walks the chunks in
// reverse with the fp32 dH in registers (thread r of each warp quadrant holds
// row 32 (w % 4) + lane, a quarter of the columns).  A producer
// warp issues the TMA copies and the tcgen05 products; per chunk only two
// products lie on the dependency chain:
//   C1 = K dH                               (M = 64 tokens, N = 128, K = 128)
//   C2 = Q^T (scale e^gamma dO) + Wc^T dDelta'   (M = 128 = Dk, N = 128, K = 64;
//        dDelta' = -sW dDelta in bf16; the first term is off the chain)
// The W code / dO conversions of a chunk run while its C1 executes, and its
// Q^T product runs while the dDelta epilogue does; P^T dO of the next chunk
// is issued behind the chunk's C2, into the window of the dH update (the
// tensor pipe runs products in issue order, so a product queued ahead of C2
// would delay it).
// The dH' entering each chunk (bf16) leaves by one bulk copy of its 32 KiB
// shared-memory image.
#include <cuda.h>
#include <cuda_bf16.h>

#include "bwd_tc.h"
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

namespace {

__device__ int g_scantc_device_error;

constexpr int kEpiThreads = 512;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kThreads = kEpiThreads + 32;  // + the producer warp

struct SSmem {
  static constexpr int KT = 0;                  // 2 x K [64 tok][128 d]
  static constexpr int QT = KT + 2 * 16384;     // 2 x Q
  static constexpr int DT = QT + 2 * 16384;     // 2 x dO [64 tok][128 n]
  static constexpr int PT = DT + 2 * 16384;     // 2 x P image [64][64]
  static constexpr int WC = PT + 2 * 8192;      // 2 x W codes u8 [64][128]
  static constexpr int WB = WC + 2 * 8192;      // W codes bf16 [64 tok][128 d]
  static constexpr int ED = WB + 16384;         // scale e^gamma dO bf16
  static constexpr int DD = ED + 16384;         // dDelta' bf16 [64 tok][128 n]
  static constexpr int DH = DD + 16384;         // dH bf16 [128 d][128 n] (2 panels)
  static constexpr int CV = DH + 32768;         // 2 x chunk vectors
  static constexpr int BYTES = CV + 2 * kCvecFloats * 4 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
};
// copies of one chunk: K, Q, dO of the CTA's value blocks, P image, W codes, vectors
template <int NB>
__host__ __device__ constexpr uint32_t in_tx() { return 2 * 16384 + NB * 8192 + 8192 + 8192 + kCvecFloats * 4; }

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
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiThreads) : "memory");
}

// NB: 64-column value blocks per CTA (2: one CTA per (sequence, head); 1: two,
// when that many CTAs still fit on the SMs at once)
template <int WM, int NB>
__global__ void __launch_bounds__(kThreads, 1) gdn_bwd_scan_tc_kernel(const __grid_constant__ BwdScanTcParams p) {
  using S = SSmem;
  constexpr int NW = 64 * NB;           // value columns of this CTA
  constexpr int CW = NW / 4;            // dH columns per epilogue thread
  constexpr uint32_t kTmemCols = 4 * NW;
  // TMEM columns: P^T dO (two buffers), K dH, and the state-gradient product
  constexpr uint32_t kA0 = 0, kA1 = 2 * NW, kA2 = 3 * NW;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t in_full[2], dh_ready, conv_done, b_c1, b_q, e_dd, b_c2, b_end;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int h = blockIdx.x / (2 / NB), n = blockIdx.y;
  const int vb0 = NB == 1 ? (blockIdx.x & 1) * 64 : 0;  // first value column
  const int hk = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == kEpiWarps;
  const int q4 = warp & 3, cq = (warp >> 2) & 3;  // lane quadrant, column quarter

  int64_t tok0, slot0;
  int L;
  if (p.cu_seqlens) {
    tok0 = p.cu_seqlens[n];
    L = (int)(p.cu_seqlens[n + 1] - tok0);
    slot0 = tok0 / kChunk + n;
  } else {
    tok0 = (int64_t)n * p.T;
    L = (int)p.T;
    slot0 = (int64_t)n * p.nt_fixed;
  }
  const int nch = (L + kChunk - 1) / kChunk;
  auto KTb = [&](int b) { return sm + S::KT + b * 16384; };
  auto QTb = [&](int b) { return sm + S::QT + b * 16384; };
  auto DTb = [&](int b) { return sm + S::DT + b * 16384; };
  auto PTb = [&](int b) { return sm + S::PT + b * 8192; };
  auto WCb = [&](int b) { return sm + S::WC + b * 8192; };
  auto CVb = [&](int b) { return reinterpret_cast<const float*>(sm + S::CV + b * kCvecFloats * 4); };
  // chunk of iteration it (reverse order), its slot
  auto chunk_of = [&](int it) { return nch - 1 - it; };
  auto sh_of = [&](int it) { return (slot0 + chunk_of(it)) * p.Hv + h; };

  if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
  if (tid == 0) {
    mbar_init(&in_full[0], 1);
    mbar_init(&in_full[1], 1);
    mbar_init(&dh_ready, kEpiWarps);
    mbar_init(&conv_done, kEpiWarps);
    mbar_init(&b_c1, 1);
    mbar_init(&b_q, 1);
    mbar_init(&e_dd, kEpiWarps);
    mbar_init(&b_c2, 1);
    mbar_init(&b_end, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool bad = false;

  if (producer) {
    // ======================= producer warp =======================
    if (lane == 0 && nch > 0) {
      // the copies of iteration it but Q (the barrier expects all bytes), then Q
      auto load_rest = [&](int it) {
        const int b = it & 1;
        const int y = (int)(tok0 + (int64_t)chunk_of(it) * kChunk);
        mbar_expect_tx(&in_full[b], in_tx<NB>());
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_2d(KTb(b) + pn * 8192, &p.tm_k, hk * 128 + pn * 64, y, &in_full[b]);
#pragma unroll
        for (int pn = 0; pn < NB; ++pn)
          tma_load_2d(DTb(b) + pn * 8192, &p.tm_do, h * 128 + vb0 + pn * 64, y, &in_full[b]);
        bulk_load_1d(PTb(b), static_cast<const unsigned char*>(p.pb) + sh_of(it) * 8192, 8192,
                     &in_full[b]);
        tma_load_2d(WCb(b), &p.tm_wc, h * 128, y, &in_full[b]);
        bulk_load_1d(sm + S::CV + b * kCvecFloats * 4, p.cvec + sh_of(it) * kCvecFloats,
                     kCvecFloats * 4, &in_full[b]);
      };
      auto load_q = [&](int it) {
        const int b = it & 1;
        const int y = (int)(tok0 + (int64_t)chunk_of(it) * kChunk);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_2d(QTb(b) + pn * 8192, &p.tm_q, hk * 128 + pn * 64, y, &in_full[b]);
      };
      const uint32_t idPd = idesc(64, NW, 1, 1), idKd = idesc(64, NW, 0, 1);
      const uint32_t idMM = idesc(128, NW, 1, 1);
      // P^T dO of iteration it -> A0[it & 1]
      auto issue_pdo = [&](int it) {
        const int b = it & 1;
        const uint64_t a = sdesc(smem_u32(PTb(b)), 8192, 1024), d = sdesc(smem_u32(DTb(b)), 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma(tmem + kA0 + NW * b, dadd(a, ks * 2048), dadd(d, ks * 2048), idPd, ks > 0);
      };
      load_rest(0);
      load_q(0);
      if (nch > 1) {
        load_rest(1);
        load_q(1);
      }
      bad |= !mbar_wait(&in_full[0], 0);
      tc_fence_after();
      if (!bad) issue_pdo(0);
      for (int it = 0; it < nch && !bad; ++it) {
        const int b = it & 1;
        const uint32_t ph = (uint32_t)it & 1u;
        // C1 = K dH once dH is written (and the previous C2 has been read)
        bad |= !mbar_wait(&dh_ready, ph);
        if (bad) break;
        tc_fence_after();
        {
          const uint64_t k = sdesc(smem_u32(KTb(b)), 16, 1024), g = sdesc(smem_u32(sm + S::DH), 16384, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma(tmem + kA1, dadd(k, (ks >> 2) * 8192 + (ks & 3) * 32), dadd(g, ks * 2048), idKd, ks > 0);
          umma_commit(&b_c1);
        }
        // C2 (first part) = Q^T (scale e^gamma dO) once the conversions (which
        // run while C1 executes) are written
        bad |= !mbar_wait(&conv_done, ph);
        if (bad) break;
        tc_fence_after();
        {
          const uint64_t a = sdesc(smem_u32(QTb(b)), 8192, 1024), e = sdesc(smem_u32(sm + S::ED), 8192, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma(tmem + kA2, dadd(a, ks * 2048), dadd(e, ks * 2048), idMM, ks > 0);
          if (it + 2 < nch) umma_commit(&b_q);  // waited for below, before Q(it + 2) lands here
        }
        // C2 += Wc^T dDelta'
        bad |= !mbar_wait(&e_dd, ph);
        if (bad) break;
        tc_fence_after();
        {
          const uint64_t a = sdesc(smem_u32(sm + S::WB), 8192, 1024), d = sdesc(smem_u32(sm + S::DD), 8192, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma(tmem + kA2, dadd(a, ks * 2048), dadd(d, ks * 2048), idMM, true);
          umma_commit(&b_c2);
        }
        // P^T dO of the next chunk (its A0 buffer was last read two chunks ago),
        // behind C2: it runs while the epilogues update dH
        if (it + 1 < nch) {
          bad |= !mbar_wait(&in_full[b ^ 1], (uint32_t)((it + 1) >> 1) & 1u);
          if (bad) break;
          tc_fence_after();
          issue_pdo(it + 1);
        }
        // this chunk's buffers: C1 and P^T dO of this chunk (issued before C1,
        // so covered by its commit) had read all but Q when the dDelta
        // epilogue signalled; Q is free once Q^T (scale e^gamma dO) is done
        if (it + 2 < nch) {
          load_rest(it + 2);
          bad |= !mbar_wait(&b_q, ph);
          if (!bad) load_q(it + 2);
        }
      }
      if (bad) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ======================= epilogue warps =======================
    const int drow = 32 * q4 + lane;             // dH row (TMEM lane of C2)
    const int c0 = CW * cq;                      // this thread's CW dH columns
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int gq = lane >> 2, tq = lane & 3;
    const int row0 = 16 * q4;                    // rows of the M = 64 products
    float dh[CW];
    {
      const float* src =
          p.dht ? p.dht + (((int64_t)n * p.Hv + h) * 128 + drow) * 128 + vb0 + c0 : nullptr;
#pragma unroll
      for (int j = 0; j < CW; j += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src) x = *reinterpret_cast<const float4*>(src + j);
        dh[j] = x.x;
        dh[j + 1] = x.y;
        dh[j + 2] = x.z;
        dh[j + 3] = x.w;
      }
    }
    // dH (bf16) -> its shared-memory image; one thread then copies the image to
    // the workspace slot of iteration it (the dH' entering that chunk).  The
    // previous copy has read the image: its wait sits in the loop, off the chain.
    auto write_dh = [&](int it) {
      unsigned char* panel = sm + S::DH + (c0 >> 6) * 16384;
#pragma unroll
      for (int k = 0; k < CW / 8; ++k) st8_bf16(panel, drow, ((c0 & 63) >> 3) + k, dh + 8 * k);
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dh_ready);  // C1 may read the image
      epi_sync();
      if (tid == 0) {
        bulk_store_1d(static_cast<unsigned char*>(p.ws_dh) + sh_of(it) * 32768 + (vb0 >> 6) * 16384,
                      sm + S::DH, NB * 16384);
        tma_store_commit();
      }
    };
    if (nch > 0) write_dh(0);
    int it = 0;
    for (; it < nch; ++it) {
      const int b = it & 1;
      const uint32_t ph = (uint32_t)it & 1u;
      const int c = chunk_of(it);
      const int Lc = min(L - c * kChunk, kChunk);
      if (epi_sync_or(bad || *reinterpret_cast<volatile int*>(&abort_flag) != 0)) {
        bad = true;
        break;
      }
      bad |= !mbar_wait(&in_full[b], (uint32_t)(it >> 1) & 1u);
      const float* cv = CVb(b);
      const float sW = p.w_scales[sh_of(it)];
      // ---- conversions: W codes -> bf16; scale e^gamma dO (rows past the end zero) ----
      for (int i = tid; i < 64 * 16; i += kEpiThreads) {
        const int r = i >> 4, c8 = i & 15;
        const uint2 u = *reinterpret_cast<const uint2*>(WCb(b) + r * 128 + c8 * 8);
        const float4 a = qdq_code4_values<WM>(u.x), bb = qdq_code4_values<WM>(u.y);
        *reinterpret_cast<uint4*>(sm + S::WB + pan_off(r, c8 * 8, 64)) =
            make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(bb.x, bb.y), pack_bf16(bb.z, bb.w));
      }
      for (int i = tid; i < NB * 64 * 8; i += kEpiThreads) {
        const int r = (i >> 3) & 63;  // physical chunk i & 7 of row r in panel i >> 9
        const uint32_t off = (uint32_t)((i >> 9) * 8192 + r * 128 + (i & 7) * 16);
        const float er = r < Lc ? p.scale * cv[kCvEg + r] : 0.f;
        const uint4 x = *reinterpret_cast<const uint4*>(DTb(b) + off);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        uint32_t ys[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[k]));
          ys[k] = pack_bf16(er * f.x, er * f.y);
        }
        *reinterpret_cast<uint4*>(sm + S::ED + off) = make_uint4(ys[0], ys[1], ys[2], ys[3]);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv_done);

      // ---- dDelta' = -sW (scale P^T dO + dec K dH) -> bf16 ----
      bad |= !mbar_wait(&b_c1, ph);
      tc_fence_after();
      {
        constexpr int NT = CW / 8;  // n tiles per thread
        float a[NT][4], k[NT][4];
        tmem_ld_frag_pair<NT>(tl + kA0 + NW * b + CW * cq, a, tl + kA1 + CW * cq, k);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int i = row0 + gq + 8 * e2, col = CW * cq + 8 * nt + 2 * tq;
            const float di = i < Lc ? cv[kCvDec + i] : 0.f;
            const float v0 = -sW * (p.scale * a[nt][2 * e2] + di * k[nt][2 * e2]);
            const float v1 = -sW * (p.scale * a[nt][2 * e2 + 1] + di * k[nt][2 * e2 + 1]);
            *reinterpret_cast<uint32_t*>(sm + S::DD + pan_off(i, col, 64)) = pack_bf16(v0, v1);
          }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      // (read before signalling: the producer refills this chunk's buffers then)
      const float egL = cv[kCvEg + 63];  // gamma is flat past the last row
      if (lane == 0) mbar_arrive(&e_dd);
      // while C2 runs: the last bulk copy of the dH image has been read, so the
      // next write_dh may overwrite it
      if (tid == 0) tma_store_wait_read();
      epi_sync();

      // ---- dH <- e^{gamma_L} dH + C2 ----
      bad |= !mbar_wait(&b_c2, ph);
      tc_fence_after();
      {
        if constexpr (NB == 2) {
          float z0[16], z1[16];
          tmem_ld16_pair(tl + kA2 + c0, z0, tl + kA2 + c0 + 16, z1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            dh[j] = egL * dh[j] + z0[j];
            dh[16 + j] = egL * dh[16 + j] + z1[j];
          }
        } else {
          float z0[16];
          tmem_ld16(tl + kA2 + c0, z0);
#pragma unroll
          for (int j = 0; j < 16; ++j) dh[j] = egL * dh[j] + z0[j];
        }
      }
      tc_fence_before();
      if (it + 1 < nch) write_dh(it + 1);
    }
    if (!bad && it == nch && p.dh0) {
      float* dst = p.dh0 + (((int64_t)n * p.Hv + h) * 128 + drow) * 128 + vb0 + c0;
#pragma unroll
      for (int j = 0; j < CW; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(dh[j], dh[j + 1], dh[j + 2], dh[j + 3]);
    }
    if (tid == 0) tma_store_wait_all();  // the workspace copies are complete
    if (bad) abort_flag = 1;
  }

  // ---- tear-down: no product or copy may be in flight when TMEM is freed ----
  __syncthreads();
  if (tid == 0 && abort_flag) atomicOr(&g_scantc_device_error, 1);
  if (producer && lane == 0) {
    if (abort_flag) {
      for (int bb = 0; bb < 2; ++bb) {  // copies still in flight land within the bounded waits
        mbar_wait(&in_full[bb], 0);
        mbar_wait(&in_full[bb], 1);
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

gdn_status launch_bwd_scan_tc(const BwdScanTcParams& p, int w_mode, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return GDN_ERR_CUDA;
  // one CTA per value block while the chains still fit on the SMs at once
  // (each chain is serial: more CTAs on free SMs shorten it), else per head
  const bool split = (int64_t)p.Hv * p.N * 2 <= sms;
  auto run = [&](auto kern, unsigned gx) -> gdn_status {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SSmem::BYTES) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
    kern<<<dim3(gx, (unsigned)p.N), kThreads, SSmem::BYTES, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  };
  const unsigned hv = (unsigned)p.Hv;
  if (w_mode == GDN_QDQ_E4M3)
    return split ? run(gdn_bwd_scan_tc_kernel<GDN_QDQ_E4M3, 1>, 2 * hv)
                 : run(gdn_bwd_scan_tc_kernel<GDN_QDQ_E4M3, 2>, hv);
  if (w_mode == GDN_QDQ_INT8)
    return split ? run(gdn_bwd_scan_tc_kernel<GDN_QDQ_INT8, 1>, 2 * hv)
                 : run(gdn_bwd_scan_tc_kernel<GDN_QDQ_INT8, 2>, hv);
  return GDN_ERR_UNSUPPORTED_MODE;
}

int bwd_scan_tc_device_error(bool reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_scantc_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (reset && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_scantc_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
