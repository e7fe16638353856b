// Shared device helpers for the sm_103a kernels: fake QDQ arithmetic,
// tensor-core fragments, shared-memory swizzle and async copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/gdn_qdq.h"

namespace gdn {

constexpr int kChunk = 64;   // chunk length (first QAT page, "What does this PR do?")
// offsets in the per (chunk, value head) vector record (kCvecFloats floats)
constexpr int kCvGam = 0, kCvEg = 64, kCvDec = 128, kCvBet = 192, kCvBeg = 256;
constexpr int kBlockV = 64;  // state-scale tile width (`state.block_v 64`)

// ---------------------------------------------------------------------------
// Fake QDQ arithmetic (bit-exact with the definition in gdn_qdq.h).
// Compiled without fast-math: '/' and the reciprocal are IEEE correctly
// rounded, and each multiply below is a single rounding (no contraction can
// apply: none of them feeds an add).
// ---------------------------------------------------------------------------
template <int MODE>
struct QdqMax;
template <>
struct QdqMax<GDN_QDQ_E4M3> {
  static constexpr float value = 448.0f;
};
template <>
struct QdqMax<GDN_QDQ_INT8> {
  static constexpr float value = 127.0f;
};

// Scale and its reciprocal from the group amax.  When fl(1/s) is not finite
// (amax == 0, or an amax so small that s = fl(amax / M) is at most 2^-128) the
// group has no usable scale: s = 0 and rcp = 0, so every code is a signed zero
// and every dequantized value is a zero of the input's sign (codes x scale
// still reproduce the values).  Without this, a zero element of such a group
// would give 0 * inf = NaN.
template <int MODE>
__device__ __forceinline__ void qdq_scale(float amax, float& s, float& rcp) {
  s = __fdiv_rn(amax, QdqMax<MODE>::value);
  rcp = __frcp_rn(s);
  if (isinf(rcp)) {
    s = 0.0f;
    rcp = 0.0f;
  }
}

// Code byte of x for scale reciprocal rcp (RNE; E4M3 saturates to finite).
template <int MODE>
__device__ __forceinline__ uint8_t qdq_code(float x, float rcp) {
  const float u = __fmul_rn(x, rcp);
  if constexpr (MODE == GDN_QDQ_E4M3) {
    return (uint8_t)__nv_cvt_float_to_fp8(u, __NV_SATFINITE, __NV_E4M3);
  } else {
    int c = __float2int_rn(u);
    c = c > 127 ? 127 : (c < -127 ? -127 : c);
    return (uint8_t)(int8_t)c;
  }
}

// Value of a code byte (exact in fp32 and in bf16).
template <int MODE>
__device__ __forceinline__ float qdq_code_value(uint8_t c) {
  if constexpr (MODE == GDN_QDQ_E4M3) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(hr));
  } else {
    return (float)(int8_t)c;
  }
}

// Values of four code bytes packed little-endian in c4 (exact in fp32).
template <int MODE>
__device__ __forceinline__ float4 qdq_code4_values(uint32_t c4) {
  if constexpr (MODE == GDN_QDQ_E4M3) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c4 & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c4 >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return make_float4((float)(int8_t)(c4 & 0xffu), (float)(int8_t)((c4 >> 8) & 0xffu),
                       (float)(int8_t)((c4 >> 16) & 0xffu), (float)(int8_t)(c4 >> 24));
  }
}

// For amax == 0 a group passes through unchanged; its codes are signed zeros
// for E4M3 and zeros for INT8.
template <int MODE>
__device__ __forceinline__ uint8_t qdq_zero_code(float x) {
  if constexpr (MODE == GDN_QDQ_E4M3) return signbit(x) ? 0x80 : 0x00;
  return 0;
}

// ---------------------------------------------------------------------------
// Warp / block reductions
// ---------------------------------------------------------------------------
// four / two bf16 (as loaded: little-endian pairs) to fp32
__device__ __forceinline__ void bf16x4(uint2 u, float (&x)[4]) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}
__device__ __forceinline__ void bf16x2(uint32_t u, float (&x)[2]) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  x[0] = a.x;
  x[1] = a.y;
}

// Sum over the 32 lanes of each of NV values (NV = 8 or 16) by halving
// exchanges: at offset o a lane keeps the upper half of its values when its
// bit o is set.  Returns value j = lane / (32 / NV) summed over all lanes
// (identical in the 32 / NV lanes that hold it).
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&x)[NV], int lane) {
  int n = NV;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? x[i] : x[i + n / 2];
          const float keep = up ? x[i + n / 2] : x[i];
          x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      n >>= 1;
    } else {
      x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
    }
  }
  return x[0];
}

// 2^x by the hardware approximation (relative error about 2^-22; subnormal
// results flush to zero)
__device__ __forceinline__ float ex2_approx_f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2eF = 1.4426950408889634f;

// Maximum over the warp of non-negative, non-NaN values (every caller passes
// maxima of |x| seeded with 0): such floats order like their bit patterns, so
// one integer max reduction gives the exact result.
__device__ __forceinline__ float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// ---------------------------------------------------------------------------
// Tensor-core fragments: mma.sync m16n8k16 bf16 x bf16 -> f32.
// A 16x16 row-major, B 16x8 (k x n), C 16x8.  Lane l: g = l/4, t = l%4;
// C holds (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// mma.sync m16n8k32 with E4M3 operands (exact products of E4M3 codes), f32
// accumulation.  Byte geometry of the fragments equals the bf16 m16n8k16
// case with two codes per 16-bit element, so the same ldmatrix addressing
// serves both (k offsets in units of two codes).
__device__ __forceinline__ void mma_e4m3(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// E4M3 codes of (x0, x1) * rcp (each product rounded to fp32 first, then RNE
// with finite saturation), packed low byte = x0, and their exact values.
__device__ __forceinline__ uint16_t e4m3_code2(float x0, float x1, float rcp, float2& val) {
  const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(
      make_float2(__fmul_rn(x0, rcp), __fmul_rn(x1, rcp)), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
  val = __half22float2(__half2(h));
  return (uint16_t)c;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------------------
// bf16 tiles in shared memory.  A tile of 64-element (128-byte) rows keeps
// 16-byte chunk ch of row r at chunk ch ^ (r & 7), so that ldmatrix of 8 rows
// touches 8 distinct bank groups; this is also the layout a TMA copy with
// 128-byte swizzling writes into a 1024-byte aligned tile.  128-element rows
// are stored as two such 64-column panels of 64 rows each (every 128-wide
// tile here has 64 rows), one TMA box per panel.
// ---------------------------------------------------------------------------
template <int RL>
__device__ __forceinline__ int swz(int row, int col) {
  static_assert(RL == 64 || RL == 128, "row length");
  // element offset of (row, col)
  const int in_panel = row * 64 + (((((col >> 3) & 7) ^ (row & 7))) << 3) + (col & 7);
  if constexpr (RL == 64) return in_panel;
  return (col >> 6) * (64 * 64) + in_panel;
}

// fp32 tile of 64 rows x 64 columns as two 32-column panels (128-byte rows,
// 16-byte chunks swizzled like swz): element offset of (row, col).
__device__ __forceinline__ int swz_f32(int row, int col) {
  return (col >> 5) * (64 * 32) + row * 32 + (((((col >> 2) & 7) ^ (row & 7))) << 2) + (col & 3);
}

// ldmatrix.x4 address of a 16x16 A fragment at (r0, c0) of a row-major tile.
template <int RL>
__device__ __forceinline__ uint32_t a_frag_addr(const __nv_bfloat16* base, int r0, int c0,
                                                int lane) {
  const int r = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int c = c0 + (lane >> 4) * 8;
  return smem_u32(base + swz<RL>(r, c));
}

// ldmatrix.x4.trans address of a 16x16 A fragment (rows m0.., cols k0..)
// when the tile stores A transposed (tile row = k, tile col = m).
template <int RL>
__device__ __forceinline__ uint32_t at_frag_addr(const __nv_bfloat16* base, int m0, int k0,
                                                 int lane) {
  const int mi = lane >> 3;
  const int r = k0 + (lane & 7) + (mi >> 1) * 8;
  const int c = m0 + (mi & 1) * 8;
  return smem_u32(base + swz<RL>(r, c));
}

// ldmatrix.x4.trans address for two B fragments (k0..k0+15, n0..n0+15) of a
// tile stored [k][n] (n contiguous): regs {b(n0)[0], b(n0)[1], b(n0+8)[0], b(n0+8)[1]}.
template <int RL>
__device__ __forceinline__ uint32_t bkn_frag_addr(const __nv_bfloat16* base, int k0, int n0,
                                                  int lane) {
  const int mi = lane >> 3;
  const int r = k0 + (lane & 7) + (mi & 1) * 8;
  const int c = n0 + (mi >> 1) * 8;
  return smem_u32(base + swz<RL>(r, c));
}

// ldmatrix.x4 (no trans) address for two B fragments of a tile stored [n][k]
// (k contiguous): regs {b(n0)[0], b(n0)[1], b(n0+8)[0], b(n0+8)[1]}.
template <int RL>
__device__ __forceinline__ uint32_t bnk_frag_addr(const __nv_bfloat16* base, int n0, int k0,
                                                  int lane) {
  const int mi = lane >> 3;
  const int r = n0 + (lane & 7) + (mi >> 1) * 8;
  const int c = k0 + (mi & 1) * 8;
  return smem_u32(base + swz<RL>(r, c));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split x into hi + lo bf16 with hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  lo = x - hi;
}

__device__ __forceinline__ void st_bf16x2(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<uint32_t*>(p) = pack_bf16(a, b);
}

// ---------------------------------------------------------------------------
// Async global -> shared copies (16 bytes; src_bytes == 0 zero-fills).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------------------
// Tensor memory access (TMA) and mbarriers.  One thread issues a copy of a
// whole box; the copy signals the box's bytes on an mbarrier that every
// consumer waits on.  Waits are bounded: after kMbarPolls polls a wait gives
// up and reports it, so a lost transfer ends the kernel with an error status
// instead of hanging the GPU.
// ---------------------------------------------------------------------------
constexpr uint32_t kMbarPolls = 1u << 22;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
// makes mbarrier initialisation visible to the asynchronous (TMA) proxy
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// true once the phase with this parity has completed; false after kMbarPolls polls
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < kMbarPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
// 2-D tiled load of one box at (x = inner element, y = row) into shared memory
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// contiguous bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// 2-D tiled store of one box from shared memory (bulk async-group completion)
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   tmap),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
// shared -> global bulk copy (bulk async-group completion; both addresses
// 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_store_1d(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// the committed stores have finished reading shared memory
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// the committed stores are complete
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
// orders this thread's shared-memory writes before later TMA reads of them
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Programmatic dependent launch.  launch_dependents lets the next kernel of the
// stream, when it was launched with programmatic stream serialization, be
// scheduled before this one ends; grid_dep_wait (a no-op in a kernel launched
// without it) returns once the preceding kernel has completed and its memory
// operations are visible.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

}  // namespace gdn

namespace gdn {

// ---------------------------------------------------------------------------
// Warp-level tile GEMM on tensor cores:
//   acc[NT][4] += A[m0:m0+16, k0:k1] * B[k0:k1, n0:n0+8*NT]      (k in steps of 16)
// A is a row-major [m][k] tile (AT = false) or is stored transposed as [k][m]
// (AT = true); B is stored [k][n] (BKN = true) or [n][k] (BKN = false).
// RLA / RLB are the row lengths (elements) of the swizzled tiles.
// ---------------------------------------------------------------------------
// UNROLL = 2 or 4 unrolls the k loop (the next steps' fragment loads then
// issue ahead of the current step's MMAs).  The default is 1, or the value of
// GDN_WGEMM_UNROLL in a translation unit that defines it before including this
// header: the backward kernels run 7 % faster unrolled by two than not, and
// 1 % faster again by four; the forward kernels choose per call site.
#ifdef GDN_WGEMM_UNROLL
constexpr int kWgemmUnroll = GDN_WGEMM_UNROLL;
#else
constexpr int kWgemmUnroll = 1;
#endif

template <int NT, bool AT, bool BKN, int RLA, int RLB, int UNROLL = kWgemmUnroll>
__device__ __forceinline__ void wgemm(float (&acc)[NT][4], const __nv_bfloat16* A, int m0,
                                      const __nv_bfloat16* B, int n0, int k0, int k1, int lane) {
  static_assert(NT % 2 == 0, "n tiles come in pairs");
  static_assert(UNROLL == 1 || UNROLL == 2 || UNROLL == 4, "unroll factor");
  auto step = [&](int k) {
    uint32_t a[4];
    if constexpr (AT)
      ldsm_x4_t(a, at_frag_addr<RLA>(A, m0, k, lane));
    else
      ldsm_x4(a, a_frag_addr<RLA>(A, m0, k, lane));
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t b[4];
      if constexpr (BKN)
        ldsm_x4_t(b, bkn_frag_addr<RLB>(B, k, n0 + 16 * np, lane));
      else
        ldsm_x4(b, bnk_frag_addr<RLB>(B, n0 + 16 * np, k, lane));
      mma_bf16(acc[2 * np], a, b[0], b[1]);
      mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
    }
  };
  if constexpr (UNROLL == 4) {
#pragma unroll 4
    for (int k = k0; k < k1; k += 16) step(k);
  } else if constexpr (UNROLL == 2) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 16) step(k);
  } else {
    for (int k = k0; k < k1; k += 16) step(k);
  }
}

// Two warp-tile GEMMs that share their A fragments (same A tile, rows m0..,
// k range): acc1 += A * B1[.., n1 : n1 + 8 NT1], acc2 += A * B2[.., n2 : n2 + 8 NT2].
// One A ldmatrix per k step serves both, easing the shared-memory pipe.
template <int NT1, int NT2, bool AT, bool BKN1, bool BKN2, int RLA, int RLB1, int RLB2,
          int UNROLL = kWgemmUnroll>
__device__ __forceinline__ void wgemm_shared_a(float (&acc1)[NT1][4], float (&acc2)[NT2][4],
                                               const __nv_bfloat16* A, int m0,
                                               const __nv_bfloat16* B1, int n1,
                                               const __nv_bfloat16* B2, int n2, int k0, int k1,
                                               int lane) {
  static_assert(NT1 % 2 == 0 && NT2 % 2 == 0, "n tiles come in pairs");
  auto step = [&](int k) {
    uint32_t a[4];
    if constexpr (AT)
      ldsm_x4_t(a, at_frag_addr<RLA>(A, m0, k, lane));
    else
      ldsm_x4(a, a_frag_addr<RLA>(A, m0, k, lane));
#pragma unroll
    for (int np = 0; np < NT1 / 2; ++np) {
      uint32_t b[4];
      if constexpr (BKN1)
        ldsm_x4_t(b, bkn_frag_addr<RLB1>(B1, k, n1 + 16 * np, lane));
      else
        ldsm_x4(b, bnk_frag_addr<RLB1>(B1, n1 + 16 * np, k, lane));
      mma_bf16(acc1[2 * np], a, b[0], b[1]);
      mma_bf16(acc1[2 * np + 1], a, b[2], b[3]);
    }
#pragma unroll
    for (int np = 0; np < NT2 / 2; ++np) {
      uint32_t b[4];
      if constexpr (BKN2)
        ldsm_x4_t(b, bkn_frag_addr<RLB2>(B2, k, n2 + 16 * np, lane));
      else
        ldsm_x4(b, bnk_frag_addr<RLB2>(B2, n2 + 16 * np, k, lane));
      mma_bf16(acc2[2 * np], a, b[0], b[1]);
      mma_bf16(acc2[2 * np + 1], a, b[2], b[3]);
    }
  };
  if constexpr (UNROLL == 4) {
#pragma unroll 4
    for (int k = k0; k < k1; k += 16) step(k);
  } else if constexpr (UNROLL == 2) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 16) step(k);
  } else {
    for (int k = k0; k < k1; k += 16) step(k);
  }
}

// Two warp-tile GEMMs that share their B fragments (same B tile, columns
// n0.., k range) and read A1, A2 (same layout, rows m0..):
// acc1 += A1 * B, acc2 += A2 * B.  acc1 and acc2 may be the same array (the
// hi and lo halves of a split A into one accumulator).
template <int NT, bool AT, bool BKN, int RLA, int RLB, int UNROLL = kWgemmUnroll>
__device__ __forceinline__ void wgemm_shared_b(float (&acc1)[NT][4], float (&acc2)[NT][4],
                                               const __nv_bfloat16* A1, const __nv_bfloat16* A2,
                                               int m0, const __nv_bfloat16* B, int n0, int k0,
                                               int k1, int lane) {
  static_assert(NT % 2 == 0, "n tiles come in pairs");
  auto step = [&](int k) {
    uint32_t a1[4], a2[4];
    if constexpr (AT) {
      ldsm_x4_t(a1, at_frag_addr<RLA>(A1, m0, k, lane));
      ldsm_x4_t(a2, at_frag_addr<RLA>(A2, m0, k, lane));
    } else {
      ldsm_x4(a1, a_frag_addr<RLA>(A1, m0, k, lane));
      ldsm_x4(a2, a_frag_addr<RLA>(A2, m0, k, lane));
    }
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t b[4];
      if constexpr (BKN)
        ldsm_x4_t(b, bkn_frag_addr<RLB>(B, k, n0 + 16 * np, lane));
      else
        ldsm_x4(b, bnk_frag_addr<RLB>(B, n0 + 16 * np, k, lane));
      mma_bf16(acc1[2 * np], a1, b[0], b[1]);
      mma_bf16(acc1[2 * np + 1], a1, b[2], b[3]);
      mma_bf16(acc2[2 * np], a2, b[0], b[1]);
      mma_bf16(acc2[2 * np + 1], a2, b[2], b[3]);
    }
  };
  if constexpr (UNROLL == 4) {
#pragma unroll 4
    for (int k = k0; k < k1; k += 16) step(k);
  } else if constexpr (UNROLL == 2) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 16) step(k);
  } else {
    for (int k = k0; k < k1; k += 16) step(k);
  }
}

// acc += Ah Bh + Ah Bl + Al Bh: the product of two hi + lo split operands to
// ~16 mantissa bits, each fragment loaded once per k step.
template <int NT, bool AT, bool BKN, int RLA, int RLB, int UNROLL = kWgemmUnroll>
__device__ __forceinline__ void wgemm_split3(float (&acc)[NT][4], const __nv_bfloat16* Ah,
                                             const __nv_bfloat16* Al, int m0,
                                             const __nv_bfloat16* Bh, const __nv_bfloat16* Bl,
                                             int n0, int k0, int k1, int lane) {
  static_assert(NT % 2 == 0, "n tiles come in pairs");
  auto step = [&](int k) {
    uint32_t ah[4], al[4];
    if constexpr (AT) {
      ldsm_x4_t(ah, at_frag_addr<RLA>(Ah, m0, k, lane));
      ldsm_x4_t(al, at_frag_addr<RLA>(Al, m0, k, lane));
    } else {
      ldsm_x4(ah, a_frag_addr<RLA>(Ah, m0, k, lane));
      ldsm_x4(al, a_frag_addr<RLA>(Al, m0, k, lane));
    }
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t bh[4], bl[4];
      if constexpr (BKN) {
        ldsm_x4_t(bh, bkn_frag_addr<RLB>(Bh, k, n0 + 16 * np, lane));
        ldsm_x4_t(bl, bkn_frag_addr<RLB>(Bl, k, n0 + 16 * np, lane));
      } else {
        ldsm_x4(bh, bnk_frag_addr<RLB>(Bh, n0 + 16 * np, k, lane));
        ldsm_x4(bl, bnk_frag_addr<RLB>(Bl, n0 + 16 * np, k, lane));
      }
      mma_bf16(acc[2 * np], ah, bh[0], bh[1]);
      mma_bf16(acc[2 * np + 1], ah, bh[2], bh[3]);
      mma_bf16(acc[2 * np], ah, bl[0], bl[1]);
      mma_bf16(acc[2 * np + 1], ah, bl[2], bl[3]);
      mma_bf16(acc[2 * np], al, bh[0], bh[1]);
      mma_bf16(acc[2 * np + 1], al, bh[2], bh[3]);
    }
  };
  if constexpr (UNROLL == 4) {
#pragma unroll 4
    for (int k = k0; k < k1; k += 16) step(k);
  } else if constexpr (UNROLL == 2) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 16) step(k);
  } else {
    for (int k = k0; k < k1; k += 16) step(k);
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
}

// Row stride (floats) of the fp32 [64][64] tiles A and T in shared memory:
// 72 keeps 64-bit accesses of 16 rows conflict free and rows 16-byte aligned.
constexpr int kSA = 72;
constexpr int kF32Tile = 64 * kSA * 4;  // bytes

// ---------------------------------------------------------------------------
// T = (I + A)^-1 for a strictly lower-triangular fp32 A [64][kSA] in shared
// memory, written to Ts (lower triangle and diagonal; the strictly upper part
// of Ts is left undefined).  Blocked forward substitution: the four 16x16
// diagonal blocks row by row (one thread per column, each row of A read as
// four 16-byte loads), then T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32
// T_22, then the lower-left 32x32 block T_LL = -T_LR A_LL T_UL.  The block
// products give each thread four consecutive columns (one 16-byte load of the
// right operand per step) and read their row of the left operand as 16-byte
// loads up front: the solve is bound by shared-memory wavefronts.  The strictly upper part of As is scratch.  All
// NTHREADS threads of the CTA call this; it synchronizes internally and Ts is
// complete on return.
// ---------------------------------------------------------------------------
template <int NTHREADS>
__device__ __forceinline__ void solve_unit_lower64(float* As, float* Ts) {
  static_assert(NTHREADS == 256 || NTHREADS == 512, "thread count");
  static_assert(kSA % 4 == 0, "rows of As, Ts start on 16 bytes");
  const int tid = threadIdx.x;
  // row i of a [*, kSA] fp32 tile, columns c0 .. c0 + 4 N - 1, as N float4 loads
  auto row4 = [](const float* base, int i, int c0, auto n, float* out) {
    constexpr int N = decltype(n)::value;
#pragma unroll
    for (int q = 0; q < N; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(base + i * kSA + c0 + 4 * q);
      out[4 * q] = v.x;
      out[4 * q + 1] = v.y;
      out[4 * q + 2] = v.z;
      out[4 * q + 3] = v.w;
    }
  };
  using I4 = std::integral_constant<int, 4>;
  using I8 = std::integral_constant<int, 8>;
  if (tid < 64) {
    // column cc of the inverse of diagonal block b, row by row: x_r = -sum_{j<r} A_rj x_j
    // (x_j = 0 above the diagonal, x_cc = 1); row r of A read as float4s
    const int b = tid >> 4, cc = tid & 15;
    const float* Ab = As + (16 * b) * kSA + 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int q = 0; q < (r + 3) / 4; ++q) {
        const float4 a = *reinterpret_cast<const float4*>(Ab + r * kSA + 4 * q);
        if (4 * q < r) s0 = fmaf(a.x, x[4 * q], s0);
        if (4 * q + 1 < r) s1 = fmaf(a.y, x[4 * q + 1], s1);
        if (4 * q + 2 < r) s0 = fmaf(a.z, x[4 * q + 2], s0);
        if (4 * q + 3 < r) s1 = fmaf(a.w, x[4 * q + 3], s1);
      }
      x[r] = (r == cc) ? 1.f : ((r < cc) ? 0.f : -(s0 + s1));
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Ts[(16 * b + r) * kSA + 16 * b + cc] = x[r];
  }
  __syncthreads();
  // X = A_10 T_00 -> As[0:16][16:32];  Y = A_32 T_22 -> As[32:48][48:64]
  if (tid < 128) {
    const int base = 32 * (tid >> 6), i = (tid >> 2) & 15, j0 = (tid & 3) * 4;
    float a[16];
    row4(As, base + 16 + i, base, I4{}, a);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 t = *reinterpret_cast<const float4*>(Ts + (base + kk) * kSA + base + j0);
      acc.x = fmaf(a[kk], t.x, acc.x);
      acc.y = fmaf(a[kk], t.y, acc.y);
      acc.z = fmaf(a[kk], t.z, acc.z);
      acc.w = fmaf(a[kk], t.w, acc.w);
    }
    *reinterpret_cast<float4*>(As + (base + i) * kSA + base + 16 + j0) = acc;
  }
  __syncthreads();
  // T_10 = -T_11 X;  T_32 = -T_33 Y
  if (tid < 128) {
    const int base = 32 * (tid >> 6), i = (tid >> 2) & 15, j0 = (tid & 3) * 4;
    float t[16];
    row4(Ts, base + 16 + i, base + 16, I4{}, t);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 x = *reinterpret_cast<const float4*>(As + (base + kk) * kSA + base + 16 + j0);
      acc.x = fmaf(t[kk], x.x, acc.x);
      acc.y = fmaf(t[kk], x.y, acc.y);
      acc.z = fmaf(t[kk], x.z, acc.z);
      acc.w = fmaf(t[kk], x.w, acc.w);
    }
    *reinterpret_cast<float4*>(Ts + (base + 16 + i) * kSA + base + j0) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  // Z = A_LL T_UL -> As[0:32][32:64]; T_UL's upper block T_01 is zero (skipped).
  // A thread computes rows i and i + 16 at four columns: each 16-byte load of
  // T serves both rows.
  if (tid < 128) {
    const int i = tid >> 3, j0 = (tid & 7) * 4;
    const bool upper_cols = j0 >= 16;
    float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // K columns 16 half .. + 15
      if (half == 0 && upper_cols) continue;
      float a0[16], a1[16];
      row4(As, 32 + i, 16 * half, I4{}, a0);
      row4(As, 48 + i, 16 * half, I4{}, a1);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float4 t = *reinterpret_cast<const float4*>(Ts + (16 * half + kk) * kSA + j0);
        c0.x = fmaf(a0[kk], t.x, c0.x);
        c0.y = fmaf(a0[kk], t.y, c0.y);
        c0.z = fmaf(a0[kk], t.z, c0.z);
        c0.w = fmaf(a0[kk], t.w, c0.w);
        c1.x = fmaf(a1[kk], t.x, c1.x);
        c1.y = fmaf(a1[kk], t.y, c1.y);
        c1.z = fmaf(a1[kk], t.z, c1.z);
        c1.w = fmaf(a1[kk], t.w, c1.w);
      }
    }
    *reinterpret_cast<float4*>(As + i * kSA + 32 + j0) = c0;
    *reinterpret_cast<float4*>(As + (i + 16) * kSA + 32 + j0) = c1;
  }
  __syncthreads();
  // T_LL = -T_LR Z; rows i < 16 of T_LR end at column 16 (its upper block is
  // undefined); a thread computes rows i and i + 16
  if (tid < 128) {
    const int i = tid >> 3, j0 = (tid & 7) * 4;
    float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // K rows 16 half .. + 15 of Z
      float t0[16], t1[16];
      if (half == 0) row4(Ts, 32 + i, 32, I4{}, t0);
      row4(Ts, 48 + i, 32 + 16 * half, I4{}, t1);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float4 z = *reinterpret_cast<const float4*>(As + (16 * half + kk) * kSA + 32 + j0);
        if (half == 0) {
          c0.x = fmaf(t0[kk], z.x, c0.x);
          c0.y = fmaf(t0[kk], z.y, c0.y);
          c0.z = fmaf(t0[kk], z.z, c0.z);
          c0.w = fmaf(t0[kk], z.w, c0.w);
        }
        c1.x = fmaf(t1[kk], z.x, c1.x);
        c1.y = fmaf(t1[kk], z.y, c1.y);
        c1.z = fmaf(t1[kk], z.z, c1.z);
        c1.w = fmaf(t1[kk], z.w, c1.w);
      }
    }
    *reinterpret_cast<float4*>(Ts + (32 + i) * kSA + j0) = make_float4(-c0.x, -c0.y, -c0.z, -c0.w);
    *reinterpret_cast<float4*>(Ts + (48 + i) * kSA + j0) = make_float4(-c1.x, -c1.y, -c1.z, -c1.w);
  }
  __syncthreads();
}

}  // namespace gdn
