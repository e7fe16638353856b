// Blackwell tensor-core helpers shared by the tcgen05 kernels: shared-memory
// matrix descriptors, the kind::f16 instruction descriptor, MMA issue and
// commit, tensor-memory (TMEM) allocation and loads, and the 128-byte-swizzled
// tile layout the descriptors read.
//
// Tile layout ("panels"): a bf16 tile of R rows x C columns is stored as C/64
// panels of R rows x 128 bytes; in each row the eight 16-byte chunks are
// permuted by chunk ^ (row & 7), and 8-row groups are 1024 bytes apart.  This
// is the 128-byte swizzle that TMA writes for a 64-column box.  The same bytes
// serve as a K-major operand (rows = M or N, columns = K: a K step of 16 moves
// 32 bytes inside the panel, every fourth step moves to the next panel) and as
// an MN-major operand (rows = K, columns = M or N: a K step moves 16 rows =
// 2048 bytes; the panels are the 64-wide M/N blocks, LBO = panel bytes).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gdn {

// shared-memory matrix descriptor: 128-byte swizzle, 8-row groups SBO apart,
// LBO = distance between 64-element blocks along M/N (MN-major operands)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor, kind::f16: bf16 x bf16 -> f32, M x N, operand majors
// (a_mn / b_mn = 1: the operand is stored M- / N-contiguous)
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// descriptor of the tile at smem address saddr + off: only the start-address
// field moves (offsets keep the tile inside the 256 KB shared window)
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t off) { return desc + (off >> 4); }

// D[tmem] (+)= A B, issued by one thread
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc));
}
// the mbarrier receives one arrival when every product issued so far by this
// thread has completed
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
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// TMEM allocation by one whole warp: the base address goes to *slot
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(slot)),
               "r"(cols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(cols));
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape)
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

// Two 16-column loads (32x32b shape) under one wait.
__device__ __forceinline__ void tmem_ld16_pair(uint32_t ta, float (&va)[16], uint32_t tb,
                                               float (&vb)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,"
      "%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[16 + i]);
  }
}

// Accumulator fragments of an M = 64 product (row r of D in TMEM lane
// 32 (r / 16) + r % 16): the warp of lane quadrant q reads rows 16 q .. 16 q + 15
// and NT x 8 columns from column c0 (16x256b shape).  Fragment layout, as the
// warp-level mma accumulators: v[nt][e] is row 16 q + (lane >> 2) + 8 (e >> 1),
// column c0 + 8 nt + 2 (lane & 3) + (e & 1).
template <int NT>
__device__ __forceinline__ void tmem_ld_frag(uint32_t taddr, float (&v)[NT][4]) {
  static_assert(NT == 2 || NT == 4, "n tiles per load");
  if constexpr (NT == 2) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i >> 2][i & 3] = __uint_as_float(r[i]);
  } else {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i >> 2][i & 3] = __uint_as_float(r[i]);
  }
}

// Two accumulator fragment loads (same shape as tmem_ld_frag) under one wait.
template <int NT>
__device__ __forceinline__ void tmem_ld_frag_pair(uint32_t ta, float (&va)[NT][4], uint32_t tb,
                                                  float (&vb)[NT][4]) {
  static_assert(NT == 2 || NT == 4, "n tiles per load");
  if constexpr (NT == 2) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n"
        "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      va[i >> 2][i & 3] = __uint_as_float(r[i]);
      vb[i >> 2][i & 3] = __uint_as_float(r[8 + i]);
    }
  } else {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%32];\n"
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
        "%28,%29,%30,%31}, [%33];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      va[i >> 2][i & 3] = __uint_as_float(r[i]);
      vb[i >> 2][i & 3] = __uint_as_float(r[16 + i]);
    }
  }
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

// byte offset of element (row, col) in one panel (128-byte rows, 64 bf16)
__device__ __forceinline__ uint32_t sw_off(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2);
}
// byte offset of (row, col) in a tile of `rows` rows stored as 64-column panels
__device__ __forceinline__ uint32_t pan_off(int row, int col, int rows) {
  return (uint32_t)((col >> 6) * rows * 128) + sw_off(row, col & 63);
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

}  // namespace gdn
