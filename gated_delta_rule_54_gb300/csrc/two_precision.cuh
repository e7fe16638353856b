// Pieces shared by the two-precision forward and its backward ("[5/8]
// ReplaySSM state QAT and two-precision GDN", "What does this PR do?"): the
// lane layout of a warp's four value columns, the read copy taken from the
// anchor at a flush, and where the anchor of each window is kept for the
// backward.
#pragma once

#include "common.cuh"

namespace gdn {

constexpr int kTpDk = 128;
constexpr int kTpCols = 4;           // value columns per warp
constexpr int kTpRows = kTpDk / 32;  // key rows per lane (lane l: rows 4l..4l+3)

// R <- Q_read(A) for a warp's four columns of H: one E4M3 scale per column
// over all 128 key rows (a warp max of |A|).  A column whose amax is zero
// passes through.  The forward and the backward's replay both call this, so
// the backward rebuilds the forward's read copy bit for bit from the saved
// anchor.
template <int RM>
__device__ __forceinline__ void tp_read_copy(const float (&A)[kTpRows][kTpCols],
                                             float (&R)[kTpRows][kTpCols]) {
#pragma unroll
  for (int c = 0; c < kTpCols; ++c) {
    float m = 0.f;
#pragma unroll
    for (int r = 0; r < kTpRows; ++r) m = fmaxf(m, fabsf(A[r][c]));
    m = warp_max(m);
    float s, rcp;
    qdq_scale<RM>(m, s, rcp);
#pragma unroll
    for (int r = 0; r < kTpRows; ++r)
      R[r][c] = m == 0.f ? A[r][c] : __fmul_rn(qdq_code_value<RM>(qdq_code<RM>(A[r][c], rcp)), s);
  }
}

// Slot of the anchor entering window w (tokens w*W .. w*W + W - 1 of the
// sequence that starts at token tok0, sequence index n).  Injective over all
// (n, w) of a call, and below tokens / W + N, for packed and batched calls.
__host__ __device__ __forceinline__ int64_t tp_anchor_slot(int64_t tok0, int64_t n, int64_t w,
                                                           int flush) {
  return tok0 / flush + n + w;
}

// Host: checks of a two-precision problem shared by the forward and the
// backward entry points, and the anchor slots of a call (tokens / W + N).
gdn_status validate_two_precision(const gdn_two_precision_problem* p);
int64_t two_precision_anchor_slots(const gdn_two_precision_problem* p);

}  // namespace gdn
