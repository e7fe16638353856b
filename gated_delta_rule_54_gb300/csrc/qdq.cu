// Standalone grouped fake QDQ (E4M3 / INT8) — the primitive behind both
// quantizer sites ("[1/4] GDN state/W QAT foundation", "What does this PR
// do?": dynamic E4M3 fake QDQ; "[2/4] GDN/KDA decode QAT with INT8 recurrent
// state": signed symmetric INT8, rounded reciprocal multiplication).
//
// Three launches on the caller's stream, no scratch: the group amax is
// reduced with atomicMax on the bit pattern of |x| (monotone for
// non-negative floats) into the caller's `scales` buffer, the second pass
// quantizes from it, and the last pass turns each amax into its scale.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

constexpr int kQdqThreads = 256;

struct GroupShape {
  int64_t rows, cols, group_cols, nb, elems;
};

__device__ __forceinline__ int64_t elem_index(const GroupShape& s, int64_t grp, int64_t e) {
  const int64_t b = grp / s.nb, j = grp % s.nb;
  const int64_t r = e / s.group_cols, c = e % s.group_cols;
  return b * s.rows * s.cols + r * s.cols + j * s.group_cols + c;
}

__global__ void __launch_bounds__(kQdqThreads) amax_kernel(const float* __restrict__ x,
                                                           unsigned int* __restrict__ amax_bits,
                                                           GroupShape s, int per) {
  const int64_t grp = blockIdx.x / per;
  const int part = blockIdx.x % per;
  float m = 0.0f;
  for (int64_t e = (int64_t)part * kQdqThreads + threadIdx.x; e < s.elems;
       e += (int64_t)per * kQdqThreads)
    m = fmaxf(m, fabsf(x[elem_index(s, grp, e)]));
  m = warp_max(m);
  __shared__ float red[kQdqThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
#pragma unroll
    for (int i = 1; i < kQdqThreads / 32; ++i) a = fmaxf(a, red[i]);
    atomicMax(amax_bits + grp, __float_as_uint(a));
  }
}

template <int MODE>
__global__ void __launch_bounds__(kQdqThreads) qdq_apply_kernel(const float* x, float* y,
                                                                const unsigned int* amax_bits,
                                                                uint8_t* codes, GroupShape s,
                                                                int per) {
  const int64_t grp = blockIdx.x / per;
  const int part = blockIdx.x % per;
  const float amax = __uint_as_float(amax_bits[grp]);
  float sc, rcp;
  qdq_scale<MODE>(amax, sc, rcp);
  for (int64_t e = (int64_t)part * kQdqThreads + threadIdx.x; e < s.elems;
       e += (int64_t)per * kQdqThreads) {
    const int64_t i = elem_index(s, grp, e);
    const float v = x[i];
    uint8_t c;
    float out;
    if (amax == 0.0f) {
      c = qdq_zero_code<MODE>(v);
      out = v;
    } else {
      c = qdq_code<MODE>(v, rcp);
      out = __fmul_rn(qdq_code_value<MODE>(c), sc);
    }
    y[i] = out;
    if (codes) codes[i] = c;
  }
}

template <int MODE>
__global__ void scale_finalize_kernel(unsigned int* amax_bits_then_scales, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    float sc, rcp;
    qdq_scale<MODE>(__uint_as_float(amax_bits_then_scales[i]), sc, rcp);
    amax_bits_then_scales[i] = __float_as_uint(sc);
  }
}

template <int MODE>
gdn_status run(const float* x, float* y, float* scales, uint8_t* codes, int64_t batch,
               int64_t rows, int64_t cols, int64_t group_cols, cudaStream_t st) {
  GroupShape s;
  s.rows = rows;
  s.cols = cols;
  s.group_cols = group_cols;
  s.nb = cols / group_cols;
  s.elems = rows * group_cols;
  const int64_t groups = batch * s.nb;
  if (groups == 0) return GDN_OK;
  unsigned int* bits = reinterpret_cast<unsigned int*>(scales);
  if (cudaMemsetAsync(bits, 0, sizeof(float) * (size_t)groups, st) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (s.elems > 0) {
    int64_t per = (s.elems + kQdqThreads * 8 - 1) / (kQdqThreads * 8);
    per = per < 1 ? 1 : (per > 64 ? 64 : per);
    if (groups * per > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED_SHAPE;
    const unsigned nblk = (unsigned)(groups * per);
    amax_kernel<<<nblk, kQdqThreads, 0, st>>>(x, bits, s, (int)per);
    qdq_apply_kernel<MODE><<<nblk, kQdqThreads, 0, st>>>(x, y, bits, codes, s, (int)per);
  }
  const int64_t nthreads = 256;
  scale_finalize_kernel<MODE><<<(unsigned)((groups + nthreads - 1) / nthreads), nthreads, 0, st>>>(
      bits, groups);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status launch_fake_qdq(int mode, const float* x, float* y, float* scales, uint8_t* codes,
                           int64_t batch, int64_t rows, int64_t cols, int64_t group_cols,
                           cudaStream_t st) {
  if (mode == GDN_QDQ_E4M3)
    return run<GDN_QDQ_E4M3>(x, y, scales, codes, batch, rows, cols, group_cols, st);
  return run<GDN_QDQ_INT8>(x, y, scales, codes, batch, rows, cols, group_cols, st);
}

}  // namespace gdn
