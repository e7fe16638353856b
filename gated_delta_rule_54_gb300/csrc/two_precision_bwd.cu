// Backward of the two-precision GDN profile: the window-wise adjoint ("[5/8]
// ReplaySSM state QAT and two-precision GDN", "What does this PR do?": an FP32
// recurrence anchor, a read copy re-derived from it at every flush, a
// window-wise adjoint in the backward).  The read copy R = Q_read(A) is taken
// through the identity straight-through estimator, so inside a window both
// states follow the ordinary delta-rule step, per column x of H:
//     x' = a x + beta u k,        u = v - a k^T x,        a = e^g
// and the adjoint of one step, for the gradient dx' of x', is
//     sd = k^T dx',   dx = a (dx' - beta sd k)
//     dv += beta sd,  dbeta += u sd,  dk += beta u dx' - a beta sd x
//     da += dx'^T x - beta sd k^T x,  dg = a da
// while o_t = scale R'^T q_t adds scale q_t do_t^T to dR' and scale R' do_t to
// dq_t.  At a window start the read copy's gradient moves to the anchor
// (dA += dR, dR = 0); dA starts as dht and ends as dh0.  With the read
// quantizer off R == A and only the anchor is carried.
//
// Layout as in the forward: a warp owns four value columns over all 128 key
// rows (lane l: rows 4l..4l+3), a CTA four warps (16 columns), and the CTAs of
// the Dv / 16 column groups of one (sequence, head) form a cluster that sums
// the per-token gradients of q, k, beta and g over all columns through
// distributed shared memory, in a fixed order, so every output is written
// once.  The grid is persistent over the (sequence, head) units.  Each window
// is walked twice from the anchor the forward saved at its start:
//   replay:  both states forward through the window, saving them every four
//            tokens and each token's column sums k^T x and u to the CTA's
//            scratch (small enough to stay in L2), and every token's dq;
//   reverse: tokens in reverse; a token's pre-step states are rebuilt from
//            the nearest saved pair (at most three steps), then the step
//            adjoint above.
// Token vectors are staged in shared memory sixteen tokens at a time.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "two_precision.cuh"

namespace gdn {

namespace {

constexpr int kBwWarps = 4;
constexpr int kBwThreads = kBwWarps * 32;
constexpr int kBwCtaCols = kBwWarps * kTpCols;  // value columns per CTA
constexpr int kBwSub = 8;                        // tokens staged at a time (>= the cluster size)
constexpr int kBwCk = 4;                         // tokens between saved states
constexpr int kBwMaxWindow = 256;                // longest window replayed: min(W, T)
constexpr int kBwMaxCtas = 1024;                 // persistent grid (bounds the scratch)
constexpr int kBwCkFloats = 2 * kBwThreads * 16;  // one saved (A, R) pair of a CTA
constexpr int kBwSclFloats = kBwWarps * 16;       // per token: k^T A, k^T R, u_A, u_R per warp

struct TpBwdParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *beta, *g;
  const float* anchors;   // [slots, Hv, 128, Dv] the forward's anchor entering every window
  const float* dout;      // [tokens, Hv, Dv]
  const float* dht;       // [N, Hv, 128, Dv] or null
  float *dq, *dk;         // [tokens, HH, 128]
  float* dv;              // [tokens, Hv, Dv]
  float *dbeta, *dg;      // [tokens, Hv]
  float* dh0;             // [N, Hv, 128, Dv] or null
  float* scratch;         // [CTAs][scratch_floats]
  int64_t scratch_floats;  // per CTA
  int64_t scl_off;         // the per-token sums inside a CTA's scratch
  const int32_t* cu_seqlens;
  int64_t T;
  int Hk, Hv, Dv, N, HH, flush;
  float scale;
};

struct TpBwdSmem {
  float k[kBwSub][kTpDk];
  float q[kBwSub][kTpDk];
  float v[kBwSub][kBwCtaCols];
  float dout[kBwSub][kBwCtaCols];
  float beta[kBwSub];
  float a[kBwSub];
  float scl[kBwSub][kBwSclFloats];
  float red[kBwWarps][kBwSub][kTpDk];  // each warp's dq or dk terms
  float reds[kBwWarps][kBwSub][2];     // each warp's dbeta, dg terms
  float csum[2][kBwSub][kTpDk];        // the CTA's sums, read by its cluster
  float csums[2][kBwSub][2];
};

__device__ __forceinline__ void f8_from_bf16(uint4 u, float* dst) {
  float x[4], y[4];
  bf16x4(make_uint2(u.x, u.y), x);
  bf16x4(make_uint2(u.z, u.w), y);
  *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(y[0], y[1], y[2], y[3]);
}

// Stage nt tokens starting at global token t0: k (and q), the CTA's 16
// columns of v and dO, beta, e^g, and (reverse sweep) the replay's sums.
__device__ __forceinline__ void tp_stage(TpBwdSmem& S, const TpBwdParams& p, int64_t t0, int nt,
                                         int h, int hk, int ccol, bool with_q,
                                         const float* scl_src) {
  const int tid = threadIdx.x;
  for (int i = tid; i < nt * 16; i += kBwThreads) {
    const int jj = i >> 4, ch = i & 15;
    const int64_t row = ((t0 + jj) * p.Hk + hk) * kTpDk;
    f8_from_bf16(__ldg(reinterpret_cast<const uint4*>(p.k + row) + ch), &S.k[jj][ch * 8]);
    if (with_q)
      f8_from_bf16(__ldg(reinterpret_cast<const uint4*>(p.q + row) + ch), &S.q[jj][ch * 8]);
  }
  for (int i = tid; i < nt * 2; i += kBwThreads) {
    const int jj = i >> 1, half = i & 1;
    const int64_t row = ((t0 + jj) * p.Hv + h) * p.Dv + ccol;
    f8_from_bf16(__ldg(reinterpret_cast<const uint4*>(p.v + row) + half), &S.v[jj][half * 8]);
  }
  for (int i = tid; i < nt * 4; i += kBwThreads) {
    const int jj = i >> 2, qd = i & 3;
    const int64_t row = ((t0 + jj) * p.Hv + h) * p.Dv + ccol;
    *reinterpret_cast<float4*>(&S.dout[jj][qd * 4]) =
        __ldg(reinterpret_cast<const float4*>(p.dout + row) + qd);
  }
  if (tid < nt) {
    const int64_t i = (t0 + tid) * p.Hv + h;
    S.beta[tid] = __ldg(p.beta + i);
    S.a[tid] = expf(__ldg(p.g + i));
  }
  if (scl_src) {
    // written earlier by this CTA: read through L2, not the read-only path
    for (int i = tid; i < nt * (kBwSclFloats / 4); i += kBwThreads)
      reinterpret_cast<float4*>(&S.scl[0][0])[i] = __ldcg(reinterpret_cast<const float4*>(scl_src) + i);
  }
}

// The CTA's four warps summed into csum[buf] (and csums with the scalars).
__device__ __forceinline__ void tp_cta_sum(TpBwdSmem& S, int buf, int nt, bool scalars) {
  for (int i = threadIdx.x; i < nt * (kTpDk / 4); i += kBwThreads) {
    const int jj = i / (kTpDk / 4), e = (i % (kTpDk / 4)) * 4;
    float4 s = *reinterpret_cast<const float4*>(&S.red[0][jj][e]);
#pragma unroll
    for (int w = 1; w < kBwWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(&S.red[w][jj][e]);
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    *reinterpret_cast<float4*>(&S.csum[buf][jj][e]) = s;
  }
  if (scalars) {
    for (int i = threadIdx.x; i < nt * 2; i += kBwThreads) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kBwWarps; ++w) s += S.reds[w][i >> 1][i & 1];
      S.csums[buf][i >> 1][i & 1] = s;
    }
  }
}

// After a cluster barrier: this CTA sums its share of the tokens over all the
// cluster's CTAs (rank order) and writes the result.
__device__ __forceinline__ void tp_cluster_sum(TpBwdSmem& S, const TpBwdParams& p, int buf, int nt,
                                               int64_t t0, int h, int hh, float* out,
                                               bool scalars) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int ncta = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int per = kBwSub / ncta;
  const int e = threadIdx.x;
  for (int jj = rank * per; jj < nt && jj < (rank + 1) * per; ++jj) {
    float s = 0.f;
    for (int r = 0; r < ncta; ++r) s += cl.map_shared_rank(&S.csum[buf][jj][0], r)[e];
    out[((t0 + jj) * p.HH + hh) * kTpDk + e] = s;
    if (scalars && e < 2) {
      float x = 0.f;
      for (int r = 0; r < ncta; ++r) x += cl.map_shared_rank(&S.csums[buf][jj][0], r)[e];
      (e == 0 ? p.dbeta : p.dg)[(t0 + jj) * p.Hv + h] = x;
    }
  }
}

// split cluster barrier: a CTA's shared-memory writes before its arrive are
// visible to the cluster after the matching wait
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// a staged block whose column sums the cluster has not yet collected
struct TpPending {
  int64_t t0;
  float* out;
  int nt, h, hh, buf;
  bool scalars, valid;
};

template <int RM>
__global__ void __launch_bounds__(kBwThreads, 4) gdn_two_precision_bwd_kernel(const TpBwdParams p) {
  constexpr bool RQ = RM != GDN_QDQ_NONE;
  constexpr int NF = RQ ? 8 : 4;    // replay sums: k^T A (0..3), k^T R (4..7)
  constexpr int NB = RQ ? 16 : 8;   // reverse sums: k^T dA, [k^T dR], dA^T A, [dR^T R]
  constexpr int LF = 32 / NF, LB = 32 / NB;
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char tp_smem[];
  TpBwdSmem& S = *reinterpret_cast<TpBwdSmem*>(tp_smem);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ccol = blockIdx.x * kBwCtaCols;
  const int c0 = ccol + warp * kTpCols;
  const int G = p.Hv / p.Hk;
  const int W = p.flush;
  float* scr = p.scratch + ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * p.scratch_floats;
  float* sclg = scr + p.scl_off;
  int buf = 0;
  // The cluster sums of a staged block are collected one block later: the
  // CTA sums go to csum[buf] and the CTA arrives on the cluster barrier; at
  // the end of the next block it waits (by then every CTA has arrived), reads
  // the cluster's sums and only then overwrites the other buffer, which every
  // CTA finished reading before that arrival.
  TpPending pend{};
  auto finish_block = [&](int nt, int64_t t0, int h, int hh, float* out, bool scalars) {
    __syncthreads();  // this block's per-warp terms are written
    if (pend.valid) {
      cluster_wait();
      tp_cluster_sum(S, p, pend.buf, pend.nt, pend.t0, pend.h, pend.hh, pend.out, pend.scalars);
    }
    tp_cta_sum(S, buf, nt, scalars);
    cluster_arrive();
    pend = TpPending{t0, out, nt, h, hh, buf, scalars, true};
    buf ^= 1;
  };

  for (int64_t u = blockIdx.y; u < (int64_t)p.Hv * p.N; u += gridDim.y) {
    const int h = (int)(u % p.Hv), n = (int)(u / p.Hv);
    const int hk = h / G;
    const int hh = p.HH == p.Hv ? h : hk;
    int64_t tok0;
    int L;
    if (p.cu_seqlens) {
      tok0 = p.cu_seqlens[n];
      L = (int)(p.cu_seqlens[n + 1] - tok0);
    } else {
      tok0 = (int64_t)n * p.T;
      L = (int)p.T;
    }
    const int64_t sbase = (((int64_t)n * p.Hv + h) * kTpDk + kTpRows * lane) * p.Dv + c0;

    float dA[kTpRows][kTpCols], dR[kTpRows][kTpCols];
#pragma unroll
    for (int r = 0; r < kTpRows; ++r) {
      const float4 x = p.dht ? __ldg(reinterpret_cast<const float4*>(p.dht + sbase + (int64_t)r * p.Dv))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      dA[r][0] = x.x;
      dA[r][1] = x.y;
      dA[r][2] = x.z;
      dA[r][3] = x.w;
#pragma unroll
      for (int c = 0; c < kTpCols; ++c) dR[r][c] = 0.f;
    }

    const int64_t nwin = ((int64_t)L + W - 1) / W;
    const int64_t slot0 = tp_anchor_slot(tok0, n, 0, W);
    for (int64_t w = nwin - 1; w >= 0; --w) {
      const int ts = (int)(w * W);
      const int wl = min(W, L - ts);
      const int64_t tw = tok0 + ts;  // the window's first token

      // ---------------- replay: forward through the window ----------------
      {
        float xA[kTpRows][kTpCols], xR[kTpRows][kTpCols];
        const float* an = p.anchors + ((slot0 + w) * p.Hv + h) * kTpDk * p.Dv +
                          (int64_t)kTpRows * lane * p.Dv + c0;
#pragma unroll
        for (int r = 0; r < kTpRows; ++r) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(an + (int64_t)r * p.Dv));
          xA[r][0] = x.x;
          xA[r][1] = x.y;
          xA[r][2] = x.z;
          xA[r][3] = x.w;
        }
        if constexpr (RQ) tp_read_copy<RM>(xA, xR);

        for (int sb = 0; sb < wl; sb += kBwSub) {
          const int nt = min(kBwSub, wl - sb);
          tp_stage(S, p, tw + sb, nt, h, hk, ccol, false, nullptr);
          __syncthreads();
          for (int jj = 0; jj < nt; ++jj) {
            const int j = sb + jj;
            if ((j & (kBwCk - 1)) == 0) {  // save the pre-step states
              float* ck = scr + (int64_t)(j / kBwCk) * kBwCkFloats + threadIdx.x * 16;
#pragma unroll
              for (int r = 0; r < kTpRows; ++r) {
                __stcg(reinterpret_cast<float4*>(ck) + r, make_float4(xA[r][0], xA[r][1], xA[r][2], xA[r][3]));
                if constexpr (RQ)
                  __stcg(reinterpret_cast<float4*>(ck + kBwThreads * 16) + r,
                         make_float4(xR[r][0], xR[r][1], xR[r][2], xR[r][3]));
              }
            }
            const float4 k4 = *reinterpret_cast<const float4*>(&S.k[jj][kTpRows * lane]);
            const float kr[kTpRows] = {k4.x, k4.y, k4.z, k4.w};
            const float4 v4 = *reinterpret_cast<const float4*>(&S.v[jj][warp * kTpCols]);
            const float vv[kTpCols] = {v4.x, v4.y, v4.z, v4.w};
            const float a = S.a[jj], b = S.beta[jj];
            float x[NF];
#pragma unroll
            for (int c = 0; c < kTpCols; ++c) {
              x[c] = 0.f;
              if constexpr (RQ) x[4 + c] = 0.f;
#pragma unroll
              for (int r = 0; r < kTpRows; ++r) {
                x[c] = fmaf(kr[r], xA[r][c], x[c]);
                if constexpr (RQ) x[4 + c] = fmaf(kr[r], xR[r][c], x[4 + c]);
              }
            }
            const float s = warp_reduce_scatter<NF>(x, lane);
            float sxA[kTpCols], sxR[kTpCols], uA[kTpCols], uR[kTpCols];
#pragma unroll
            for (int c = 0; c < kTpCols; ++c) {
              sxA[c] = __shfl_sync(0xffffffffu, s, c * LF);
              sxR[c] = RQ ? __shfl_sync(0xffffffffu, s, (4 + c) * LF) : sxA[c];
              uA[c] = vv[c] - a * sxA[c];
              uR[c] = vv[c] - a * sxR[c];
            }
            if (lane < 4) {
              float e[kTpCols];
#pragma unroll
              for (int c = 0; c < kTpCols; ++c)
                e[c] = lane == 0 ? sxA[c] : lane == 1 ? sxR[c] : lane == 2 ? uA[c] : uR[c];
              const float4 val = make_float4(e[0], e[1], e[2], e[3]);
              __stcg(reinterpret_cast<float4*>(sclg + ((int64_t)j * kBwWarps + warp) * 16) + lane, val);
            }
            // the step, as in the forward
#pragma unroll
            for (int c = 0; c < kTpCols; ++c)
#pragma unroll
              for (int r = 0; r < kTpRows; ++r) {
                const float bk = b * kr[r];
                xA[r][c] = fmaf(bk, uA[c], a * xA[r][c]);
                if constexpr (RQ) xR[r][c] = fmaf(bk, uR[c], a * xR[r][c]);
              }
            // dq_t = scale R' do_t over this warp's columns
            const float4 d4 = *reinterpret_cast<const float4*>(&S.dout[jj][warp * kTpCols]);
            const float dd[kTpCols] = {d4.x, d4.y, d4.z, d4.w};
            float dq[kTpRows];
#pragma unroll
            for (int r = 0; r < kTpRows; ++r) {
              float t = 0.f;
#pragma unroll
              for (int c = 0; c < kTpCols; ++c) t = fmaf(RQ ? xR[r][c] : xA[r][c], dd[c], t);
              dq[r] = p.scale * t;
            }
            *reinterpret_cast<float4*>(&S.red[warp][jj][kTpRows * lane]) =
                make_float4(dq[0], dq[1], dq[2], dq[3]);
          }
          finish_block(nt, tw + sb, h, hh, p.dq, false);
        }
      }

      // ---------------- reverse sweep ----------------
      const int nsb = (wl + kBwSub - 1) / kBwSub;
      for (int s = nsb - 1; s >= 0; --s) {
        const int sb = s * kBwSub;
        const int nt = min(kBwSub, wl - sb);
        tp_stage(S, p, tw + sb, nt, h, hk, ccol, true, sclg + (int64_t)sb * kBwSclFloats);
        __syncthreads();
        for (int jj = nt - 1; jj >= 0; --jj) {
          const int j = sb + jj;
          const int g0 = j & ~(kBwCk - 1);
          // the pre-step states of token j, rebuilt from the pair saved at g0
          // (read again for every token: fewer live registers)
          float xA[kTpRows][kTpCols], xR[kTpRows][kTpCols];
          {
            const float* ck = scr + (int64_t)(j / kBwCk) * kBwCkFloats + threadIdx.x * 16;
#pragma unroll
            for (int r = 0; r < kTpRows; ++r) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(ck) + r);
              xA[r][0] = x.x;
              xA[r][1] = x.y;
              xA[r][2] = x.z;
              xA[r][3] = x.w;
              if constexpr (RQ) {
                const float4 y = __ldcg(reinterpret_cast<const float4*>(ck + kBwThreads * 16) + r);
                xR[r][0] = y.x;
                xR[r][1] = y.y;
                xR[r][2] = y.z;
                xR[r][3] = y.w;
              }
            }
          }
          for (int i = g0; i < j; ++i) {
            const int ii = i - sb;
            const float4 k4 = *reinterpret_cast<const float4*>(&S.k[ii][kTpRows * lane]);
            const float kr[kTpRows] = {k4.x, k4.y, k4.z, k4.w};
            const float4 ua = *reinterpret_cast<const float4*>(&S.scl[ii][warp * 16 + 8]);
            const float4 ur = *reinterpret_cast<const float4*>(&S.scl[ii][warp * 16 + 12]);
            const float uA[kTpCols] = {ua.x, ua.y, ua.z, ua.w};
            const float uR[kTpCols] = {ur.x, ur.y, ur.z, ur.w};
            const float a = S.a[ii], b = S.beta[ii];
#pragma unroll
            for (int c = 0; c < kTpCols; ++c)
#pragma unroll
              for (int r = 0; r < kTpRows; ++r) {
                const float bk = b * kr[r];
                xA[r][c] = fmaf(bk, uA[c], a * xA[r][c]);
                if constexpr (RQ) xR[r][c] = fmaf(bk, uR[c], a * xR[r][c]);
              }
          }

          const float4 k4 = *reinterpret_cast<const float4*>(&S.k[jj][kTpRows * lane]);
          const float kr[kTpRows] = {k4.x, k4.y, k4.z, k4.w};
          const float4 q4 = *reinterpret_cast<const float4*>(&S.q[jj][kTpRows * lane]);
          const float qs[kTpRows] = {p.scale * q4.x, p.scale * q4.y, p.scale * q4.z, p.scale * q4.w};
          const float4 d4 = *reinterpret_cast<const float4*>(&S.dout[jj][warp * kTpCols]);
          const float dd[kTpCols] = {d4.x, d4.y, d4.z, d4.w};
          const float* sc = &S.scl[jj][warp * 16];
          const float a = S.a[jj], b = S.beta[jj];

          // o_t reads the post-step read state
#pragma unroll
          for (int r = 0; r < kTpRows; ++r)
#pragma unroll
            for (int c = 0; c < kTpCols; ++c) {
              if constexpr (RQ) dR[r][c] = fmaf(qs[r], dd[c], dR[r][c]);
              else dA[r][c] = fmaf(qs[r], dd[c], dA[r][c]);
            }

          float x[NB];
#pragma unroll
          for (int c = 0; c < kTpCols; ++c) {
            float sa = 0.f, pa = 0.f, sr = 0.f, pr = 0.f;
#pragma unroll
            for (int r = 0; r < kTpRows; ++r) {
              sa = fmaf(kr[r], dA[r][c], sa);
              pa = fmaf(dA[r][c], xA[r][c], pa);
              if constexpr (RQ) {
                sr = fmaf(kr[r], dR[r][c], sr);
                pr = fmaf(dR[r][c], xR[r][c], pr);
              }
            }
            if constexpr (RQ) {
              x[c] = sa;
              x[4 + c] = sr;
              x[8 + c] = pa;
              x[12 + c] = pr;
            } else {
              x[c] = sa;
              x[4 + c] = pa;
            }
          }
          const float red = warp_reduce_scatter<NB>(x, lane);
          float sdA[kTpCols], sdR[kTpCols];
#pragma unroll
          for (int c = 0; c < kTpCols; ++c) {
            sdA[c] = __shfl_sync(0xffffffffu, red, c * LB);
            sdR[c] = RQ ? __shfl_sync(0xffffffffu, red, (4 + c) * LB) : 0.f;
          }
          // sum of dx'^T x over the warp's columns (and both states)
          float pt = (lane / LB >= NB / 2 && lane % LB == 0) ? red : 0.f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) pt += __shfl_xor_sync(0xffffffffu, pt, o);

          float dbw = 0.f, daw = pt;
#pragma unroll
          for (int c = 0; c < kTpCols; ++c) {
            const float sxA = sc[c], sxR = sc[4 + c], uA = sc[8 + c], uR = sc[12 + c];
            dbw = fmaf(uA, sdA[c], dbw);
            daw = fmaf(-b * sxA, sdA[c], daw);
            if constexpr (RQ) {
              dbw = fmaf(uR, sdR[c], dbw);
              daw = fmaf(-b * sxR, sdR[c], daw);
            }
          }
          const int64_t tok = tw + j;
          if (lane == 0) {
            *reinterpret_cast<float4*>(p.dv + (tok * p.Hv + h) * p.Dv + c0) =
                make_float4(b * (sdA[0] + sdR[0]), b * (sdA[1] + sdR[1]), b * (sdA[2] + sdR[2]),
                            b * (sdA[3] + sdR[3]));
            S.reds[warp][jj][0] = dbw;
            S.reds[warp][jj][1] = a * daw;
          }
          // dk: beta u dx' - a beta sd x over both states, then the state step back
          float dkr[kTpRows];
#pragma unroll
          for (int r = 0; r < kTpRows; ++r) {
            float t = 0.f;
#pragma unroll
            for (int c = 0; c < kTpCols; ++c) {
              t = fmaf(sc[8 + c], dA[r][c], t);
              t = fmaf(-a * sdA[c], xA[r][c], t);
              if constexpr (RQ) {
                t = fmaf(sc[12 + c], dR[r][c], t);
                t = fmaf(-a * sdR[c], xR[r][c], t);
              }
            }
            dkr[r] = b * t;
          }
          *reinterpret_cast<float4*>(&S.red[warp][jj][kTpRows * lane]) =
              make_float4(dkr[0], dkr[1], dkr[2], dkr[3]);
#pragma unroll
          for (int c = 0; c < kTpCols; ++c)
#pragma unroll
            for (int r = 0; r < kTpRows; ++r) {
              dA[r][c] = a * fmaf(-b * sdA[c], kr[r], dA[r][c]);
              if constexpr (RQ) dR[r][c] = a * fmaf(-b * sdR[c], kr[r], dR[r][c]);
            }
        }
        finish_block(nt, tw + sb, h, hh, p.dk, true);
      }
      // the window's read copy came from the anchor (straight through)
      if constexpr (RQ) {
#pragma unroll
        for (int r = 0; r < kTpRows; ++r)
#pragma unroll
          for (int c = 0; c < kTpCols; ++c) {
            dA[r][c] += dR[r][c];
            dR[r][c] = 0.f;
          }
      }
    }

    if (p.dh0) {
#pragma unroll
      for (int r = 0; r < kTpRows; ++r)
        *reinterpret_cast<float4*>(p.dh0 + sbase + (int64_t)r * p.Dv) =
            make_float4(dA[r][0], dA[r][1], dA[r][2], dA[r][3]);
    }
  }
  if (pend.valid) {
    cluster_wait();
    tp_cluster_sum(S, p, pend.buf, pend.nt, pend.t0, pend.h, pend.hh, pend.out, pend.scalars);
  }
  // the cluster's CTAs read each other's shared memory up to their last sums:
  // none may exit before all are done
  cl.sync();
}

// dq or dk per value head [rows, Hk * G, 128] summed over the G value heads of
// each key head into [rows, Hk, 128]
__global__ void tp_group_sum_kernel(const float4* __restrict__ src, float4* __restrict__ dst,
                                    int64_t n4, int G) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / (kTpDk / 4), e = i % (kTpDk / 4);
    float4 s = src[(row * G) * (kTpDk / 4) + e];
    for (int gi = 1; gi < G; ++gi) {
      const float4 x = src[(row * G + gi) * (kTpDk / 4) + e];
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    dst[i] = s;
  }
}

// Sizes of one backward call.
struct TpBwdPlan {
  int cg, nclu;               // CTAs per cluster (Dv / 16), clusters in the grid
  int64_t scratch_floats;     // per CTA
  int64_t scl_off;
  int64_t scratch_bytes;      // all CTAs
  int64_t group_bytes;        // per-value-head dq and dk (grouped heads), each
  int64_t total;
};

TpBwdPlan tp_bwd_plan(const gdn_two_precision_problem* p) {
  TpBwdPlan pl{};
  pl.cg = p->Dv / kBwCtaCols;
  const int64_t units = (int64_t)p->Hv * p->N;
  pl.nclu = (int)std::min<int64_t>(std::max<int64_t>(units, 1), kBwMaxCtas / pl.cg);
  // no tokens: the kernel only passes dht to dh0 and needs no scratch
  const int64_t wp = p->N * p->B * p->T > 0 ? std::min<int64_t>(p->flush, p->T) : 0;
  const int64_t nck = (wp + kBwCk - 1) / kBwCk;
  pl.scl_off = nck * kBwCkFloats;
  pl.scratch_floats = (pl.scl_off + wp * kBwSclFloats + 63) / 64 * 64;
  pl.scratch_bytes = (int64_t)pl.nclu * pl.cg * pl.scratch_floats * 4;
  const int G = p->Hv / p->Hk;
  pl.group_bytes = G > 1 ? (p->B * p->T * p->Hv * kTpDk * 4 + 255) / 256 * 256 : 0;
  pl.total = pl.scratch_bytes + 2 * pl.group_bytes;
  return pl;
}

gdn_status validate_two_precision_bwd(const gdn_two_precision_problem* p) {
  const gdn_status s = validate_two_precision(p);
  if (s != GDN_OK) return s;
  if (std::min<int64_t>(p->flush, p->T) > kBwMaxWindow) return GDN_ERR_UNSUPPORTED_SHAPE;
  return GDN_OK;
}

template <int RM>
gdn_status launch_tp_bwd_kernel(const TpBwdParams& prm, const TpBwdPlan& pl, cudaStream_t st) {
  auto kern = gdn_two_precision_bwd_kernel<RM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(TpBwdSmem)) != cudaSuccess)
    return GDN_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.cg, (unsigned)pl.nclu, 1);
  cfg.blockDim = dim3(kBwThreads);
  cfg.dynamicSmemBytes = sizeof(TpBwdSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_two_precision_bwd_workspace_bytes(const gdn_two_precision_problem* p) {
  if (validate_two_precision_bwd(p) != GDN_OK) return 0;
  return (size_t)tp_bwd_plan(p).total;
}

gdn_status gdn_two_precision_bwd(const gdn_two_precision_problem* p, const void* q,
                                 const void* k, const void* v, const float* beta,
                                 const float* g, const float* anchors, const float* dO,
                                 const float* dht, float* dq, float* dk, float* dv,
                                 float* dbeta, float* dg, float* dh0, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const gdn_status s = validate_two_precision_bwd(p);
  if (s != GDN_OK) return s;
  const bool tokens = p->B * p->T > 0;
  if (tokens && (!q || !k || !v || !beta || !g || !anchors || !dO || !dq || !dk || !dv ||
                 !dbeta || !dg))
    return GDN_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)beta, (const void*)g, (const void*)anchors,
                          (const void*)dO, (const void*)dht, (const void*)dq, (const void*)dk,
                          (const void*)dv, (const void*)dbeta, (const void*)dg, (const void*)dh0,
                          (const void*)workspace, (const void*)p->cu_seqlens})
    if (ptr && ((uintptr_t)ptr & 15)) return GDN_ERR_MISALIGNED;
  const TpBwdPlan pl = tp_bwd_plan(p);
  if ((int64_t)workspace_bytes < pl.total || (pl.total > 0 && !workspace))
    return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (p->N == 0 || (!tokens && !dh0)) return GDN_OK;

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int G = p->Hv / p->Hk;
  char* ws = static_cast<char*>(workspace);
  TpBwdParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.beta = beta;
  prm.g = g;
  prm.anchors = anchors;
  prm.dout = dO;
  prm.dht = dht;
  prm.dq = G > 1 ? reinterpret_cast<float*>(ws + pl.scratch_bytes) : dq;
  prm.dk = G > 1 ? reinterpret_cast<float*>(ws + pl.scratch_bytes + pl.group_bytes) : dk;
  prm.dv = dv;
  prm.dbeta = dbeta;
  prm.dg = dg;
  prm.dh0 = dh0;
  prm.scratch = reinterpret_cast<float*>(ws);
  prm.scratch_floats = pl.scratch_floats;
  prm.scl_off = pl.scl_off;
  prm.cu_seqlens = p->cu_seqlens;
  prm.T = p->T;
  prm.Hk = p->Hk;
  prm.Hv = p->Hv;
  prm.Dv = p->Dv;
  prm.N = p->N;
  prm.HH = G > 1 ? p->Hv : p->Hk;
  prm.flush = p->flush;
  prm.scale = p->scale;
  const gdn_status ls = p->read_mode == GDN_QDQ_E4M3
                            ? launch_tp_bwd_kernel<GDN_QDQ_E4M3>(prm, pl, st)
                            : launch_tp_bwd_kernel<GDN_QDQ_NONE>(prm, pl, st);
  if (ls != GDN_OK) return ls;
  if (G > 1 && tokens) {
    const int64_t n4 = p->B * p->T * p->Hk * (kTpDk / 4);
    const unsigned blocks = (unsigned)std::min<int64_t>((n4 + 255) / 256, 4096);
    tp_group_sum_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(prm.dq),
                                                reinterpret_cast<float4*>(dq), n4, G);
    tp_group_sum_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(prm.dk),
                                                reinterpret_cast<float4*>(dk), n4, G);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

}  // extern "C"
