/*
 * Oracle O1: token-by-token gated delta rule recurrence, plain C, fp64.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).
 *
 * The recurrence is the gated delta rule that GatedDeltaNet trains ("[1/4]
 * GDN state/W QAT foundation", section "What does this PR do?": exact
 * recurrent references), in the published form
 *     S_t = a_t * S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t
 * with a_t = exp(g_t).  It is written here for H = S^T (Dk x Dv), which is
 * the same thing transposed:
 *     H <- exp(g_t) * H
 *     H <- H + b_t * k_t (v_t - H^T k_t)^T
 *     o_t = scale * H^T q_t
 * (expanding the first form: a(I - b k k^T)H' + b k v^T = aH' + b k (v - aH'^T k)^T.)
 *
 * State fake QDQ ("[1/4]" page, Usage: `gdn_state_quantizer`, `state.block_v
 * 64`; "[2/4]" page: per-head [Dk, block_v] scales): at every chunk boundary
 * of the chunked form, i.e. before token t of a sequence with t % chunk == 0
 * (t = 0 included, so the initial state is quantized too), every [Dk,
 * block_v] column tile of H is rounded to fp32, quantized with the fp32 QDQ
 * of qdq.c, and the dequantized values replace the carried state.  The final
 * state returned is not quantized.  The W site has no counterpart in a token
 * recurrence; the chunked oracle covers it.
 *
 * Value head h reads query/key head h / (Hv / Hk).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_qdq_groups(const float* x, float* y, float* scales, uint8_t* codes,
                      int64_t batch, int64_t rows, int64_t cols, int64_t group_cols,
                      int mode);

/*
 * Shapes: q, k [B, T, Hk, Dk]; v [B, T, Hv, Dv]; beta, g [B, T, Hv] (all
 * fp32 values, bf16 inputs widened exactly).  cu_seqlens (nullable) has N+1
 * offsets into the token axis of a B == 1 batch; without it N == B and every
 * sequence has T tokens.  h0 [N, Hv, Dk, Dv] fp32 (nullable = zeros).
 * Outputs: o [B, T, Hv, Dv] fp64, ht [N, Hv, Dk, Dv] fp64 (nullable).
 * If state_codes / state_scales are given, the quantized state entering each
 * chunk is recorded at chunk index chunk_base[n] + c:
 *   state_codes  [n_chunks, Hv, Dk, Dv] code bytes
 *   state_scales [n_chunks, Hv, Dv / block_v]
 * Returns 0, or -1 on bad arguments.
 */
int oracle_gdn_recurrent(const float* q, const float* k, const float* v, const float* beta,
                         const float* g, const float* h0, const int32_t* cu_seqlens, int B,
                         int T, int Hk, int Hv, int Dk, int Dv, int N, double scale,
                         int state_mode, int block_v, int chunk, double* o, double* ht,
                         uint8_t* state_codes, float* state_scales, const int64_t* chunk_base,
                         int n_threads) {
  if (!q || !k || !v || !beta || !g || !o || Hk <= 0 || Hv % Hk != 0 || Dk <= 0 || Dv <= 0 ||
      chunk <= 0 || (state_mode != 0 && (block_v <= 0 || Dv % block_v != 0)))
    return -1;
  if (cu_seqlens ? (B != 1) : (N != B)) return -1;
  if ((state_codes || state_scales) && !chunk_base) return -1;
  const int G = Hv / Hk;
  const int nvb = state_mode ? Dv / block_v : 1;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t nh = 0; nh < (int64_t)N * Hv; ++nh) {
    const int n = (int)(nh / Hv), h = (int)(nh % Hv), hk = h / G;
    int64_t t0, L, b;
    if (cu_seqlens) {
      t0 = cu_seqlens[n];
      L = (int64_t)cu_seqlens[n + 1] - cu_seqlens[n];
      b = 0;
    } else {
      t0 = 0;
      L = T;
      b = n;
    }
    double* H = (double*)malloc(sizeof(double) * (size_t)Dk * Dv);
    double* u = (double*)malloc(sizeof(double) * (size_t)Dv);
    float* hf = (float*)malloc(sizeof(float) * (size_t)Dk * Dv);
    float* hq = (float*)malloc(sizeof(float) * (size_t)Dk * Dv);
    float* sc = (float*)malloc(sizeof(float) * (size_t)nvb);
    uint8_t* cd = (uint8_t*)malloc((size_t)Dk * Dv);
    if (!H || !u || !hf || !hq || !sc || !cd) {
#pragma omp atomic write
      bad = 1;
      free(H); free(u); free(hf); free(hq); free(sc); free(cd);
      continue;
    }
    for (int64_t i = 0; i < (int64_t)Dk * Dv; ++i)
      H[i] = h0 ? (double)h0[((int64_t)n * Hv + h) * Dk * Dv + i] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t tok = (int64_t)b * T + t0 + t;
      if (state_mode != 0 && t % chunk == 0) {
        for (int64_t i = 0; i < (int64_t)Dk * Dv; ++i) hf[i] = (float)H[i];
        oracle_qdq_groups(hf, hq, sc, cd, 1, Dk, Dv, block_v, state_mode);
        for (int64_t i = 0; i < (int64_t)Dk * Dv; ++i) H[i] = (double)hq[i];
        if (state_codes || state_scales) {
          int64_t ci = chunk_base[n] + t / chunk;
          if (state_codes) memcpy(state_codes + (ci * Hv + h) * Dk * Dv, cd, (size_t)Dk * Dv);
          if (state_scales)
            for (int j = 0; j < nvb; ++j) state_scales[(ci * Hv + h) * nvb + j] = sc[j];
        }
      }
      const float* kt = k + (tok * Hk + hk) * Dk;
      const float* qt = q + (tok * Hk + hk) * Dk;
      const float* vt = v + (tok * Hv + h) * Dv;
      const double a = exp((double)g[tok * Hv + h]);
      const double bt = (double)beta[tok * Hv + h];
      for (int64_t i = 0; i < (int64_t)Dk * Dv; ++i) H[i] *= a;
      /* u = v_t - H^T k_t */
      for (int j = 0; j < Dv; ++j) u[j] = 0.0;
      for (int i = 0; i < Dk; ++i) {
        const double ki = (double)kt[i];
        const double* Hi = H + (int64_t)i * Dv;
        for (int j = 0; j < Dv; ++j) u[j] += Hi[j] * ki;
      }
      for (int j = 0; j < Dv; ++j) u[j] = (double)vt[j] - u[j];
      for (int i = 0; i < Dk; ++i) {
        const double bk = bt * (double)kt[i];
        for (int j = 0; j < Dv; ++j) H[(int64_t)i * Dv + j] += bk * u[j];
      }
      /* o_t = scale * H^T q_t */
      double* ot = o + (tok * Hv + h) * Dv;
      for (int j = 0; j < Dv; ++j) u[j] = 0.0;
      for (int i = 0; i < Dk; ++i) {
        const double qi = (double)qt[i];
        const double* Hi = H + (int64_t)i * Dv;
        for (int j = 0; j < Dv; ++j) u[j] += Hi[j] * qi;
      }
      for (int j = 0; j < Dv; ++j) ot[j] = scale * u[j];
    }
    if (ht)
      memcpy(ht + ((int64_t)n * Hv + h) * Dk * Dv, H, sizeof(double) * (size_t)Dk * Dv);
    free(H); free(u); free(hf); free(hq); free(sc); free(cd);
  }
  return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
