/*
 * Oracle: dynamic fake quantize-dequantize (QDQ), plain C, fp32, bit-exact.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file; only tests, the smoke check and the CPU baseline of the
 * benchmark do.
 *
 * What it computes (GatedDeltaNet state/W QAT pages):
 *   - "[1/4] GDN state/W QAT foundation", section "What does this PR do?":
 *     dynamic FP8 E4M3 fake QDQ at the state and W sites, identity STE;
 *     the quantizer config `num_bits: (4, 3), type: dynamic` (section Usage).
 *   - "[2/4] GDN/KDA decode QAT with INT8 recurrent state", section
 *     "What does this PR do?": signed symmetric dynamic INT8, zero point
 *     zero, codes in [-127, 127], round to nearest even; section Testing:
 *     scale arithmetic is the rounded reciprocal multiplication that Torch
 *     scalar division performs (x * fl(1/s)), not a true division.
 *
 * For one group of fp32 values x:
 *   a   = max_i |x_i|                       (exact)
 *   if a == 0: scale = 0, y = x, codes are signed zeros
 *   s   = fl(a / M)      M = 448 (E4M3) or 127 (INT8), correctly rounded
 *   r   = fl(1 / s)      correctly rounded
 *   if r is not finite (a tiny nonzero a: s at most 2^-128, where binary32
 *       cannot hold 1/s), the pages give no scale to use; this oracle reads
 *       it as a group scaled to zero: s = 0 and r = 0, and the steps below
 *       then give signed-zero codes and y = fl(decode(c) * 0).  Taking r = inf
 *       literally would turn a zero element into 0 * inf = NaN.
 *   u_i = fl(x_i * r)
 *   c_i = E4M3: round-to-nearest-even onto the OCP E4M3FN grid, finite
 *               values beyond 448 saturate to +-448 (sign kept, -0 kept)
 *         INT8: nearest integer, ties to even, clamped to [-127, 127]
 *   y_i = fl(decode(c_i) * s)
 *
 * The E4M3 grid is written from the format definition (1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
 * NaN, largest finite value 1.75 * 2^8 = 448, subnormal step 2^-9), not from
 * any conversion routine.
 *
 * Compile with -ffp-contract=off and without -ffast-math: every operation
 * here must be a single IEEE-754 binary32 operation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_QDQ_NONE 0
#define ORACLE_QDQ_E4M3 1
#define ORACLE_QDQ_INT8 2

/* Value of an E4M3FN code byte, from the bit fields. */
float oracle_e4m3_decode(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  float val;
  if (e == 0xF && m == 0x7) {
    val = NAN;
  } else if (e == 0) {
    val = ldexpf((float)m, -9);              /* subnormal: m * 2^-9 */
  } else {
    val = ldexpf((float)(8 + m), e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
  }
  return sign ? -val : val;
}

/* Code byte of an exactly representable non-negative E4M3 magnitude. */
static uint8_t e4m3_bits_of_magnitude(float a) {
  if (a == 0.0f) return 0;
  if (a < ldexpf(1.0f, -6)) {
    return (uint8_t)(int)(a / ldexpf(1.0f, -9)); /* exponent field 0 */
  }
  int e2;
  (void)frexpf(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;       /* a in [2^E, 2^(E+1)) */
  int m = (int)(a / ldexpf(1.0f, E - 3)) - 8;
  return (uint8_t)(((E + 7) << 3) | m);
}

/* Round u to the E4M3FN grid: nearest, ties to even, saturate finite
 * overflow to +-448.  Returns the code byte. */
uint8_t oracle_e4m3_encode(float u) {
  uint8_t sign = signbit(u) ? 0x80 : 0x00;
  if (isnan(u)) return (uint8_t)(sign | 0x7F);
  float a = fabsf(u);
  if (a >= 448.0f) return (uint8_t)(sign | 0x7E); /* satfinite (also +-inf) */
  if (a == 0.0f) return sign;
  int e2;
  (void)frexpf(a, &e2);
  int E = e2 - 1;
  if (E < -6) E = -6; /* below the normal range the step stays 2^-9 */
  float q = ldexpf(1.0f, E - 3); /* grid step in this binade */
  /* a / q is exact (power-of-two scaling); nearbyintf rounds half to even
   * under the default rounding mode. */
  float m = nearbyintf(a / q);
  float r = m * q; /* exact: m <= 16 */
  /* r <= 448 here: a < 448 = 14 * 32 in the top binade */
  return (uint8_t)(sign | e4m3_bits_of_magnitude(r));
}

/* Nearest integer, ties to even, clamped to [-127, 127]. */
int8_t oracle_int8_encode(float u) {
  float m = nearbyintf(u);
  if (m > 127.0f) m = 127.0f;
  if (m < -127.0f) m = -127.0f;
  return (int8_t)(int)m;
}

/* One group: n values laid out as `rows` rows of `row_len` floats with
 * consecutive rows `row_stride` floats apart.  Writes y (same layout),
 * the code bytes (same layout, nullable) and returns the scale. */
static float qdq_group(const float* x, float* y, uint8_t* codes, int64_t rows,
                       int64_t row_len, int64_t row_stride, int mode) {
  float a = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < row_len; ++j) {
      float v = fabsf(x[r * row_stride + j]);
      if (v > a) a = v;
    }
  if (a == 0.0f) {
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t j = 0; j < row_len; ++j) {
        float v = x[r * row_stride + j];
        y[r * row_stride + j] = v;
        if (codes) codes[r * row_stride + j] = (mode == ORACLE_QDQ_E4M3 && signbit(v)) ? 0x80 : 0x00;
      }
    return 0.0f;
  }
  const float M = (mode == ORACLE_QDQ_E4M3) ? 448.0f : 127.0f;
  volatile float s = a / M;     /* one correctly rounded binary32 division */
  volatile float rcp = 1.0f / s;
  if (isinf(rcp)) {
    s = 0.0f;
    rcp = 0.0f;
  }
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < row_len; ++j) {
      int64_t i = r * row_stride + j;
      float u = x[i] * rcp;
      if (mode == ORACLE_QDQ_E4M3) {
        uint8_t c = oracle_e4m3_encode(u);
        y[i] = oracle_e4m3_decode(c) * s;
        if (codes) codes[i] = c;
      } else {
        int8_t c = oracle_int8_encode(u);
        y[i] = (float)c * s;
        if (codes) codes[i] = (uint8_t)c;
      }
    }
  return s;
}

/*
 * Grouped QDQ of a contiguous [batch, rows, cols] fp32 tensor: one group per
 * (batch index, block of `group_cols` consecutive columns) spanning all rows.
 * scales: [batch, cols / group_cols] (nullable); codes: like x (nullable).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_qdq_groups(const float* x, float* y, float* scales, uint8_t* codes,
                      int64_t batch, int64_t rows, int64_t cols, int64_t group_cols,
                      int mode) {
  if (!x || !y || batch < 0 || rows < 0 || cols < 0 || group_cols <= 0 ||
      (cols % group_cols) != 0)
    return -1;
  if (mode != ORACLE_QDQ_E4M3 && mode != ORACLE_QDQ_INT8) {
    if (mode != ORACLE_QDQ_NONE) return -1;
    memmove(y, x, (size_t)(batch * rows * cols) * sizeof(float));
    return 0;
  }
  int64_t nb = cols / group_cols;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t j = 0; j < nb; ++j) {
      int64_t off = b * rows * cols + j * group_cols;
      float s = qdq_group(x + off, y + off, codes ? codes + off : 0, rows, group_cols,
                          cols, mode);
      if (scales) scales[b * nb + j] = s;
    }
  return 0;
}

/* Element-wise helpers for the tests. */
void oracle_e4m3_encode_array(const float* u, uint8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = oracle_e4m3_encode(u[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_e4m3_decode(c[i]);
}

void oracle_int8_encode_array(const float* u, int8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = oracle_int8_encode(u[i]);
}
