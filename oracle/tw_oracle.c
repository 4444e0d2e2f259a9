/*
 * tw_oracle.c -- plain, slow CPU oracle for the W1.58A8 ternary path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the package smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library: every step below is written out from the method's definition.
 *
 * Sources (web pages on ternary-weight inference; cited by page title and
 * section):
 *   [P1] "1bit-systems：在AMD Strix Halo上实现纯Rust本地三值权重LLM推理",
 *        sections "三值量化：1.58-bit的魔法" (weights in {-1,0,+1}, 1.58 bit)
 *        and "技术架构：Rust在上，HIP在下" (an RMSNorm kernel next to the
 *        ternary GEMV).
 *   [P2] "BitNet-rs：Rust实现的高效1比特大语言模型推理引擎", section
 *        "技术实现细节" (activations quantised to 8 bit).
 *   [P3] bitnet.cpp CPU tutorial (m.qwbw.cn/news/64613), section 1.1 (ternary
 *        weights stored 2-bit aligned; the product needs only a sign check and
 *        an add) and section 3.2 (conversion absmean-quantises every weight
 *        onto the ternary set).
 *   [P5] "BitNet 1 位 LLM 独立推理引擎：位串行 GEMM 内核与 LUT 优化工程实践",
 *        正文 paragraph 4 (I2_S is the plain 2-bit format) and paragraph 3 (TL2
 *        packs several weights into one small index so fewer bytes are loaded).
 * The pages give no formula for absmean, the activation scale, the rounding
 * mode or the bit layout; this file follows these readings:
 *   - one absmean scale per tensor, gamma = mean |W| with the sum taken
 *     exactly and rounded once to double, then gamma = (float)(S / (N*K));
 *   - t = clamp(round_half_even(W / gamma), -1, 1) with an IEEE fp32 divide;
 *     gamma == 0 gives t = 0;
 *   - packed byte b of row n holds t[n][4b+j] + 1 in bits 2j..2j+1 (code 0 =
 *     -1, 1 = 0, 2 = +1, 3 invalid), rows contiguous, K % 4 == 0;
 *   - per token a = max|x|; x_q = clamp(round_half_even(fl(fl(x*127)/a)),
 *     -128, 127); s_x = a; a == 0 gives x_q = 0 and s_x = 0;
 *   - RMSNorm: r = exact sum of x^2 rounded once to double,
 *     ms = (float)(r / K), inv = 1 / sqrtf(ms + eps) (fp32),
 *     u = fl(fl(x * inv) * g), then the activation quantisation above on u;
 *   - five trits per byte (the denser layout): RB = 16 * ceil(K / 80) bytes
 *     per row; byte i holds weights 4i..4i+3 as base-3 digits 0..3 and weight
 *     4 RB + i as digit 4, each digit t + 1; weights at k >= K count as 0;
 *   - residual: h_out = fl32(h + y);
 *   - acc = sum_k t * x_q exactly (int64, must fit int32);
 *   - y = (float)(((double)acc * gamma * s_x) / 127.0).
 * Compile with -ffp-contract=off and without fast-math so every fp32 step is
 * one IEEE-rounded operation.
 *
 * Parity pins: every function here is checked by tests that do not use this
 * file's code (math.fsum for the exact sums, numpy int64 / float64 matmul of
 * the unpacked weights, closed forms and hand-worked fixtures).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  TWO_OK = 0,
  TWO_ERR_NULL = 1,
  TWO_ERR_SHAPE = 2,
  TWO_ERR_INVALID_CODE = 3,   /* a packed 2-bit field holds 3 */
  TWO_ERR_NONFINITE = 4,      /* an input is NaN or infinite */
  TWO_ERR_NEGATIVE = 5,       /* exact sum given a negative value */
  TWO_ERR_OVERFLOW = 6        /* an accumulator does not fit int32 */
};

/* ------------------------------------------------------------------------ */
/* Exact sum of non-negative doubles.                                         */
/*                                                                            */
/* A long fixed-point integer whose bit 0 is worth 2^-1074 (the smallest     */
/* double subnormal).  Every finite double is an integer multiple of that,   */
/* so adding doubles into it is exact; the sum is rounded once, to nearest   */
/* with ties to even, at the end.                                             */
/* ------------------------------------------------------------------------ */
#define BIG_DIGITS 72 /* 72 x 32 = 2304 bits: 2098 bits of range + count headroom */

typedef struct {
  uint32_t d[BIG_DIGITS]; /* little-endian base-2^32 digits */
} big_t;

static void big_clear(big_t *a) { memset(a->d, 0, sizeof(a->d)); }

/* a += v * 2^pos */
static void big_add_shifted(big_t *a, uint64_t v, int pos) {
  int i = pos / 32;
  int o = pos % 32;
  unsigned __int128 w = ((unsigned __int128)v) << o;
  uint64_t carry = 0;
  for (int j = 0; j < 3 || carry; ++j) {
    uint64_t piece = (j < 3) ? (uint64_t)(w >> (32 * j)) & 0xffffffffu : 0;
    uint64_t s = (uint64_t)a->d[i + j] + piece + carry;
    a->d[i + j] = (uint32_t)s;
    carry = s >> 32;
  }
}

/* a += x, x finite and >= 0 */
static void big_add_double(big_t *a, double x) {
  uint64_t bits;
  memcpy(&bits, &x, sizeof(bits));
  int e = (int)((bits >> 52) & 0x7ff);
  uint64_t frac = bits & ((1ull << 52) - 1);
  if (e == 0) {
    if (frac) big_add_shifted(a, frac, 0); /* subnormal: frac * 2^-1074 */
  } else {
    /* (2^52 + frac) * 2^(e - 1075) = (2^52 + frac) * 2^(e - 1) * 2^-1074 */
    big_add_shifted(a, frac | (1ull << 52), e - 1);
  }
}

static int big_bit(const big_t *a, int idx) {
  if (idx < 0) return 0;
  return (a->d[idx / 32] >> (idx % 32)) & 1u;
}

/* Round the integer to the nearest double (ties to even), times 2^-1074. */
static double big_to_double(const big_t *a) {
  int top = BIG_DIGITS - 1;
  while (top >= 0 && a->d[top] == 0) --top;
  if (top < 0) return 0.0;
  int msb = top * 32 + (31 - __builtin_clz(a->d[top]));
  if (msb <= 52) {
    /* fits in 53 bits: exact */
    uint64_t m = 0;
    for (int b = msb; b >= 0; --b) m = (m << 1) | (uint64_t)big_bit(a, b);
    return ldexp((double)m, -1074);
  }
  uint64_t m = 0;
  for (int b = msb; b > msb - 53; --b) m = (m << 1) | (uint64_t)big_bit(a, b);
  int round_bit = big_bit(a, msb - 53);
  int sticky = 0;
  for (int b = msb - 54; b >= 0 && !sticky; --b) sticky = big_bit(a, b);
  if (round_bit && (sticky || (m & 1u))) m += 1; /* may become 2^53: still exact */
  return ldexp((double)m, msb - 52 - 1074);
}

/* Exact sum of n non-negative finite doubles, rounded once to nearest-even. */
int two_exact_sum(const double *v, int64_t n, double *out) {
  if (!v || !out) return TWO_ERR_NULL;
  if (n < 0) return TWO_ERR_SHAPE;
  big_t acc;
  big_clear(&acc);
  for (int64_t i = 0; i < n; ++i) {
    if (!isfinite(v[i])) return TWO_ERR_NONFINITE;
    if (v[i] < 0) return TWO_ERR_NEGATIVE;
    big_add_double(&acc, v[i]);
  }
  *out = big_to_double(&acc);
  return TWO_OK;
}

/* ------------------------------------------------------------------------ */
/* Absmean ternarisation and 2-bit packing ([P3] 3.2, 1.1; [P5] para 4).    */
/* ------------------------------------------------------------------------ */

/* gamma = (float)(S / n), S = exact sum of |W| rounded to double.  The exact
 * sum is also returned so tests can pin it. */
int two_absmean(const float *W, int64_t n, float *gamma, double *sum_out) {
  if (!W || !gamma) return TWO_ERR_NULL;
  if (n <= 0) return TWO_ERR_SHAPE;
  big_t acc;
  big_clear(&acc);
  for (int64_t i = 0; i < n; ++i) {
    if (!isfinite(W[i])) return TWO_ERR_NONFINITE;
    big_add_double(&acc, fabs((double)W[i]));
  }
  double S = big_to_double(&acc);
  if (sum_out) *sum_out = S;
  *gamma = (float)(S / (double)n);
  return TWO_OK;
}

/* t = clamp(round_half_even(w / gamma), -1, 1); gamma == 0 gives 0. */
static int ternarise(float w, float gamma) {
  if (gamma == 0.0f) return 0;
  float q = w / gamma;     /* one IEEE fp32 divide */
  float r = nearbyintf(q); /* default rounding mode: nearest, ties to even */
  if (r > 1.0f) return 1;
  if (r < -1.0f) return -1;
  return (int)r;
}

/* Pack rows of W with a given scale (the scale of the whole tensor). */
int two_pack_rows_with_scale(const float *W, int64_t rows, int64_t K, float gamma,
                             uint8_t *packed) {
  if (!W || !packed) return TWO_ERR_NULL;
  if (rows <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t b = 0; b < K / 4; ++b) {
      unsigned byte = 0;
      for (int j = 0; j < 4; ++j) {
        float w = W[n * K + 4 * b + j];
        if (!isfinite(w)) return TWO_ERR_NONFINITE;
        int t = ternarise(w, gamma);
        byte |= (unsigned)(t + 1) << (2 * j);
      }
      packed[n * (K / 4) + b] = (uint8_t)byte;
    }
  }
  return TWO_OK;
}

int two_pack_ternary(const float *W, int64_t N, int64_t K, uint8_t *packed,
                     float *w_scale) {
  if (!W || !packed || !w_scale) return TWO_ERR_NULL;
  if (N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  float gamma;
  int st = two_absmean(W, N * K, &gamma, NULL);
  if (st != TWO_OK) return st;
  st = two_pack_rows_with_scale(W, N, K, gamma, packed);
  if (st != TWO_OK) return st;
  *w_scale = gamma;
  return TWO_OK;
}

/* Inverse of the packing: t in {-1,0,1}; a field holding 3 is an error. */
int two_unpack_ternary(const uint8_t *packed, int64_t N, int64_t K, int8_t *t) {
  if (!packed || !t) return TWO_ERR_NULL;
  if (N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      unsigned byte = packed[n * (K / 4) + k / 4];
      unsigned code = (byte >> (2 * (k % 4))) & 3u;
      if (code == 3u) return TWO_ERR_INVALID_CODE;
      t[n * K + k] = (int8_t)((int)code - 1);
    }
  }
  return TWO_OK;
}

/* ------------------------------------------------------------------------ */
/* Five trits per byte ([P5] 正文 paragraph 3: TL2 stores three weights in a  */
/* 5-bit index so fewer bytes are loaded; 3^5 = 243 <= 256 takes the same    */
/* idea to 1.6 bits per weight).  Reading of the layout (the page fixes none):*/
/*   a row takes RB = 16 * ceil(K / 80) bytes;                                */
/*   byte i of a row holds the weights k = 4i, 4i+1, 4i+2, 4i+3 as its base-3 */
/*   digits 0..3 and the weight k = 4*RB + i as its digit 4:                  */
/*     byte = sum_{j<4} (t[4i+j] + 1) * 3^j + (t[4*RB + i] + 1) * 81;         */
/*   weights at k >= K count as t = 0.  Bytes 243..255 are invalid.           */
/* ------------------------------------------------------------------------ */
int64_t two_t5_row_bytes(int64_t K) { return K <= 0 ? 0 : 16 * ((K + 79) / 80); }

/* Weight k of a row sits in byte `*byte` as base-3 digit `*digit`. */
static void t5_place(int64_t k, int64_t RB, int64_t *byte, int *digit) {
  if (k < 4 * RB) {
    *byte = k / 4;
    *digit = (int)(k % 4);
  } else {
    *byte = k - 4 * RB;
    *digit = 4;
  }
}

int two_pack_trits5(const int8_t *t, int64_t N, int64_t K, uint8_t *out) {
  if (!t || !out) return TWO_ERR_NULL;
  if (N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  const int64_t RB = two_t5_row_bytes(K);
  for (int64_t n = 0; n < N; ++n) {
    /* every digit starts as the code of t = 0 */
    for (int64_t b = 0; b < RB; ++b) out[n * RB + b] = 1 + 3 + 9 + 27 + 81;
    for (int64_t k = 0; k < K; ++k) {
      int v = t[n * K + k];
      if (v < -1 || v > 1) return TWO_ERR_INVALID_CODE;
      int64_t b;
      int d;
      t5_place(k, RB, &b, &d);
      int w = 1;
      for (int j = 0; j < d; ++j) w *= 3;
      out[n * RB + b] = (uint8_t)(out[n * RB + b] + v * w); /* code (v + 1) replaces code 1 */
    }
  }
  return TWO_OK;
}

/* Inverse of two_pack_trits5.  A byte above 242, or a nonzero weight at k >= K,
 * is an error. */
int two_unpack_trits5(const uint8_t *p, int64_t N, int64_t K, int8_t *t) {
  if (!p || !t) return TWO_ERR_NULL;
  if (N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  const int64_t RB = two_t5_row_bytes(K);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < RB; ++b) {
      int v = p[n * RB + b];
      if (v > 242) return TWO_ERR_INVALID_CODE;
      for (int d = 0; d < 5; ++d) {
        int code = v % 3;
        v /= 3;
        int64_t k = d < 4 ? 4 * b + d : 4 * RB + b;
        if (k < K) t[n * K + k] = (int8_t)(code - 1);
        else if (code != 1) return TWO_ERR_INVALID_CODE;
      }
    }
  }
  return TWO_OK;
}

/* Absmean ternarisation (as two_pack_ternary) stored five trits per byte. */
int two_pack_ternary5(const float *W, int64_t N, int64_t K, uint8_t *out, float *w_scale) {
  if (!W || !out || !w_scale) return TWO_ERR_NULL;
  if (N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  float gamma;
  int st = two_absmean(W, N * K, &gamma, NULL);
  if (st != TWO_OK) return st;
  int8_t *t = (int8_t *)malloc((size_t)K);
  if (!t) return TWO_ERR_NULL;
  for (int64_t n = 0; n < N && st == TWO_OK; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      float w = W[n * K + k];
      if (!isfinite(w)) {
        st = TWO_ERR_NONFINITE;
        break;
      }
      t[k] = (int8_t)ternarise(w, gamma);
    }
    if (st == TWO_OK) st = two_pack_trits5(t, 1, K, out + n * two_t5_row_bytes(K));
  }
  free(t);
  if (st == TWO_OK) *w_scale = gamma;
  return st;
}

/* ------------------------------------------------------------------------ */
/* Per-token absmax int8 activation quantisation ([P2] 技术实现细节).        */
/* ------------------------------------------------------------------------ */
int two_quant_act(const float *x, int64_t M, int64_t K, int8_t *x_q, float *s_x,
                  int32_t *x_sum) {
  if (!x || !x_q || !s_x) return TWO_ERR_NULL;
  if (M <= 0 || K <= 0) return TWO_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    const float *row = x + m * K;
    float a = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      if (!isfinite(row[k])) return TWO_ERR_NONFINITE;
      float v = fabsf(row[k]);
      if (v > a) a = v;
    }
    int64_t sum = 0;
    for (int64_t k = 0; k < K; ++k) {
      int q = 0;
      if (a > 0.0f) {
        float p = row[k] * 127.0f; /* fl(x * 127) */
        float d = p / a;           /* fl(fl(x * 127) / a) */
        float r = nearbyintf(d);   /* ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -128.0f) r = -128.0f;
        q = (int)r;
      }
      x_q[m * K + k] = (int8_t)q;
      sum += q;
    }
    s_x[m] = a;
    if (x_sum) x_sum[m] = (int32_t)sum;
  }
  return TWO_OK;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm ([P1] 技术架构; constants are this file's reading).               */
/* ------------------------------------------------------------------------ */
/* 1 / sqrtf(ms + eps) of one row, ms = (float)(r / K), r = the exact sum of squares
 * rounded once to double (returned in *r_out). */
static int rms_inv_row(const float *row, int64_t K, float eps, float *inv_out, double *r_out) {
  big_t acc;
  big_clear(&acc);
  for (int64_t k = 0; k < K; ++k) {
    if (!isfinite(row[k])) return TWO_ERR_NONFINITE;
    double v = (double)row[k];
    big_add_double(&acc, v * v); /* the square of a float is exact in double */
  }
  double r = big_to_double(&acc);
  *r_out = r;
  float ms = (float)(r / (double)K);
  *inv_out = 1.0f / sqrtf(ms + eps);
  return TWO_OK;
}

/* The RMSNorm scale alone, per row. */
int two_rms_inv(const float *x, float eps, int64_t M, int64_t K, float *inv) {
  if (!x || !inv) return TWO_ERR_NULL;
  if (M <= 0 || K <= 0) return TWO_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    double r;
    int st = rms_inv_row(x + m * K, K, eps, inv + m, &r);
    if (st != TWO_OK) return st;
  }
  return TWO_OK;
}

int two_rmsnorm(const float *x, const float *g, float eps, int64_t M, int64_t K,
                float *u, double *sumsq_out) {
  if (!x || !g || !u) return TWO_ERR_NULL;
  if (M <= 0 || K <= 0) return TWO_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    const float *row = x + m * K;
    double r;
    float inv;
    int st = rms_inv_row(row, K, eps, &inv, &r);
    if (st != TWO_OK) return st;
    if (sumsq_out) sumsq_out[m] = r;
    for (int64_t k = 0; k < K; ++k) {
      float t = row[k] * inv;
      u[m * K + k] = t * g[k];
    }
  }
  return TWO_OK;
}

int two_rmsnorm_quant_act(const float *x, const float *g, float eps, int64_t M,
                          int64_t K, int8_t *x_q, float *s_x, int32_t *x_sum) {
  if (!x || !g || !x_q || !s_x) return TWO_ERR_NULL;
  if (M <= 0 || K <= 0) return TWO_ERR_SHAPE;
  float *u = (float *)malloc((size_t)(M * K) * sizeof(float));
  if (!u) return TWO_ERR_SHAPE;
  int st = two_rmsnorm(x, g, eps, M, K, u, NULL);
  if (st == TWO_OK) st = two_quant_act(u, M, K, x_q, s_x, x_sum);
  free(u);
  return st;
}

/* ------------------------------------------------------------------------ */
/* Residual add after an output projection ("1-bit 大模型官方推理框架", summary */
/* on kernel fusion: the add is fused into the product's epilogue on the GPU): */
/* h_out = fl32(h + y), one IEEE fp32 addition per element.                   */
/* ------------------------------------------------------------------------ */
int two_residual_add(const float *h, const float *y, int64_t n, float *out) {
  if (!h || !y || !out) return TWO_ERR_NULL;
  if (n <= 0) return TWO_ERR_SHAPE;
  for (int64_t i = 0; i < n; ++i) {
    if (!isfinite(h[i]) || !isfinite(y[i])) return TWO_ERR_NONFINITE;
    out[i] = h[i] + y[i];
  }
  return TWO_OK;
}

/* ------------------------------------------------------------------------ */
/* Integer ternary product and dequantisation ([P3] 1.1: sign check + add).  */
/* ------------------------------------------------------------------------ */
/* Output rows are independent: with -fopenmp (the all-core CPU baseline build) they are
 * shared out over threads; every output is still the same sum in the same order. */
int two_ternary_matmul(const uint8_t *packed, float w_scale, const int8_t *x_q,
                       const float *s_x, int64_t M, int64_t N, int64_t K, float *y,
                       int32_t *acc_out) {
  if (!packed || !x_q || !s_x || !y) return TWO_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  int status = TWO_OK;
  for (int64_t m = 0; m < M; ++m) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      int64_t acc = 0;
      int bad = TWO_OK;
      for (int64_t k = 0; k < K; ++k) {
        unsigned byte = packed[n * (K / 4) + k / 4];
        unsigned code = (byte >> (2 * (k % 4))) & 3u;
        if (code == 3u) {
          bad = TWO_ERR_INVALID_CODE;
          break;
        }
        int t = (int)code - 1;
        int xv = x_q[m * K + k];
        if (t == 1) acc += xv;       /* +1: add */
        else if (t == -1) acc -= xv; /* -1: subtract; 0: skip */
      }
      if (bad == TWO_OK && (acc > INT32_MAX || acc < INT32_MIN)) bad = TWO_ERR_OVERFLOW;
      if (bad != TWO_OK) {
#pragma omp atomic write
        status = bad;
        continue;
      }
      if (acc_out) acc_out[m * N + n] = (int32_t)acc;
      y[m * N + n] = (float)(((double)acc * (double)w_scale * (double)s_x[m]) / 127.0);
    }
    if (status != TWO_OK) return status;
  }
  return TWO_OK;
}

/* The product over rows stored five trits per byte: each row is decoded with
 * two_unpack_trits5, then summed and dequantised exactly as two_ternary_matmul. */
int two_ternary_matmul5(const uint8_t *p5, float w_scale, const int8_t *x_q, const float *s_x,
                        int64_t M, int64_t N, int64_t K, float *y, int32_t *acc_out) {
  if (!p5 || !x_q || !s_x || !y) return TWO_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0 || K % 4 != 0) return TWO_ERR_SHAPE;
  const int64_t RB = two_t5_row_bytes(K);
  int status = TWO_OK;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    int8_t *t = (int8_t *)malloc((size_t)K);
    int bad = t ? two_unpack_trits5(p5 + n * RB, 1, K, t) : TWO_ERR_NULL;
    for (int64_t m = 0; m < M && bad == TWO_OK; ++m) {
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k) {
        int xv = x_q[m * K + k];
        if (t[k] == 1) acc += xv;
        else if (t[k] == -1) acc -= xv;
      }
      if (acc > INT32_MAX || acc < INT32_MIN) {
        bad = TWO_ERR_OVERFLOW;
        break;
      }
      if (acc_out) acc_out[m * N + n] = (int32_t)acc;
      y[m * N + n] = (float)(((double)acc * (double)w_scale * (double)s_x[m]) / 127.0);
    }
    free(t);
    if (bad != TWO_OK) {
#pragma omp atomic write
      status = bad;
    }
  }
  return status;
}

/* Threads the row loop above may use: 1 in the plain build. */
int two_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
