/*
 * mfa_oracle.c -- plain, slow, double-precision CPU oracle for decode-time
 * Multi-matrix Factorization Attention (MFA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load or call this code.  It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it computes (sources):
 *   - "Step-3 is Large yet Affordable: Model-system Co-design for Cost-effective
 *     Decoding" (paper summary page), section 2 and Table 1 (model card): MFA
 *     uses 64 query heads that all share ONE key head and ONE value head, each
 *     of dimension 256.
 *   - Same page, section 8.1: decode attention over the per-sequence KV cache
 *     (the custom Flash-Attention kernel of the attention instance); section 7:
 *     an 8-bit KV cache takes 512 bytes per token per layer (K 256 B + V 256 B).
 *   - The attention itself is plain scaled dot-product attention:
 *       s_j        = scale * sum_i q[b,h,i] * k[b,j,i]           (j < L_b)
 *       out[b,h,:] = sum_j exp(s_j - m) v[b,j,:] / sum_j exp(s_j - m)
 *       lse[b,h]   = m + ln(sum_j exp(s_j - m)),  m = max_j s_j
 *     with natural logarithms of the scaled logits (reading: the pages give no
 *     log base; natural log is the usual convention).
 *   - "DuckLLM decode fixed-cost reduction" page, section 7.6 (decode context
 *     kernel): the length seen by attention after an append includes the token
 *     just appended; the append offset and the attention length come from one
 *     device-owned counter.
 *   - E4M3 codes follow the OCP 8-bit floating point specification (OFP8),
 *     E4M3 format: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities,
 *     NaN = S.1111.111, largest finite magnitude 448.
 *   - Same page, section 5.2: KV may be stored in 4 bits and the attention
 *     computed in 8 bits. E2M1 codes follow the OCP Microscaling (MX)
 *     specification's FP4 element format: 1 sign, 2 exponent (bias 1), 1
 *     mantissa bit, no infinities or NaN, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - FP8 scale granularity: one fp32 scale per token, separately for K and V,
 *     s = absmax / 448 (fp32 division), code = RNE-to-E4M3(x / s) (fp32
 *     division) saturated to +-448; absmax == 0 gives s = 1 and all-zero codes.
 *   - The dequantised FP8 value is decode(code) * s, exact in fp64.
 *   - 4-bit KV: one fp32 scale per token (K and V separately), s = absmax / 6,
 *     code = nearest E2M1 value to x / s (ties to the even mantissa, saturating
 *     to +-6, sign kept on zero), two codes per byte with element 2k in the low
 *     nibble; the dequantised value is decode(code) * s. Every E2M1 value is an
 *     E4M3 value, so "computing in 8 bits" loses nothing further.
 *   - A sequence with L_b == 0 yields out = 0 and lse = -inf.
 *   - Unused slots of a sequence's last page never contribute, whatever they hold.
 *
 * Everything is computed element by element in fp64 in the definition's order;
 * no blocking, tiling, splitting or online rescaling.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_f32(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* OFP8 E4M3 decode from the format definition. */
double oracle_e4m3_to_f64(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: (m/8) * 2^(1-7) */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest E4M3 value to x (ties to even mantissa), magnitudes above the largest
 * finite value clamp to 448 (saturating conversion); NaN maps to 0x7F.  The sign
 * of x is kept, so a negative value that rounds to zero gives 0x80. */
uint8_t oracle_e4m3_from_f32(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* spacing of representable values around a: binade [2^e, 2^(e+1)) has 8
   * mantissa steps (spacing 2^(e-3)) for e >= -6; below 2^-6 the subnormals are
   * spaced 2^-9, the same as the first normal binade */
  int e;
  if (a < ldexp(1.0, -6)) {
    e = -6;
  } else {
    int fe;
    frexp(a, &fe); /* a = f * 2^fe, f in [0.5, 1) */
    e = fe - 1;
  }
  double quantum = ldexp(1.0, e - 3);
  double r = nearbyint(a / quantum); /* default rounding mode: to nearest, ties to even */
  double v = r * quantum;
  if (v >= 448.0) return (uint8_t)(sign | 0x7E);
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) {
    int mant = (int)(v / ldexp(1.0, -9));
    return (uint8_t)(sign | mant);
  }
  int fe;
  frexp(v, &fe);
  int ev = fe - 1; /* v in [2^ev, 2^(ev+1)) */
  int mant = (int)((v / ldexp(1.0, ev) - 1.0) * 8.0);
  return (uint8_t)(sign | ((ev + 7) << 3) | mant);
}

void oracle_e4m3_from_f32_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_f32(x[i]);
}

void oracle_e4m3_to_f64_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(c[i]);
}

/* OCP MX FP4 (E2M1) decode from the format definition: exponent field 0 is
 * subnormal, m * 2^(1-1) * 2^-1; otherwise (1 + m/2) * 2^(e-1). */
double oracle_e2m1_to_f64(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -mag : mag;
}

/* Nearest E2M1 code to x: the candidate magnitude closest to |x|, a tie going
 * to the code whose mantissa bit is 0; beyond the largest value the code
 * saturates at 6. The sign of x is kept (a negative x that rounds to zero
 * gives code 8). */
uint8_t oracle_e2m1_from_f32(float x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double a = fabs((double)x);
  if (isnan(x)) return (uint8_t)(sign | 7);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - oracle_e2m1_to_f64((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

void oracle_e2m1_to_f64_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_to_f64(c[i]);
}

void oracle_e2m1_from_f32_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_from_f32(x[i]);
}

/* Per-token 4-bit quantisation of bf16 rows x[n_tokens][d] (d even): one fp32
 * scale per row (absmax / 6), codes = E2M1(x / scale), packed two per byte,
 * element 2k in the low nibble of byte k. */
void oracle_quantize_tokens_e2m1(const uint16_t* x, int64_t n_tokens, int d, uint8_t* packed, float* scales) {
  for (int64_t t = 0; t < n_tokens; ++t) {
    const uint16_t* row = x + t * (int64_t)d;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
      float a = fabsf(bf16_to_f32(row[i]));
      if (a > amax) amax = a;
    }
    float s = (amax > 0.0f) ? amax / 6.0f : 1.0f;
    scales[t] = s;
    for (int i = 0; i < d; i += 2) {
      uint8_t lo = oracle_e2m1_from_f32(bf16_to_f32(row[i]) / s);
      uint8_t hi = oracle_e2m1_from_f32(bf16_to_f32(row[i + 1]) / s);
      packed[t * (int64_t)(d / 2) + i / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* Per-token FP8 quantisation of bf16 rows x[n_tokens][d]: one fp32 scale per
 * row (absmax / 448), codes = E4M3(x / scale). */
void oracle_quantize_tokens_e4m3(const uint16_t* x, int64_t n_tokens, int d,
                                 uint8_t* codes, float* scales) {
  for (int64_t t = 0; t < n_tokens; ++t) {
    const uint16_t* row = x + t * (int64_t)d;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
      float a = fabsf(bf16_to_f32(row[i]));
      if (a > amax) amax = a;
    }
    float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    scales[t] = s;
    for (int i = 0; i < d; ++i) {
      float y = bf16_to_f32(row[i]) / s;
      codes[t * (int64_t)d + i] = oracle_e4m3_from_f32(y);
    }
  }
}

/* Cache formats (the kv_fp8 argument): 0 bf16, 1 E4M3 + per-token scale,
 * 2 packed E2M1 + per-token scale. */
enum { KV_BF16 = 0, KV_E4M3 = 1, KV_E2M1 = 2 };

/* Value of element i of the cache row at `slot` (slot = page * page_size + row),
 * as an exact fp64 number: the bf16 value, or decode(code) * scale. */
static double cache_value(const void* cache, const float* scale_arr, int kv_fp8,
                          const double* e4m3_table, int64_t slot, int d, int i) {
  if (kv_fp8 == KV_E2M1) {
    const uint8_t byte = ((const uint8_t*)cache)[slot * (d / 2) + i / 2];
    return oracle_e2m1_to_f64((i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15)) * (double)scale_arr[slot];
  }
  if (kv_fp8) {
    const uint8_t* c = (const uint8_t*)cache;
    return e4m3_table[c[slot * d + i]] * (double)scale_arr[slot];
  }
  const uint16_t* c = (const uint16_t*)cache;
  return oracle_bf16_to_f64(c[slot * d + i]);
}

enum { ORACLE_OK = 0, ORACLE_BAD_PAGE = -1, ORACLE_BAD_LEN = -2, ORACLE_BAD_ARG = -3 };

/* One output row (sequence b, head h) by the definition above.
 * The KV position j of sequence b lives in page page_table[b][j / page_size],
 * row j % page_size of that page. */
static int decode_row(const uint16_t* q, const void* k_cache, const void* v_cache,
                      const float* k_scale, const float* v_scale, int kv_fp8,
                      const double* e4m3_table, const int32_t* page_table,
                      const int32_t* seq_lens, int H, int D, int page_size,
                      int max_pages, int64_t num_pages, double scale, int b, int h,
                      double* out_row, double* lse_out) {
  int64_t n = seq_lens[b];
  if (n < 0 || n > (int64_t)max_pages * page_size) return ORACLE_BAD_LEN;
  for (int i = 0; i < D; ++i) out_row[i] = 0.0;
  if (n == 0) {
    *lse_out = -INFINITY;
    return ORACLE_OK;
  }
  const uint16_t* qrow = q + ((int64_t)b * H + h) * D;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
  if (!s || !slot) {
    free(s);
    free(slot);
    return ORACLE_BAD_ARG;
  }
  /* logits */
  for (int64_t j = 0; j < n; ++j) {
    int32_t page = page_table[(int64_t)b * max_pages + j / page_size];
    if (page < 0 || page >= num_pages) {
      free(s);
      free(slot);
      return ORACLE_BAD_PAGE;
    }
    slot[j] = (int64_t)page * page_size + j % page_size;
    double dot = 0.0;
    for (int i = 0; i < D; ++i)
      dot += oracle_bf16_to_f64(qrow[i]) *
             cache_value(k_cache, k_scale, kv_fp8, e4m3_table, slot[j], D, i);
    s[j] = scale * dot;
  }
  /* softmax and weighted sum of values */
  double m = s[0];
  for (int64_t j = 1; j < n; ++j)
    if (s[j] > m) m = s[j];
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) z += exp(s[j] - m);
  for (int64_t j = 0; j < n; ++j) {
    double p = exp(s[j] - m);
    for (int i = 0; i < D; ++i)
      out_row[i] += p * cache_value(v_cache, v_scale, kv_fp8, e4m3_table, slot[j], D, i);
  }
  for (int i = 0; i < D; ++i) out_row[i] /= z;
  *lse_out = m + log(z);
  free(s);
  free(slot);
  return ORACLE_OK;
}

/*
 * Decode attention for selected (b, h) rows over a paged cache.
 *   q          [B][H][D] bf16 bits
 *   k_cache    [num_pages][page_size][D]  bf16 bits, or E4M3 codes if kv_fp8 == 1,
 *              or [num_pages][page_size][D/2] packed E2M1 codes if kv_fp8 == 2
 *   v_cache    same layout as k_cache
 *   k_scale    [num_pages][page_size] fp32 (FP8 only, else may be NULL)
 *   v_scale    same (FP8 only)
 *   page_table [B][max_pages] int32, seq_lens [B] int32
 *   rows_b/rows_h [n_rows]: the rows to compute; out [n_rows][D], lse [n_rows]
 * Returns 0, or a negative code for a bad page id / length / argument.
 */
int oracle_mfa_decode_rows(const uint16_t* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int kv_fp8,
                           const int32_t* page_table, const int32_t* seq_lens, int B, int H,
                           int D, int page_size, int max_pages, int64_t num_pages, double scale,
                           const int32_t* rows_b, const int32_t* rows_h, int64_t n_rows,
                           double* out, double* lse, int n_threads) {
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out || !lse) return ORACLE_BAD_ARG;
  if (B <= 0 || H <= 0 || D <= 0 || page_size <= 0 || max_pages <= 0) return ORACLE_BAD_ARG;
  if (kv_fp8 && (!k_scale || !v_scale)) return ORACLE_BAD_ARG;
  double e4m3_table[256];
  for (int c = 0; c < 256; ++c) e4m3_table[c] = oracle_e4m3_to_f64((uint8_t)c);
  int status = ORACLE_OK;
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
  for (int64_t r = 0; r < n_rows; ++r) {
    int b = rows_b[r], h = rows_h[r];
    int st;
    if (b < 0 || b >= B || h < 0 || h >= H)
      st = ORACLE_BAD_ARG;
    else
      st = decode_row(q, k_cache, v_cache, k_scale, v_scale, kv_fp8, e4m3_table, page_table,
                      seq_lens, H, D, page_size, max_pages, num_pages, scale, b, h,
                      out + r * (int64_t)D, lse + r);
    if (st != ORACLE_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/* All B*H rows, out [B][H][D], lse [B][H]. */
int oracle_mfa_decode(const uint16_t* q, const void* k_cache, const void* v_cache,
                      const float* k_scale, const float* v_scale, int kv_fp8,
                      const int32_t* page_table, const int32_t* seq_lens, int B, int H, int D,
                      int page_size, int max_pages, int64_t num_pages, double scale, double* out,
                      double* lse, int n_threads) {
  if (B <= 0 || H <= 0) return ORACLE_BAD_ARG;
  int64_t n_rows = (int64_t)B * H;
  int32_t* rb = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rows);
  int32_t* rh = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rows);
  if (!rb || !rh) {
    free(rb);
    free(rh);
    return ORACLE_BAD_ARG;
  }
  for (int64_t r = 0; r < n_rows; ++r) {
    rb[r] = (int32_t)(r / H);
    rh[r] = (int32_t)(r % H);
  }
  int st = oracle_mfa_decode_rows(q, k_cache, v_cache, k_scale, v_scale, kv_fp8, page_table,
                                  seq_lens, B, H, D, page_size, max_pages, num_pages, scale, rb,
                                  rh, n_rows, out, lse, n_threads);
  free(rb);
  free(rh);
  return st;
}

/* The KV append of one decode step, on host copies: token t of sequence b goes
 * to position seq_lens[b] + t (page page_table[b][pos / page_size], row
 * pos % page_size); afterwards seq_lens[b] grows by n_new.  bf16 rows are
 * copied; with kv_fp8 = 1 (E4M3) or 2 (packed E2M1) they are quantised per
 * token as above.
 * k_new/v_new: [B][n_new][D] bf16 bits.  Returns 0 or a negative code. */
int oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new, int n_new, void* k_cache,
                     void* v_cache, float* k_scale, float* v_scale, int kv_fp8,
                     const int32_t* page_table, int32_t* seq_lens, int B, int D, int page_size,
                     int max_pages, int64_t num_pages) {
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !seq_lens) return ORACLE_BAD_ARG;
  if (B <= 0 || D <= 0 || n_new < 0) return ORACLE_BAD_ARG;
  if (kv_fp8 && (!k_scale || !v_scale)) return ORACLE_BAD_ARG;
  uint8_t* codes = (uint8_t*)malloc((size_t)D);
  if (!codes) return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b) {
    int64_t start = seq_lens[b];
    if (start < 0 || start + n_new > (int64_t)max_pages * page_size) {
      status = ORACLE_BAD_LEN;
      continue;
    }
    int bad = 0;
    for (int t = 0; t < n_new && !bad; ++t) {
      int64_t pos = start + t;
      int32_t page = page_table[(int64_t)b * max_pages + pos / page_size];
      if (page < 0 || page >= num_pages) {
        bad = 1;
        break;
      }
      int64_t slot = (int64_t)page * page_size + pos % page_size;
      const uint16_t* kr = k_new + ((int64_t)b * n_new + t) * D;
      const uint16_t* vr = v_new + ((int64_t)b * n_new + t) * D;
      if (kv_fp8 == KV_E2M1) {
        oracle_quantize_tokens_e2m1(kr, 1, D, codes, &k_scale[slot]);
        memcpy((uint8_t*)k_cache + slot * (D / 2), codes, (size_t)(D / 2));
        oracle_quantize_tokens_e2m1(vr, 1, D, codes, &v_scale[slot]);
        memcpy((uint8_t*)v_cache + slot * (D / 2), codes, (size_t)(D / 2));
      } else if (kv_fp8) {
        oracle_quantize_tokens_e4m3(kr, 1, D, codes, &k_scale[slot]);
        memcpy((uint8_t*)k_cache + slot * D, codes, (size_t)D);
        oracle_quantize_tokens_e4m3(vr, 1, D, codes, &v_scale[slot]);
        memcpy((uint8_t*)v_cache + slot * D, codes, (size_t)D);
      } else {
        memcpy((uint16_t*)k_cache + slot * D, kr, sizeof(uint16_t) * (size_t)D);
        memcpy((uint16_t*)v_cache + slot * D, vr, sizeof(uint16_t) * (size_t)D);
      }
    }
    if (bad) {
      status = ORACLE_BAD_PAGE;
      continue;
    }
    seq_lens[b] = (int32_t)(start + n_new);
  }
  free(codes);
  return status;
}
