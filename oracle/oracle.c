/*
 * CPU oracle for one PagedAttention step: rotary, paged cache write and
 * causal grouped-query attention over the paged pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file.  The library under test never
 * calls it and shares no code with it.
 *
 * It computes the plain definition, slowly and in the obvious order, so that
 * a reader can check it against the design pages by eye:
 *
 *   - "PagedAttention - CUDA Design Document" (onnxruntime 1.29.0 docs,
 *     contrib_ops/cuda/paged_attention), section 5.1 (slot derivation),
 *     section 4.8 (token j of sequence b sits at position past_b + j),
 *     section 8 implementation note P5 (causal bound kv_len = past + j + 1,
 *     window admits [kv_len - W, kv_len), softcap * tanh(x * scale / softcap)),
 *     section 9.3.1 (a block_table entry of -1 masks its positions),
 *     section 12.5 (rotary_dim = 2 * cos_cache.shape[1]; channels past it are
 *     copied);
 *   - "Design: WebGPU PagedAttention" (onnxruntime 1.29.0 docs), section 3.3
 *     (q_len_b = cum[b+1] - cum[b]) and section 4.1 (GQA head grouping by
 *     n_reps = num_heads / kv_num_heads);
 *   - onnxruntime issue 29714 (cuDNN SDPA decode tier), section 4.3 item 7:
 *     a row with no admitted key outputs 0, not NaN.
 *
 * Precision.  Attention is evaluated in fp64 from exactly converted fp16
 * inputs: scores, max, exponentials, the weighted sum and the normaliser are
 * all doubles, two passes over the admitted keys (max first, then the sums).
 * Rotary is the one place where the result must be an fp16 bit pattern that
 * both sides reproduce exactly; it is evaluated in fp32 with one rounding per
 * operation and no fused multiply-add (build with -ffp-contract=off):
 *     t1 = x1*c, t2 = x2*s, y1 = t1 - t2;  t3 = x2*c, t4 = x1*s, y2 = t3 + t4
 * and each y is rounded to fp16 to nearest-even.  The pages leave this
 * precision open (they report host and device rotary differing by one fp16
 * ulp); fixing the op order is the reading this project takes.
 *
 * Layouts (row-major): query [T, H*D]; key, value [T, Hk*D];
 * key_cache, value_cache [NB, bs, Hk, D]; block_table [B, MB];
 * cum [B+1]; past [B]; cos/sin [P, R/2].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Status codes returned by every entry point. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARGUMENT 1
#define ORACLE_BAD_DEVICE_DATA 2

/* ---- IEEE binary16 conversions, written from the format definition ---- */

/* Exact binary16 -> double.  1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 is subnormal (fraction * 2^-24). */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (single rounding). */
uint16_t oracle_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return sign | 0x7e00;
  double a = fabs(x);
  if (a >= 65520.0) return sign | 0x7c00; /* halfway to 2^16 rounds up */
  if (a < ldexp(1.0, -14)) {
    /* subnormal quantum is 2^-24; scaling by 2^24 is exact */
    double m = nearbyint(ldexp(a, 24));
    return sign | (uint16_t)m; /* m == 1024 encodes the smallest normal */
  }
  int e;
  (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
  double m = nearbyint(ldexp(a, 11 - e)); /* significand in [1024, 2048] */
  int ee = e - 1;
  if (m == 2048.0) {
    m = 1024.0;
    ee += 1;
  }
  if (ee > 15) return sign | 0x7c00;
  return sign | (uint16_t)((ee + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* ---- sequence bookkeeping (WebGPU design section 3.3) ---- */

/* Index of the sequence that owns packed row t, by a linear scan of the
 * cumulative lengths; -1 when t is outside [cum[0], cum[B]). */
static int owner_of_row(const int32_t* cum, int B, int t) {
  for (int b = 0; b < B; ++b)
    if (t >= cum[b] && t < cum[b + 1]) return b;
  return -1;
}

static int check_lengths(const int32_t* cum, const int32_t* past, int B, int T) {
  if (B < 0 || T < 0) return ORACLE_BAD_ARGUMENT;
  if (B == 0) return T == 0 ? ORACLE_OK : ORACLE_BAD_ARGUMENT;
  if (cum[0] != 0 || cum[B] != T) return ORACLE_BAD_DEVICE_DATA;
  for (int b = 0; b < B; ++b) {
    if (cum[b + 1] < cum[b]) return ORACLE_BAD_DEVICE_DATA;
    if (past[b] < 0) return ORACLE_BAD_DEVICE_DATA;
  }
  return ORACLE_OK;
}

/* ---- rotary (CUDA design section 12.5; RoFormer rotation) ---- */

/* Rotates every head of every packed row of x ([T, nheads*D]) at the row's
 * position past_b + j and writes fp16 bit patterns to y (may alias x).
 * half_rot = cos_cache.shape[1], so rotary_dim R = 2*half_rot; channels
 * >= R are copied.  interleaved = 0 pairs (i, i + R/2), interleaved = 1
 * pairs (2i, 2i + 1). */
int oracle_rotary(const uint16_t* x, uint16_t* y, int T, int nheads, int D,
                  const int32_t* cum, const int32_t* past, int B,
                  const uint16_t* cos_cache, const uint16_t* sin_cache,
                  int half_rot, int max_position, int interleaved) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  if (2 * half_rot > D || half_rot < 0) return ORACLE_BAD_ARGUMENT;
  for (int t = 0; t < T; ++t) {
    int b = owner_of_row(cum, B, t);
    int pos = past[b] + (t - cum[b]);
    if (pos >= max_position) return ORACLE_BAD_DEVICE_DATA;
    for (int h = 0; h < nheads; ++h) {
      const uint16_t* xr = x + ((size_t)t * nheads + h) * D;
      uint16_t* yr = y + ((size_t)t * nheads + h) * D;
      uint16_t tmp[1024];
      if (D > 1024) return ORACLE_BAD_ARGUMENT;
      memcpy(tmp, xr, sizeof(uint16_t) * D);
      for (int i = 0; i < half_rot; ++i) {
        int i1 = interleaved ? 2 * i : i;
        int i2 = interleaved ? 2 * i + 1 : i + half_rot;
        float x1 = (float)oracle_half_to_double(xr[i1]);
        float x2 = (float)oracle_half_to_double(xr[i2]);
        float c = (float)oracle_half_to_double(cos_cache[(size_t)pos * half_rot + i]);
        float s = (float)oracle_half_to_double(sin_cache[(size_t)pos * half_rot + i]);
        float t1 = x1 * c;
        float t2 = x2 * s;
        float y1 = t1 - t2;
        float t3 = x2 * c;
        float t4 = x1 * s;
        float y2 = t3 + t4;
        tmp[i1] = oracle_double_to_half((double)y1);
        tmp[i2] = oracle_double_to_half((double)y2);
      }
      memcpy(yr, tmp, sizeof(uint16_t) * D);
    }
  }
  return ORACLE_OK;
}

/* ---- reshape_and_cache (CUDA design section 5.1, derived slot) ---- */

/* For every new token t of sequence b (position past_b + j):
 *   block_id = block_table[b][pos / bs], slot = block_id * bs + pos % bs,
 *   key_cache[slot, k, :] = key[t, k, :], value_cache likewise.
 * A -1 entry means "not mapped": nothing is written for that token.
 * Other out-of-range entries are bad device data. */
int oracle_cache_write(const uint16_t* key, const uint16_t* value,
                       uint16_t* key_cache, uint16_t* value_cache,
                       const int32_t* block_table, int MB,
                       const int32_t* cum, const int32_t* past, int B, int T,
                       int Hk, int D, int bs, int NB) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  size_t row = (size_t)Hk * D;
  for (int b = 0; b < B; ++b) {
    for (int t = cum[b]; t < cum[b + 1]; ++t) {
      int pos = past[b] + (t - cum[b]);
      int i = pos / bs;
      if (i >= MB) return ORACLE_BAD_DEVICE_DATA;
      int blk = block_table[(size_t)b * MB + i];
      if (blk == -1) continue;
      if (blk < -1 || blk >= NB) return ORACLE_BAD_DEVICE_DATA;
      size_t slot = (size_t)blk * bs + pos % bs;
      memcpy(key_cache + slot * row, key + (size_t)t * row, row * sizeof(uint16_t));
      memcpy(value_cache + slot * row, value + (size_t)t * row, row * sizeof(uint16_t));
    }
  }
  return ORACLE_OK;
}

/* ---- attention (CUDA design section 8 note P5, section 9) ---- */

/* Output rows r in [row_begin, row_end), r = t * H + h, each D doubles in
 * out[(r - row_begin) * D ...].  query holds the (already rotated) fp16 Q.
 * For row (t, h): b owns t, j = t - cum[b], pos = past_b + j,
 * kv_len = pos + 1, kv head k = h / (H / Hk), admitted positions
 * p in [lo, kv_len) with lo = max(0, kv_len - W) when W >= 1 else 0, minus
 * positions whose block_table entry is -1.  x_p = scale * <q, K_p>,
 * optionally x_p = softcap * tanh(x_p / softcap); out = sum_p w_p V_p / sum_p w_p
 * with w_p = exp(x_p - max_p x_p); no admitted position gives out = 0.
 * scale == 0 selects 1/sqrt(D). */
int oracle_attention(const uint16_t* query, const uint16_t* key_cache,
                     const uint16_t* value_cache, const int32_t* block_table,
                     int MB, const int32_t* cum, const int32_t* past, int B,
                     int T, int H, int Hk, int D, int bs, int NB, double scale,
                     double softcap, int window, long long row_begin,
                     long long row_end, double* out) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  if (Hk <= 0 || H % Hk != 0) return ORACLE_BAD_ARGUMENT;
  if (!(window == -1 || window >= 1)) return ORACLE_BAD_ARGUMENT;
  if (softcap < 0) return ORACLE_BAD_ARGUMENT;
  if (row_begin < 0 || row_end > (long long)T * H || row_begin > row_end)
    return ORACLE_BAD_ARGUMENT;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int G = H / Hk;
  double q[1024];
  if (D > 1024) return ORACLE_BAD_ARGUMENT;
  for (long long r = row_begin; r < row_end; ++r) {
    int t = (int)(r / H), h = (int)(r % H);
    int k = h / G;
    int b = owner_of_row(cum, B, t);
    int pos = past[b] + (t - cum[b]);
    int kv_len = pos + 1;
    int lo = 0;
    if (window >= 1 && kv_len - window > 0) lo = kv_len - window;
    double* o = out + (size_t)(r - row_begin) * D;
    for (int c = 0; c < D; ++c) {
      q[c] = oracle_half_to_double(query[((size_t)t * H + h) * D + c]);
      o[c] = 0.0;
    }
    /* pass 1: scores and their maximum */
    double xmax = -INFINITY;
    int any = 0;
    for (int p = lo; p < kv_len; ++p) {
      if (p / bs >= MB) return ORACLE_BAD_DEVICE_DATA;
      int blk = block_table[(size_t)b * MB + p / bs];
      if (blk == -1) continue;
      if (blk < -1 || blk >= NB) return ORACLE_BAD_DEVICE_DATA;
      const uint16_t* kr = key_cache + (((size_t)blk * bs + p % bs) * Hk + k) * D;
      double x = 0.0;
      for (int c = 0; c < D; ++c) x += q[c] * oracle_half_to_double(kr[c]);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      if (x > xmax) xmax = x;
      any = 1;
    }
    if (!any) continue; /* fully masked row: output stays 0 */
    /* pass 2: weights and the weighted sum of V */
    double denom = 0.0;
    for (int p = lo; p < kv_len; ++p) {
      int blk = block_table[(size_t)b * MB + p / bs];
      if (blk == -1) continue;
      size_t slot = (size_t)blk * bs + p % bs;
      const uint16_t* kr = key_cache + (slot * Hk + k) * D;
      const uint16_t* vr = value_cache + (slot * Hk + k) * D;
      double x = 0.0;
      for (int c = 0; c < D; ++c) x += q[c] * oracle_half_to_double(kr[c]);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      double w = exp(x - xmax);
      denom += w;
      for (int c = 0; c < D; ++c) o[c] += w * oracle_half_to_double(vr[c]);
    }
    for (int c = 0; c < D; ++c) o[c] /= denom;
  }
  return ORACLE_OK;
}
