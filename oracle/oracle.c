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
 *     a row with no admitted key outputs 0, not NaN;
 *   - "PagedAttention - CUDA Design Document" section 7 (QK-Norm: per-head
 *     RMS normalization of Q and K, before rotary, the normalized K cached)
 *     and section 4 (packed QKV: query rows [Q heads | K heads | V heads]
 *     when key and value are absent);
 *   - "PagedAttention - CUDA Design Document" section 12 (multi-head latent
 *     attention: one cache of latent rows, V = their first v_head_size
 *     channels, rotary over channels [rotary_offset, rotary_offset + R));
 *   - "PagedAttention - CUDA Design Document" section 8 (quantized cache:
 *     int8 or float8 e4m3fn codes, symmetric, dequantized as code * scale,
 *     PER_TENSOR scale [1] or PER_CHANNEL scale [kv_num_heads * head_size],
 *     K and V quantized as they are written) and section 6.1 (head_sink: one
 *     extra logit s_h per query head that enters the softmax denominator only,
 *     m = max(s_h, max_j x_j)).
 *
 * Quantize-on-write reading.  The pages fix dequantization (x = q * scale,
 * zero point 0) but not the rounding of the write.  This oracle takes the
 * plainest one: y = x / scale in fp32 (IEEE division), then int8 = y rounded
 * to nearest-even and saturated to [-128, 127] (NaN -> 0: int8 has no NaN),
 * e4m3fn = y rounded to nearest-even and saturated to the largest finite
 * value (+-448; NaN stays NaN).
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
 * bfloat16.  The kernel is registered for fp16 and bfloat16 activations,
 * each with a cache of its own type or an 8-bit one ("PagedAttention - CUDA
 * Design Document", section 8.2); this oracle covers both.  With a
 * bfloat16 cache every 16-bit input (query, key, value, the pools, the
 * cos/sin tables, head_sink) is read as bfloat16 (exact in fp64), rotary
 * runs the same fp32 operation order and rounds each y to bfloat16 to
 * nearest-even, and the cache write copies the bits.  Over an 8-bit cache
 * (ORACLE_ACT_BF16 added to the cache type) the activations are bfloat16
 * the same way and each written value is quantized from its bfloat16 value
 * exactly as an fp16 value would be.
 *
 * Layouts (row-major): query [T, H*D]; key, value [T, Hk*D];
 * key_cache, value_cache [NB, bs, Hk, D]; block_table [B, MB];
 * cum [B+1]; past [B]; cos/sin [P, R/2].
 */
#include <math.h>
#include <stddef.h>
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

/* ---- bfloat16 conversions, written from the format definition ---- */

/* Exact bfloat16 -> double.  1 sign bit, 8 exponent bits (bias 127), 7
 * fraction bits: the upper half of an IEEE binary32 word. */
double oracle_bf16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133); /* subnormal: fraction * 2^(1 - 127 - 7) */
  } else if (e == 255) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(128 + f), e - 134);
  }
  return sign ? -v : v;
}

/* double -> bfloat16, round to nearest, ties to even (single rounding). */
uint16_t oracle_double_to_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return sign | 0x7fc0;
  double a = fabs(x);
  /* largest finite 0x7f7f = (2 - 2^-7) * 2^127; halfway to 2^128 rounds up */
  if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return sign | 0x7f80;
  if (a < ldexp(1.0, -126)) {
    /* subnormal quantum is 2^-133; scaling by 2^133 is exact */
    double m = nearbyint(ldexp(a, 133));
    return sign | (uint16_t)m; /* m == 128 encodes the smallest normal */
  }
  int e;
  (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
  double m = nearbyint(ldexp(a, 8 - e)); /* significand in [128, 256] */
  int ee = e - 1;
  if (m == 256.0) {
    m = 128.0;
    ee += 1;
  }
  if (ee > 127) return sign | 0x7f80;
  return sign | (uint16_t)((ee + 127) << 7) | (uint16_t)((int)m - 128);
}

/* A 16-bit element (fp16 or bf16 bits) as a double. */
static double elem16_to_double(uint16_t v, int bf16) {
  return bf16 ? oracle_bf16_to_double(v) : oracle_half_to_double(v);
}

/* ---- float8 e4m3fn, written from the format definition ---- */

/* Exact e4m3fn -> double.  1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits; exponent 0 is subnormal (fraction * 2^-9); there is no infinity and
 * the one NaN pattern per sign is exponent 15 with fraction 7. */
double oracle_e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int f = c & 7;
  double v;
  if (e == 15 && f == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)f, -9);
  } else {
    v = ldexp((double)(8 + f), e - 10);
  }
  return sign ? -v : v;
}

/* fp32 -> e4m3fn, round to nearest, ties to even; finite values beyond the
 * largest finite magnitude (448) and infinities saturate to +-448; NaN maps
 * to the NaN pattern. */
uint8_t oracle_float_to_e4m3(float x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7e;
  if (a < ldexp(1.0, -6)) {
    /* subnormal quantum is 2^-9; scaling by 2^9 is exact */
    double m = nearbyint(ldexp(a, 9));
    return sign | (uint8_t)m; /* m == 8 encodes the smallest normal */
  }
  int e;
  (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
  double m = nearbyint(ldexp(a, 4 - e)); /* significand in [8, 16] */
  int ee = e - 1;
  if (m == 16.0) {
    m = 8.0;
    ee += 1;
  }
  if (ee > 8 || (ee == 8 && m > 14.0)) return sign | 0x7e;
  return sign | (uint8_t)((ee + 7) << 3) | (uint8_t)((int)m - 8);
}

/* Cache element types: fp16 (no quantization), int8, float8 e4m3fn. */
#define ORACLE_CACHE_FP16 0
#define ORACLE_CACHE_INT8 1
#define ORACLE_CACHE_FP8 2
#define ORACLE_CACHE_BF16 3 /* 16-bit cache of bfloat16 elements */
/* Added to an 8-bit cache type: the activations (query, key, value,
 * head_sink) are bfloat16 (section 8.2 registers bfloat16 activations with
 * int8 and float8 caches too); a bfloat16 cache implies it. */
#define ORACLE_ACT_BF16 16
#define ORACLE_CACHE_TYPE(t) ((t) & 15)

/* Code of 16-bit value h (fp16, or bfloat16 with ORACLE_ACT_BF16) under
 * scale s (reading stated in the header). */
uint8_t oracle_quantize(uint16_t h, float s, int cache_dtype) {
  float y = (float)elem16_to_double(h, (cache_dtype & ORACLE_ACT_BF16) != 0) / s;
  if (ORACLE_CACHE_TYPE(cache_dtype) == ORACLE_CACHE_FP8) return oracle_float_to_e4m3(y);
  float r = nearbyintf(y);
  if (r != r) r = 0.0f; /* int8 has no NaN: a NaN value stores code 0 */
  if (r > 127.0f) r = 127.0f;
  if (r < -128.0f) r = -128.0f;
  return (uint8_t)(int8_t)r;
}

/* Value of cache element i of a row (fp16 bits or an 8-bit code), as a
 * double: code * scale for the 8-bit types. */
static double cache_value(const void* row, int i, int cache_dtype, double scale) {
  if (cache_dtype == ORACLE_CACHE_FP16) return oracle_half_to_double(((const uint16_t*)row)[i]);
  if (cache_dtype == ORACLE_CACHE_BF16) return oracle_bf16_to_double(((const uint16_t*)row)[i]);
  uint8_t c = ((const uint8_t*)row)[i];
  if (cache_dtype == ORACLE_CACHE_INT8) return (double)(int8_t)c * scale;
  return oracle_e4m3_to_double(c) * scale;
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
int oracle_rotary_offset(const uint16_t* x, uint16_t* y, int T, int nheads, int D,
                         const int32_t* cum, const int32_t* past, int B,
                         const uint16_t* cos_cache, const uint16_t* sin_cache,
                         int half_rot, int max_position, int interleaved, int offset);

/* Rotary at channel offset 0 (the common case). */
int oracle_rotary(const uint16_t* x, uint16_t* y, int T, int nheads, int D,
                  const int32_t* cum, const int32_t* past, int B,
                  const uint16_t* cos_cache, const uint16_t* sin_cache,
                  int half_rot, int max_position, int interleaved) {
  return oracle_rotary_offset(x, y, T, nheads, D, cum, past, B, cos_cache, sin_cache, half_rot, max_position,
                              interleaved, 0);
}

/* Rotary over channels [offset, offset + 2*half_rot) of every head (CUDA
 * design section 12.5, rotary_offset; the pairs are taken inside that
 * range), every other channel copied. */
static int rotary_impl(const uint16_t* x, uint16_t* y, int T, int nheads, int D, const int32_t* cum,
                       const int32_t* past, int B, const uint16_t* cos_cache, const uint16_t* sin_cache,
                       int half_rot, int max_position, int interleaved, int offset, int bf16);

int oracle_rotary_offset(const uint16_t* x, uint16_t* y, int T, int nheads, int D,
                         const int32_t* cum, const int32_t* past, int B,
                         const uint16_t* cos_cache, const uint16_t* sin_cache,
                         int half_rot, int max_position, int interleaved, int offset) {
  return rotary_impl(x, y, T, nheads, D, cum, past, B, cos_cache, sin_cache, half_rot, max_position, interleaved,
                     offset, 0);
}

/* The same rotation of bfloat16 rows with bfloat16 tables: each y rounded
 * to bfloat16 to nearest-even. */
int oracle_rotary_bf16(const uint16_t* x, uint16_t* y, int T, int nheads, int D,
                       const int32_t* cum, const int32_t* past, int B,
                       const uint16_t* cos_cache, const uint16_t* sin_cache,
                       int half_rot, int max_position, int interleaved, int offset) {
  return rotary_impl(x, y, T, nheads, D, cum, past, B, cos_cache, sin_cache, half_rot, max_position, interleaved,
                     offset, 1);
}

static int rotary_impl(const uint16_t* x, uint16_t* y, int T, int nheads, int D, const int32_t* cum,
                       const int32_t* past, int B, const uint16_t* cos_cache, const uint16_t* sin_cache,
                       int half_rot, int max_position, int interleaved, int offset, int bf16) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  if (offset < 0 || offset + 2 * half_rot > D || half_rot < 0) return ORACLE_BAD_ARGUMENT;
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
        int i1 = offset + (interleaved ? 2 * i : i);
        int i2 = offset + (interleaved ? 2 * i + 1 : i + half_rot);
        float x1 = (float)elem16_to_double(xr[i1], bf16);
        float x2 = (float)elem16_to_double(xr[i2], bf16);
        float c = (float)elem16_to_double(cos_cache[(size_t)pos * half_rot + i], bf16);
        float s = (float)elem16_to_double(sin_cache[(size_t)pos * half_rot + i], bf16);
        float t1 = x1 * c;
        float t2 = x2 * s;
        float y1 = t1 - t2;
        float t3 = x2 * c;
        float t4 = x1 * s;
        float y2 = t3 + t4;
        tmp[i1] = bf16 ? oracle_double_to_bf16((double)y1) : oracle_double_to_half((double)y1);
        tmp[i2] = bf16 ? oracle_double_to_bf16((double)y2) : oracle_double_to_half((double)y2);
      }
      memcpy(yr, tmp, sizeof(uint16_t) * D);
    }
  }
  return ORACLE_OK;
}

/* ---- QK-Norm (CUDA design section 7.1) ---- */

/* RMS normalization of every head of every row of x ([T, nheads*D] fp16),
 * written as fp16 to y (may alias x): per head
 *   y[c] = fp16( (x[c] * r) * w[c] ),  r = 1 / sqrt(sum_j x[j]^2 / D + eps),
 * the sum of squares in fp32.  The pages fix the formula and an fp32 sum,
 * not its order; this oracle takes the plainest one: one running fp32 sum
 * over the channels in ascending order, one rounding per square and per
 * add.  The mean is the sum times 1/D (exact: D is a power of two), then
 * + eps, IEEE square root, IEEE reciprocal. */
static int qk_norm_impl(const uint16_t* x, uint16_t* y, int T, int nheads, int D, const uint16_t* w, float eps,
                        int bf16) {
  if (D <= 0 || D > 1024 || (D & (D - 1)) != 0) return ORACLE_BAD_ARGUMENT;
  for (int t = 0; t < T; ++t) {
    for (int h = 0; h < nheads; ++h) {
      const uint16_t* xr = x + ((size_t)t * nheads + h) * D;
      uint16_t* yr = y + ((size_t)t * nheads + h) * D;
      float sum = 0.0f;
      for (int c = 0; c < D; ++c) {
        float v = (float)elem16_to_double(xr[c], bf16);
        float sq = v * v;
        sum = sum + sq;
      }
      float mean = sum * (1.0f / (float)D);
      float v = mean + eps;
      float r = 1.0f / sqrtf(v);
      uint16_t tmp[1024];
      for (int c = 0; c < D; ++c) {
        float a = (float)elem16_to_double(xr[c], bf16) * r;
        float b = a * (float)elem16_to_double(w[c], bf16);
        tmp[c] = bf16 ? oracle_double_to_bf16((double)b) : oracle_double_to_half((double)b);
      }
      memcpy(yr, tmp, sizeof(uint16_t) * D);
    }
  }
  return ORACLE_OK;
}

int oracle_qk_norm(const uint16_t* x, uint16_t* y, int T, int nheads, int D, const uint16_t* w, float eps) {
  return qk_norm_impl(x, y, T, nheads, D, w, eps, 0);
}

/* The same normalization of bfloat16 rows with a bfloat16 weight, each
 * output rounded to bfloat16 to nearest-even. */
int oracle_qk_norm_bf16(const uint16_t* x, uint16_t* y, int T, int nheads, int D, const uint16_t* w, float eps) {
  return qk_norm_impl(x, y, T, nheads, D, w, eps, 1);
}

/* ---- reshape_and_cache (CUDA design section 5.1 derived slot, 5.2
 * explicit slot_mapping) ---- */

/* Destination slot of packed row t of sequence b at position pos, or -1 for
 * no write.  With slot_mapping (section 5.2) the entry is authoritative:
 * -1 skips the row, other values must lie in [0, NB*bs).  Without it the
 * slot is derived from block_table (section 5.1).  Returns -2 for bad
 * device data. */
static long long write_slot(const int32_t* slot_mapping, const int32_t* block_table, int MB, int b, int t,
                            int pos, int bs, int NB) {
  if (slot_mapping) {
    long long s = slot_mapping[t];
    if (s == -1) return -1;
    if (s < 0 || s >= (long long)NB * bs) return -2;
    return s;
  }
  int i = pos / bs;
  if (i >= MB) return -2;
  int blk = block_table[(size_t)b * MB + i];
  if (blk == -1) return -1;
  if (blk < -1 || blk >= NB) return -2;
  return (long long)blk * bs + pos % bs;
}

/* For every new token t of sequence b (position past_b + j):
 *   block_id = block_table[b][pos / bs], slot = block_id * bs + pos % bs,
 *   key_cache[slot, k, :] = key[t, k, :], value_cache likewise.
 * A -1 entry means "not mapped": nothing is written for that token.
 * Other out-of-range entries are bad device data.  slot_mapping (may be
 * NULL) replaces the derivation: slot = slot_mapping[t], -1 = no write. */
int oracle_cache_write(const uint16_t* key, const uint16_t* value,
                       uint16_t* key_cache, uint16_t* value_cache,
                       const int32_t* block_table, int MB,
                       const int32_t* cum, const int32_t* past, int B, int T,
                       int Hk, int D, int bs, int NB, const int32_t* slot_mapping) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  size_t row = (size_t)Hk * D;
  for (int b = 0; b < B; ++b) {
    for (int t = cum[b]; t < cum[b + 1]; ++t) {
      int pos = past[b] + (t - cum[b]);
      long long ws = write_slot(slot_mapping, block_table, MB, b, t, pos, bs, NB);
      if (ws == -1) continue;
      if (ws < 0) return ORACLE_BAD_DEVICE_DATA;
      size_t slot = (size_t)ws;
      memcpy(key_cache + slot * row, key + (size_t)t * row, row * sizeof(uint16_t));
      memcpy(value_cache + slot * row, value + (size_t)t * row, row * sizeof(uint16_t));
    }
  }
  return ORACLE_OK;
}

/* Quantized write (CUDA design section 8.4): as oracle_cache_write, but
 * every element is stored as its 8-bit code under the element's scale:
 * per_channel = 0 -> scale[0]; per_channel = 1 -> scale[k * D + c]. */
int oracle_cache_write_quant(const uint16_t* key, const uint16_t* value,
                             uint8_t* key_cache, uint8_t* value_cache,
                             const float* k_scale, const float* v_scale,
                             int per_channel, int cache_dtype,
                             const int32_t* block_table, int MB,
                             const int32_t* cum, const int32_t* past, int B, int T,
                             int Hk, int D, int bs, int NB, const int32_t* slot_mapping) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  if (ORACLE_CACHE_TYPE(cache_dtype) != ORACLE_CACHE_INT8 && ORACLE_CACHE_TYPE(cache_dtype) != ORACLE_CACHE_FP8)
    return ORACLE_BAD_ARGUMENT;
  size_t row = (size_t)Hk * D;
  for (int b = 0; b < B; ++b) {
    for (int t = cum[b]; t < cum[b + 1]; ++t) {
      int pos = past[b] + (t - cum[b]);
      long long ws = write_slot(slot_mapping, block_table, MB, b, t, pos, bs, NB);
      if (ws == -1) continue;
      if (ws < 0) return ORACLE_BAD_DEVICE_DATA;
      size_t slot = (size_t)ws;
      for (size_t e = 0; e < row; ++e) {
        size_t si = per_channel ? e : 0; /* e = k * D + c */
        key_cache[slot * row + e] = oracle_quantize(key[(size_t)t * row + e], k_scale[si], cache_dtype);
        value_cache[slot * row + e] = oracle_quantize(value[(size_t)t * row + e], v_scale[si], cache_dtype);
      }
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
/* General form.  key_cache / value_cache hold fp16 bits (cache_dtype 0),
 * bfloat16 bits (cache_dtype 3: query and head_sink are then bfloat16 too)
 * or 8-bit codes (cache_dtype 1, 2; + ORACLE_ACT_BF16 for a bfloat16 query
 * and sink) dequantized as code * scale with k_scale / v_scale indexed
 * by [k * D + c] (per_channel = 1) or [0]; head_sink ([H] fp16, may be NULL)
 * adds exp(s_h - m) to the denominator, m = max(s_h, max_p x_p). */
int oracle_attention_ex(const uint16_t* query, const void* key_cache,
                        const void* value_cache, int cache_dtype,
                        const float* k_scale, const float* v_scale, int per_channel,
                        const uint16_t* head_sink, const int32_t* block_table,
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
  /* bfloat16 query and sink: a bfloat16 cache, or ORACLE_ACT_BF16 with an 8-bit one */
  const int bf16 = cache_dtype == ORACLE_CACHE_BF16 || (cache_dtype & ORACLE_ACT_BF16) != 0;
  cache_dtype = ORACLE_CACHE_TYPE(cache_dtype);
  const int c16 = cache_dtype == ORACLE_CACHE_FP16 || cache_dtype == ORACLE_CACHE_BF16;
  if (!c16 && (k_scale == NULL || v_scale == NULL)) return ORACLE_BAD_ARGUMENT;
  size_t esize = c16 ? 2 : 1;
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
      q[c] = elem16_to_double(query[((size_t)t * H + h) * D + c], bf16);
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
      const void* kr = (const uint8_t*)key_cache + (((size_t)blk * bs + p % bs) * Hk + k) * D * esize;
      double x = 0.0;
      for (int c = 0; c < D; ++c)
        x += q[c] * cache_value(kr, c, cache_dtype, k_scale ? k_scale[per_channel ? k * D + c : 0] : 1.0);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      if (x > xmax) xmax = x;
      any = 1;
    }
    if (!any) continue; /* fully masked row: output stays 0 */
    double sink = head_sink ? elem16_to_double(head_sink[h], bf16) : -INFINITY;
    if (sink > xmax) xmax = sink;
    /* pass 2: weights and the weighted sum of V */
    double denom = 0.0;
    for (int p = lo; p < kv_len; ++p) {
      int blk = block_table[(size_t)b * MB + p / bs];
      if (blk == -1) continue;
      size_t slot = (size_t)blk * bs + p % bs;
      const void* kr = (const uint8_t*)key_cache + (slot * Hk + k) * D * esize;
      const void* vr = (const uint8_t*)value_cache + (slot * Hk + k) * D * esize;
      double x = 0.0;
      for (int c = 0; c < D; ++c)
        x += q[c] * cache_value(kr, c, cache_dtype, k_scale ? k_scale[per_channel ? k * D + c : 0] : 1.0);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      double w = exp(x - xmax);
      denom += w;
      for (int c = 0; c < D; ++c)
        o[c] += w * cache_value(vr, c, cache_dtype, v_scale ? v_scale[per_channel ? k * D + c : 0] : 1.0);
    }
    if (head_sink) denom += exp(sink - xmax); /* the sink's term: denominator only */
    for (int c = 0; c < D; ++c) o[c] /= denom;
  }
  return ORACLE_OK;
}

/* Absorbed multi-head latent attention (CUDA design section 12): one cache
 * [NB, bs, 1, D] (D = latent width + rotary width), every query head h of
 * row t attends with x_p = scale * <q[t,h,0:D], L_p[0:D]> (optionally
 * softcapped) and the output is the softmax-weighted sum of L_p[0:Dv], the
 * first Dv channels of the same cached rows.  Masks as oracle_attention_ex.
 * out holds Dv doubles per row. */
int oracle_attention_latent(const uint16_t* query, const uint16_t* latent_cache, const int32_t* block_table,
                            int MB, const int32_t* cum, const int32_t* past, int B, int T, int H, int D, int Dv,
                            int bs, int NB, double scale, double softcap, int window, long long row_begin,
                            long long row_end, double* out) {
  int st = check_lengths(cum, past, B, T);
  if (st) return st;
  if (Dv < 1 || Dv > D || D > 1024 || scale <= 0.0) return ORACLE_BAD_ARGUMENT;
  if (!(window == -1 || window >= 1) || softcap < 0) return ORACLE_BAD_ARGUMENT;
  if (row_begin < 0 || row_end > (long long)T * H || row_begin > row_end) return ORACLE_BAD_ARGUMENT;
  double q[1024];
  for (long long r = row_begin; r < row_end; ++r) {
    int t = (int)(r / H), h = (int)(r % H);
    int b = owner_of_row(cum, B, t);
    int pos = past[b] + (t - cum[b]);
    int kv_len = pos + 1;
    int lo = (window >= 1 && kv_len - window > 0) ? kv_len - window : 0;
    double* o = out + (size_t)(r - row_begin) * Dv;
    for (int c = 0; c < D; ++c) q[c] = oracle_half_to_double(query[((size_t)t * H + h) * D + c]);
    for (int c = 0; c < Dv; ++c) o[c] = 0.0;
    double xmax = -INFINITY;
    int any = 0;
    for (int p = lo; p < kv_len; ++p) {
      if (p / bs >= MB) return ORACLE_BAD_DEVICE_DATA;
      int blk = block_table[(size_t)b * MB + p / bs];
      if (blk == -1) continue;
      if (blk < -1 || blk >= NB) return ORACLE_BAD_DEVICE_DATA;
      const uint16_t* lr = latent_cache + ((size_t)blk * bs + p % bs) * D;
      double x = 0.0;
      for (int c = 0; c < D; ++c) x += q[c] * oracle_half_to_double(lr[c]);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      if (x > xmax) xmax = x;
      any = 1;
    }
    if (!any) continue;
    double denom = 0.0;
    for (int p = lo; p < kv_len; ++p) {
      int blk = block_table[(size_t)b * MB + p / bs];
      if (blk == -1) continue;
      const uint16_t* lr = latent_cache + ((size_t)blk * bs + p % bs) * D;
      double x = 0.0;
      for (int c = 0; c < D; ++c) x += q[c] * oracle_half_to_double(lr[c]);
      x *= scale;
      if (softcap > 0.0) x = softcap * tanh(x / softcap);
      double w = exp(x - xmax);
      denom += w;
      for (int c = 0; c < Dv; ++c) o[c] += w * oracle_half_to_double(lr[c]);
    }
    for (int c = 0; c < Dv; ++c) o[c] /= denom;
  }
  return ORACLE_OK;
}

/* fp16 cache, no sink. */
int oracle_attention(const uint16_t* query, const uint16_t* key_cache,
                     const uint16_t* value_cache, const int32_t* block_table,
                     int MB, const int32_t* cum, const int32_t* past, int B,
                     int T, int H, int Hk, int D, int bs, int NB, double scale,
                     double softcap, int window, long long row_begin,
                     long long row_end, double* out) {
  return oracle_attention_ex(query, key_cache, value_cache, ORACLE_CACHE_FP16, NULL, NULL, 0, NULL,
                             block_table, MB, cum, past, B, T, H, Hk, D, bs, NB, scale, softcap,
                             window, row_begin, row_end, out);
}
