/*
 * Paged-KV GQA attention oracle: a plain, slow, fp64 CPU statement of what
 * libpagedattn computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path; nothing in the product calls it.
 *
 * Sources (page title, section):
 *   [P1] "Модуль 12: Финальный проект: мини-движок инференса" (LLM Inference
 *        Systems course), task 12.1 and the qwen_serve/paged.py listing
 *        (PagedKVCache docstring, PagedKVCache.write, PagedKVCache.read) and the
 *        qwen_serve/model.py listing (Qwen3Model.forward, attention loop).
 *   [P2] "Модуль 04: KV-кэш и арифметика памяти", section 1 (the attention
 *        output formula), kv_cache.py section 2 (attend: GQA by repeating KV
 *        heads, mask on absolute positions k_pos <= q_pos).
 *   [P3] "Phase 10: LLMs from Scratch — Inference Optimization", step 2
 *        (scaled dot-product attention with a causal mask).
 *
 * Every floating-point input arrives as raw 16-bit patterns (IEEE binary16 or
 * bfloat16) and is widened exactly to double.  Nothing is rounded on the way:
 * scores, softmax and the weighted sum of values are all fp64, and masked keys
 * are excluded from the sums rather than filled with a large negative number.
 *
 * Layout of one layer's pool [P1, PagedKVCache docstring]: K and V each as
 * [num_blocks][block_size][num_kv_heads][head_dim]; block b is the outer
 * index, the in-block slot the next one.  A flat slot number is
 * block * block_size + offset.
 *
 * Sliding window [P2 section 4 (ring buffer of capacity W) and section 5.2]:
 * with a window W > 0 the query at absolute position p sees only the keys at
 * positions max(0, p - W + 1) .. p (the mask stays on absolute positions);
 * blocks wholly before that range are never read.
 *
 * The int8 pool [P2 section 5, KV8Cache]: K and V codes int8 in the same
 * layout, one fp32 scale per (token, KV head) for K and one for V.  The
 * quantising write and the dequantising read follow the pages' fp32 steps
 * exactly; attention then runs in fp64 on the dequantised values.
 *
 * q/k RMSNorm and rotary embedding before the write [P1 qwen_serve/model.py:
 * rms_norm, _rope_tables, _rotate_half, apply_rope and their use in
 * Qwen3Model.forward; P2 section 4: the key is rotated to its absolute position
 * before it is stored].  These steps have their precision fixed by the page:
 * the mean of squares and the reciprocal square root in fp32, every other
 * operation a 16-bit tensor operation (computed exactly, rounded once to the
 * 16-bit format, ties to even).  The oracle takes the same rounding points.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* ---- exact widening of the 16-bit formats --------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -133);              /* f * 2^-126 * 2^-7 */
  } else if (e == 255) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(128 + f), e - 134);   /* (1 + f/128) * 2^(e-127) */
  }
  return sign ? -mag : mag;
}

static double widen(uint16_t bits, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(bits) : oracle_f16_to_f64(bits);
}

/*
 * The 16-bit value nearest to x, ties to even (IEEE round to nearest): with f
 * fraction bits and exponent bias b, a finite value of magnitude in
 * [2^(e), 2^(e+1)) for e >= 1 - b is a multiple of 2^(e - f); below 2^(1 - b)
 * (subnormal) of 2^(1 - b - f).  Magnitudes that round beyond the largest
 * finite value become infinity.
 */
uint16_t oracle_f64_to_16(double x, int dtype) {
  const int f = dtype == ORACLE_BF16 ? 7 : 10;
  const int b = dtype == ORACLE_BF16 ? 127 : 15;
  const int emax = dtype == ORACLE_BF16 ? 127 : 15;          /* largest unbiased exponent */
  const uint16_t sign = signbit(x) ? (uint16_t)0x8000 : 0;
  const uint16_t inf = (uint16_t)((2 * emax + 1) << f);      /* exponent field all ones */
  if (isnan(x)) return (uint16_t)(sign | inf | (1 << (f - 1)));
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | inf);
  int e2;
  frexp(a, &e2);                                             /* a = m 2^e2, m in [0.5, 1) */
  int e = a == 0.0 ? 1 - b : e2 - 1;
  if (e < 1 - b) e = 1 - b;
  const double quantum = ldexp(1.0, e - f);
  const double r = nearbyint(a / quantum) * quantum;         /* round to nearest, ties to even */
  if (r == 0.0) return sign;
  frexp(r, &e2);
  e = e2 - 1;
  if (e > emax) return (uint16_t)(sign | inf);
  if (e < 1 - b) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, 1 - b - f)));   /* subnormal */
  const uint16_t frac = (uint16_t)(r / ldexp(1.0, e - f) - ldexp(1.0, f));
  return (uint16_t)(sign | ((e + b) << f) | frac);
}

static uint16_t narrow(double x, int dtype) { return oracle_f64_to_16(x, dtype); }

/*
 * FP8 E4M3 (the "fn" variant: 4 exponent bits, bias 7, 3 fraction bits, no
 * infinity, S.1111.111 is NaN, largest finite 448).  Decoding: exponent field
 * 0 is subnormal, f * 2^-9; otherwise (1 + f / 8) * 2^(e - 7).
 */
double oracle_e4m3_to_f64(uint8_t c) {
  const int sign = (c >> 7) & 1, e = (c >> 3) & 0xf, f = c & 7;
  double mag;
  if (e == 15 && f == 7) {
    mag = NAN;
  } else if (e == 0) {
    mag = ldexp((double)f, -9);
  } else {
    mag = ldexp((double)(8 + f), e - 10);
  }
  return sign ? -mag : mag;
}

/*
 * The E4M3 value nearest to x, ties to even; magnitudes that round beyond
 * 448 saturate to 448 (the "satfinite" conversion).  A finite value of
 * magnitude in [2^e, 2^(e+1)), e >= -6, is a multiple of 2^(e - 3); below 2^-6
 * of 2^-9.
 */
uint8_t oracle_f64_to_e4m3(double x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return (uint8_t)(sign | 0x7f);
  double a = fabs(x);
  if (a > 448.0) a = 448.0;
  int e2;
  frexp(a, &e2);
  int e = a == 0.0 ? -6 : e2 - 1;
  if (e < -6) e = -6;
  const double quantum = ldexp(1.0, e - 3);
  double r = nearbyint(a / quantum) * quantum;
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  frexp(r, &e2);
  e = e2 - 1;
  if (e < -6) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));      /* subnormal */
  const uint8_t frac = (uint8_t)(r / ldexp(1.0, e - 3) - 8.0);
  return (uint8_t)(sign | ((e + 7) << 3) | frac);
}

/* ---- KV write [P1, PagedKVCache.write] ------------------------------------- */

/*
 * For each new token t in order, copy its K and V rows (num_kv_heads x
 * head_dim 16-bit values) into flat slot slot_mapping[t] of the pool.  Tokens
 * are processed in order, so a repeated slot keeps the last token's row (the
 * page's sequential loop).  A slot outside [0, num_blocks*block_size) is
 * skipped and counted; the return value is the number of skipped tokens.
 */
int64_t oracle_kv_cache_write(uint16_t *k_cache, uint16_t *v_cache,
                              int64_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim,
                              const uint16_t *k, const uint16_t *v,
                              const int64_t *slot_mapping, int64_t num_tokens) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  int64_t skipped = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) {
      ++skipped;
      continue;
    }
    int64_t block = slot / block_size, offset = slot % block_size;
    int64_t dst = (block * block_size + offset) * row;
    for (int64_t x = 0; x < row; ++x) {
      k_cache[dst + x] = k[t * row + x];
      v_cache[dst + x] = v[t * row + x];
    }
  }
  return skipped;
}

/* ---- q/k RMSNorm + rotary embedding, then the KV write ---------------------- */

/*
 * rms_norm of one head row of head_dim 16-bit values [P1 model.py rms_norm]:
 * var = mean(x^2) and inv = rsqrt(var + eps), both fp32 (each the fp32 value
 * nearest the exact one); y = (x * inv) in fp32, rounded to the 16-bit format;
 * out = y * weight, a 16-bit product.
 */
static void rms_norm_row(const uint16_t *x, const uint16_t *weight, float eps, int32_t head_dim, int dtype,
                         uint16_t *out) {
  double ss = 0.0;
  for (int32_t i = 0; i < head_dim; ++i) {
    const double xi = widen(x[i], dtype);
    ss += xi * xi;
  }
  const float var = (float)(ss / head_dim);
  const float s = var + eps;
  const float inv = (float)(1.0 / sqrt((double)s));
  for (int32_t i = 0; i < head_dim; ++i) {
    const float y = (float)widen(x[i], dtype) * inv;
    const uint16_t yb = narrow((double)y, dtype);
    out[i] = narrow(widen(yb, dtype) * widen(weight[i], dtype), dtype);
  }
}

/*
 * Rotary embedding of one head row at one position [P1 model.py apply_rope,
 * _rotate_half; tables from _rope_tables, NeoX layout]: with h = head_dim / 2
 * and rotate_half(z) = (-z[h..), z[..h)), out = z * cos + rotate_half(z) * sin,
 * each product and the sum a 16-bit tensor operation.
 */
static void rope_row(const uint16_t *z, const uint16_t *cos_row, const uint16_t *sin_row, int32_t head_dim,
                     int dtype, uint16_t *out) {
  const int32_t h = head_dim / 2;
  for (int32_t i = 0; i < head_dim; ++i) {
    const double rot = i < h ? -widen(z[i + h], dtype) : widen(z[i - h], dtype);
    const uint16_t a = narrow(widen(z[i], dtype) * widen(cos_row[i], dtype), dtype);
    const uint16_t b = narrow(rot * widen(sin_row[i], dtype), dtype);
    const float sum = (float)(widen(a, dtype) + widen(b, dtype));
    out[i] = narrow((double)sum, dtype);
  }
}

/*
 * For each token t in order [P1 Qwen3Model.forward: q_norm/k_norm, then
 * apply_rope at the token's absolute position, then PagedKVCache.write of the
 * rotated k and the unchanged v; P2 section 4: rotate before storing]:
 *   q_out[t][g] = rope(rms_norm(q[t][g], q_weight), positions[t]) for each query head g,
 *   the pool slot slot_mapping[t] receives rope(rms_norm(k[t][h], k_weight)) and v[t][h].
 * A token whose position lies outside [0, max_position) or whose slot lies
 * outside the pool is skipped entirely (nothing written); returns the number
 * of skipped tokens.
 */
int64_t oracle_qk_norm_rope_kv_write(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const uint16_t *q_weight, const uint16_t *k_weight, float eps,
                                     const uint16_t *cos_table, const uint16_t *sin_table, int32_t max_position,
                                     const int32_t *positions, const int64_t *slot_mapping, int64_t num_tokens,
                                     int32_t num_q_heads, int32_t dtype, uint16_t *q_out, uint16_t *k_cache,
                                     uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_dim) {
  int64_t skipped = 0;
  uint16_t *normed = malloc(sizeof(uint16_t) * (size_t)head_dim);
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int32_t pos = positions[t];
    const int64_t slot = slot_mapping[t];
    if (pos < 0 || pos >= max_position || slot < 0 || slot >= num_blocks * block_size) {
      ++skipped;
      continue;
    }
    const uint16_t *cos_row = cos_table + (int64_t)pos * head_dim;
    const uint16_t *sin_row = sin_table + (int64_t)pos * head_dim;
    for (int32_t g = 0; g < num_q_heads; ++g) {
      const int64_t row = (t * num_q_heads + g) * (int64_t)head_dim;
      rms_norm_row(q + row, q_weight, eps, head_dim, dtype, normed);
      rope_row(normed, cos_row, sin_row, head_dim, dtype, q_out + row);
    }
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
      const int64_t dst = (slot * num_kv_heads + h) * (int64_t)head_dim;
      rms_norm_row(k + src, k_weight, eps, head_dim, dtype, normed);
      rope_row(normed, cos_row, sin_row, head_dim, dtype, k_cache + dst);
      for (int32_t x = 0; x < head_dim; ++x) v_cache[dst + x] = v[src + x];
    }
  }
  free(normed);
  return skipped;
}

/* ---- copy-on-write block copy [P1, SequenceCache._cow_copy] --------------- */

/*
 * The page copies a shared block for the sequence that writes into it: the
 * fresh block receives every layer's K and V of the old one, k[:, dst] =
 * k[:, src].  This is one layer of that: for each pair i in order, block
 * pairs[2i + 1] of k_cache and v_cache receives block pairs[2i].  Returns the
 * number of pairs skipped because a block id lies outside [0, num_blocks).
 */
int64_t oracle_kv_block_copy(uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, const int32_t *pairs, int64_t num_pairs) {
  const int64_t per_block = (int64_t)block_size * num_kv_heads * head_dim;
  int64_t skipped = 0;
  for (int64_t i = 0; i < num_pairs; ++i) {
    const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      ++skipped;
      continue;
    }
    for (int64_t x = 0; x < per_block; ++x) {
      k_cache[dst * per_block + x] = k_cache[src * per_block + x];
      v_cache[dst * per_block + x] = v_cache[src * per_block + x];
    }
  }
  return skipped;
}

/* ---- gather read [P1, PagedKVCache.read] ----------------------------------- */

/*
 * Rows of positions [0, upto) of one KV head, gathered through a block table:
 * logical position j lives in block table entry j / block_size at in-block
 * offset j % block_size.  Writes upto*head_dim doubles to k_out and v_out.
 * Returns 0, or -1 if a needed block id is outside [0, num_blocks).
 */
static int gather_range(const uint16_t *k_cache, const uint16_t *v_cache, int dtype, int64_t num_blocks,
                        int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                        const int32_t *block_table_row, int32_t kv_head, int32_t from, int32_t upto,
                        double *k_out, double *v_out);

int oracle_gather_head(const uint16_t *k_cache, const uint16_t *v_cache, int dtype,
                       int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t *block_table_row,
                       int32_t kv_head, int32_t upto, double *k_out, double *v_out) {
  return gather_range(k_cache, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, block_table_row,
                      kv_head, 0, upto, k_out, v_out);
}

/* Rows of positions [from, upto), written from row 0 of k_out / v_out. */
static int gather_range(const uint16_t *k_cache, const uint16_t *v_cache, int dtype, int64_t num_blocks,
                        int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                        const int32_t *block_table_row, int32_t kv_head, int32_t from, int32_t upto,
                        double *k_out, double *v_out) {
  k_out -= (int64_t)from * head_dim;
  v_out -= (int64_t)from * head_dim;
  for (int32_t j = from; j < upto; ++j) {
    int32_t entry = j / block_size, offset = j % block_size;
    int64_t block = block_table_row[entry];
    if (block < 0 || block >= num_blocks) return -1;
    int64_t base = ((block * block_size + offset) * num_kv_heads + kv_head) * (int64_t)head_dim;
    for (int32_t x = 0; x < head_dim; ++x) {
      k_out[(int64_t)j * head_dim + x] = widen(k_cache[base + x], dtype);
      v_out[(int64_t)j * head_dim + x] = widen(v_cache[base + x], dtype);
    }
  }
  return 0;
}

/* ---- int8 pool: quantising write and dequantising read [P2 section 5] ------- */

/*
 * Scales are stored [num_blocks][num_kv_heads][block_size]: the scale of the
 * token in slot (block, offset) for KV head h is at (block * num_kv_heads + h)
 * * block_size + offset.  (The pages keep one scale per (position, head) of a
 * contiguous cache; this head-major order inside a block is the library's
 * paged layout of the same numbers.)
 *
 * Write, per token and KV head, for K and for V [KV8Cache.write]: the 16-bit
 * values x are widened exactly to fp32; scale = max |x| / 127 + 1e-8 and
 * code = clip(rint(x / scale), -127, 127), each an fp32 operation rounded to
 * nearest (rint: ties to even).  Returns the number of skipped slots (outside
 * the pool).
 */
int64_t oracle_kv_cache_write_q8(int8_t *k_cache, int8_t *v_cache, float *k_scale, float *v_scale,
                                 int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, const uint16_t *k, const uint16_t *v, int32_t dtype,
                                 const int64_t *slot_mapping, int64_t num_tokens) {
  int64_t skipped = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) {
      ++skipped;
      continue;
    }
    const int64_t block = slot / block_size, offset = slot % block_size;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int pass = 0; pass < 2; ++pass) {
        const uint16_t *src = (pass == 0 ? k : v) + (t * num_kv_heads + h) * (int64_t)head_dim;
        int8_t *dst = (pass == 0 ? k_cache : v_cache) + (slot * num_kv_heads + h) * (int64_t)head_dim;
        float *scl = pass == 0 ? k_scale : v_scale;
        float amax = 0.0f;
        for (int32_t x = 0; x < head_dim; ++x) {
          const float a = fabsf((float)widen(src[x], dtype));
          if (a > amax) amax = a;
        }
        float scale = amax / 127.0f;
        scale = scale + 1e-8f;
        for (int32_t x = 0; x < head_dim; ++x) {
          float c = rintf((float)widen(src[x], dtype) / scale);
          if (c > 127.0f) c = 127.0f;
          if (c < -127.0f) c = -127.0f;
          dst[x] = (int8_t)c;
        }
        scl[(block * num_kv_heads + h) * block_size + offset] = scale;
      }
    }
  }
  return skipped;
}

/* Read [KV8Cache.read]: rows of positions [0, upto) of one KV head, each value
 * code * scale as an fp32 product, widened to double.  Returns 0 or -1 (block
 * id outside the pool). */
static int gather_range_q8(const int8_t *k_cache, const int8_t *v_cache, const float *k_scale,
                           const float *v_scale, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                           int32_t head_dim, const int32_t *block_table_row, int32_t kv_head, int32_t from,
                           int32_t upto, int fp8, double *k_out, double *v_out);

int oracle_gather_head_q8(const int8_t *k_cache, const int8_t *v_cache, const float *k_scale,
                          const float *v_scale, int64_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, const int32_t *block_table_row,
                          int32_t kv_head, int32_t upto, double *k_out, double *v_out) {
  return gather_range_q8(k_cache, v_cache, k_scale, v_scale, num_blocks, block_size, num_kv_heads, head_dim,
                         block_table_row, kv_head, 0, upto, 0, k_out, v_out);
}

static int gather_range_q8(const int8_t *k_cache, const int8_t *v_cache, const float *k_scale,
                           const float *v_scale, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                           int32_t head_dim, const int32_t *block_table_row, int32_t kv_head, int32_t from,
                           int32_t upto, int fp8, double *k_out, double *v_out) {
  k_out -= (int64_t)from * head_dim;
  v_out -= (int64_t)from * head_dim;
  for (int32_t j = from; j < upto; ++j) {
    const int32_t entry = j / block_size;
    const int32_t offset = j % block_size;
    int64_t block = block_table_row[entry];
    if (block < 0 || block >= num_blocks) return -1;
    const int64_t base = ((block * block_size + offset) * num_kv_heads + kv_head) * (int64_t)head_dim;
    const int64_t sidx = (block * num_kv_heads + kv_head) * block_size + offset;
    const float ks = k_scale[sidx], vs = v_scale[sidx];
    for (int32_t x = 0; x < head_dim; ++x) {
      /* a code's value: the integer (int8) or the E4M3 number (fp8), times its scale in fp32 */
      const float kc = fp8 ? (float)oracle_e4m3_to_f64((uint8_t)k_cache[base + x]) : (float)k_cache[base + x];
      const float vc = fp8 ? (float)oracle_e4m3_to_f64((uint8_t)v_cache[base + x]) : (float)v_cache[base + x];
      const float kf = kc * ks;
      const float vf = vc * vs;
      k_out[(int64_t)j * head_dim + x] = (double)kf;
      v_out[(int64_t)j * head_dim + x] = (double)vf;
    }
  }
  return 0;
}

/* ---- one query row of attention [P1 Qwen3Model.forward; P2 section 1] ------ */

/*
 * out = sum_j p_j v_j with p_j = exp(S_j - max S) / sum_i exp(S_i - max S) and
 * S_j = scale * <q, k_j>, over the n visible keys (rows 0..n-1 of kk / vv).
 * The max is subtracted as the pages' softmax does; in exact arithmetic it
 * cancels.  s is scratch of n doubles.
 */
static void attend_row(const double *q, const double *kk, const double *vv,
                       int32_t n, int32_t d, double scale, double *s, double *out) {
  double m = -INFINITY;
  for (int32_t j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int32_t x = 0; x < d; ++x) dot += q[x] * kk[(int64_t)j * d + x];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int32_t j = 0; j < n; ++j) {
    s[j] = exp(s[j] - m);
    z += s[j];
  }
  for (int32_t x = 0; x < d; ++x) out[x] = 0.0;
  for (int32_t j = 0; j < n; ++j) {
    double p = s[j] / z;
    for (int32_t x = 0; x < d; ++x) out[x] += p * vv[(int64_t)j * d + x];
  }
}

/* ---- shared problem description and a small thread pool ------------------- */

typedef struct {
  const uint16_t *q;            /* [rows][num_q_heads][head_dim] */
  int dtype;
  const uint16_t *k_cache, *v_cache;
  int64_t num_blocks;
  int32_t block_size, num_kv_heads, head_dim;
  const int32_t *block_tables;  /* [num_groups][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;
  int32_t num_q_heads;
  double scale;
  double *out;                  /* [rows][num_q_heads][head_dim] */
  /* One "group" is a decode sequence or a prefill chunk: a block-table row
   * plus the query rows [row0, row0 + nrows) whose absolute positions are
   * pos0 + i, i < nrows.  Query row i sees keys [0, pos0 + i]. */
  int32_t num_groups;
  const int32_t *group_row0, *group_nrows, *group_pos0;
  int64_t next;                 /* work counter: (group, kv head) items */
  pthread_mutex_t lock;
  int error;
  /* int8 pool instead of k_cache / v_cache when k8 is not NULL */
  const int8_t *k8, *v8;
  const float *k_scale, *v_scale;
  /* sliding window W (0: none): row at position p sees keys max(0, p - W + 1) .. p */
  int32_t window;
  /* with k8: the codes are E4M3 numbers instead of integers */
  int fp8;
} problem_t;

static void run_item(problem_t *P, int32_t g, int32_t h, double *kk, double *vv,
                     double *s, double *qd) {
  const int32_t d = P->head_dim;
  const int32_t G = P->num_q_heads / P->num_kv_heads;
  const int32_t nrows = P->group_nrows[g], row0 = P->group_row0[g], pos0 = P->group_pos0[g];
  const int32_t nkeys = pos0 + nrows;   /* keys the last row of the group sees */
  /* first key any row of the group sees (the first row's window start) */
  const int32_t glo = (P->window > 0 && pos0 - P->window + 1 > 0) ? pos0 - P->window + 1 : 0;
  const int32_t *bt_row = P->block_tables + (int64_t)g * P->max_blocks_per_seq;
  const int grc = P->k8 ? gather_range_q8(P->k8, P->v8, P->k_scale, P->v_scale, P->num_blocks, P->block_size,
                                          P->num_kv_heads, d, bt_row, h, glo, nkeys, P->fp8, kk, vv)
                        : gather_range(P->k_cache, P->v_cache, P->dtype, P->num_blocks, P->block_size,
                                       P->num_kv_heads, d, bt_row, h, glo, nkeys, kk, vv);
  if (grc != 0) {
    pthread_mutex_lock(&P->lock);
    P->error = -1;
    pthread_mutex_unlock(&P->lock);
    return;
  }
  /* Query head qh reads KV head qh / G: the G query heads of one KV head are
   * contiguous [P1 model.py view(T, n_kv, group, D); P2 attend np.repeat]. */
  for (int32_t qh = h * G; qh < (h + 1) * G; ++qh) {
    for (int32_t i = 0; i < nrows; ++i) {
      const int64_t base = ((int64_t)(row0 + i) * P->num_q_heads + qh) * d;
      for (int32_t x = 0; x < d; ++x) qd[x] = widen(P->q[base + x], P->dtype);
      const int32_t p = pos0 + i;
      const int32_t lo = (P->window > 0 && p - P->window + 1 > 0) ? p - P->window + 1 : 0;
      attend_row(qd, kk + (int64_t)(lo - glo) * d, vv + (int64_t)(lo - glo) * d, p - lo + 1, d, P->scale, s,
                 P->out + base);
    }
  }
}

static void *worker(void *arg) {
  problem_t *P = (problem_t *)arg;
  int32_t maxkeys = 0;
  for (int32_t g = 0; g < P->num_groups; ++g)
    if (P->group_pos0[g] + P->group_nrows[g] > maxkeys) maxkeys = P->group_pos0[g] + P->group_nrows[g];
  const int32_t d = P->head_dim;
  double *kk = (double *)malloc(sizeof(double) * (size_t)(maxkeys > 0 ? maxkeys : 1) * d);
  double *vv = (double *)malloc(sizeof(double) * (size_t)(maxkeys > 0 ? maxkeys : 1) * d);
  double *s = (double *)malloc(sizeof(double) * (size_t)(maxkeys > 0 ? maxkeys : 1));
  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  if (!kk || !vv || !s || !qd) {
    pthread_mutex_lock(&P->lock);
    P->error = -2;
    pthread_mutex_unlock(&P->lock);
  } else {
    for (;;) {
      pthread_mutex_lock(&P->lock);
      int64_t item = P->next++;
      pthread_mutex_unlock(&P->lock);
      if (item >= (int64_t)P->num_groups * P->num_kv_heads) break;
      run_item(P, (int32_t)(item / P->num_kv_heads), (int32_t)(item % P->num_kv_heads), kk, vv, s, qd);
    }
  }
  free(kk);
  free(vv);
  free(s);
  free(qd);
  return NULL;
}

static int run_problem(problem_t *P, int32_t num_threads) {
  if (P->num_kv_heads <= 0 || P->num_q_heads % P->num_kv_heads != 0) return -3;
  if (num_threads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    num_threads = n > 0 ? (int32_t)n : 1;
  }
  int64_t items = (int64_t)P->num_groups * P->num_kv_heads;
  if (num_threads > items) num_threads = items > 0 ? (int32_t)items : 1;
  P->next = 0;
  P->error = 0;
  pthread_mutex_init(&P->lock, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
  int started = 0;
  for (int32_t i = 0; i < num_threads; ++i)
    if (pthread_create(&th[i], NULL, worker, P) == 0) ++started;
  if (started == 0) worker(P);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&P->lock);
  return P->error;
}

/* ---- decode [P1 Qwen3Model.forward with T = 1] ------------------------------ */

/*
 * One query token per sequence s, at absolute position context_lens[s] - 1,
 * already present in the pool: q[s][qh] attends to keys 0 .. context_lens[s]-1
 * of KV head qh / (num_q_heads / num_kv_heads).  Output [num_seqs][Hq][d] fp64.
 * Returns 0, -1 for a block id out of range, -3 for a bad head split, -4 for a
 * context length < 1 or beyond the block table.
 */
static int decode_problem(problem_t *P, const int32_t *context_lens, int32_t num_seqs,
                          int32_t num_threads);

int oracle_paged_attn_decode(const uint16_t *q, int32_t dtype,
                             const uint16_t *k_cache, const uint16_t *v_cache,
                             int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                             int32_t num_seqs, int32_t num_q_heads, double scale,
                             double *out, int32_t num_threads) {
  problem_t P = {q, dtype, k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  return decode_problem(&P, context_lens, num_seqs, num_threads);
}

/* Decode with a sliding window of W keys [P2 sections 4 and 5.2]: sequence s
 * sees positions max(0, context_lens[s] - W) .. context_lens[s] - 1. */
int oracle_paged_attn_decode_window(const uint16_t *q, int32_t dtype, const uint16_t *k_cache,
                                    const uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                                    int32_t num_kv_heads, int32_t head_dim, const int32_t *block_tables,
                                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, double scale, int32_t window, double *out,
                                    int32_t num_threads) {
  if (window < 1) return -4;
  problem_t P = {q, dtype, k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.window = window;
  return decode_problem(&P, context_lens, num_seqs, num_threads);
}

/* The same decode on the int8 pool [P2 section 5]: keys and values are the
 * dequantised fp32 numbers of KV8Cache.read. */
int oracle_paged_attn_decode_q8(const uint16_t *q, int32_t dtype, const int8_t *k_cache,
                                const int8_t *v_cache, const float *k_scale, const float *v_scale,
                                int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                int32_t head_dim, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                double scale, double *out, int32_t num_threads) {
  problem_t P = {q, dtype, NULL, NULL, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.k8 = k_cache;
  P.v8 = v_cache;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  return decode_problem(&P, context_lens, num_seqs, num_threads);
}

/*
 * The fp8 pool: the int8 pool's layout and per-(token, KV head) scales, with
 * E4M3 codes.  Write, per token and KV head, for K and for V: the values x
 * widened exactly to fp32, scale = max |x| / 448 + 1e-8 and code =
 * e4m3(x / scale) (an fp32 division, then the nearest E4M3 value, ties to
 * even; |x / scale| <= 448 by construction).  Read: e4m3 value * scale in fp32.
 * Returns the number of skipped slots (outside the pool).
 */
int64_t oracle_kv_cache_write_f8(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                                 int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, const uint16_t *k, const uint16_t *v, int32_t dtype,
                                 const int64_t *slot_mapping, int64_t num_tokens) {
  int64_t skipped = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) {
      ++skipped;
      continue;
    }
    const int64_t block = slot / block_size, offset = slot % block_size;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int pass = 0; pass < 2; ++pass) {
        const uint16_t *src = (pass == 0 ? k : v) + (t * num_kv_heads + h) * (int64_t)head_dim;
        uint8_t *dst = (pass == 0 ? k_cache : v_cache) + (slot * num_kv_heads + h) * (int64_t)head_dim;
        float *scl = pass == 0 ? k_scale : v_scale;
        float amax = 0.0f;
        for (int32_t x = 0; x < head_dim; ++x) {
          const float a = fabsf((float)widen(src[x], dtype));
          if (a > amax) amax = a;
        }
        float scale = amax / 448.0f;
        scale += 1e-8f;
        for (int32_t x = 0; x < head_dim; ++x) {
          const float y = (float)widen(src[x], dtype) / scale;
          dst[x] = oracle_f64_to_e4m3((double)y);
        }
        const int64_t sidx = (block * num_kv_heads + h) * block_size + offset;   /* [block][head][offset] */
        scl[sidx] = scale;
      }
    }
  }
  return skipped;
}

/* Decode over the fp8 pool: keys and values are e4m3 value * scale. */
int oracle_paged_attn_decode_f8(const uint16_t *q, int32_t dtype, const uint8_t *k_cache,
                                const uint8_t *v_cache, const float *k_scale, const float *v_scale,
                                int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                int32_t head_dim, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                double scale, double *out, int32_t num_threads) {
  problem_t P = {q, dtype, NULL, NULL, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.k8 = (const int8_t *)k_cache;
  P.v8 = (const int8_t *)v_cache;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  P.fp8 = 1;
  return decode_problem(&P, context_lens, num_seqs, num_threads);
}

static int decode_problem(problem_t *P, const int32_t *context_lens, int32_t num_seqs,
                          int32_t num_threads) {
  const int32_t max_blocks_per_seq = P->max_blocks_per_seq, block_size = P->block_size;
  int32_t *row0 = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
  int32_t *nrows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
  int32_t *pos0 = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
  int rc = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t n = context_lens[s];
    if (n < 1 || n > max_blocks_per_seq * block_size) rc = -4;
    row0[s] = s;
    nrows[s] = 1;
    pos0[s] = n - 1;
  }
  if (rc == 0) {
    P->num_groups = num_seqs;
    P->group_row0 = row0;
    P->group_nrows = nrows;
    P->group_pos0 = pos0;
    rc = run_problem(P, num_threads);
  }
  free(row0);
  free(nrows);
  free(pos0);
  return rc;
}

/* ---- chunked prefill [P1 Qwen3Model.forward with T > 1; P2 attend mask] ----- */

/*
 * Chunk c holds chunk_lens[c] new query tokens at absolute positions
 * chunk_starts[c] + i; their rows are packed in chunk order (chunk c starts at
 * row sum_{c' < c} chunk_lens[c']).  Row i of chunk c sees keys
 * 0 .. chunk_starts[c] + i (key position <= query position), read through
 * block-table row c.  context_lens[c] must equal chunk_starts[c] +
 * chunk_lens[c] (the chunk's own K/V are written before attending).
 * Returns 0, -1 for a block id out of range, -3 for a bad head split, -4 for
 * inconsistent chunk metadata.
 */
int oracle_paged_attn_prefill_window(const uint16_t *q, int32_t dtype, const uint16_t *k_cache,
                                     const uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_dim, const int32_t *chunk_starts,
                                     const int32_t *chunk_lens, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_chunks,
                                     int32_t num_q_heads, double scale, int32_t window, double *out,
                                     int32_t num_threads);

int oracle_paged_attn_prefill(const uint16_t *q, int32_t dtype,
                              const uint16_t *k_cache, const uint16_t *v_cache,
                              int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, const int32_t *chunk_starts,
                              const int32_t *chunk_lens, const int32_t *block_tables,
                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_chunks, int32_t num_q_heads, double scale,
                              double *out, int32_t num_threads) {
  return oracle_paged_attn_prefill_window(q, dtype, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                                          head_dim, chunk_starts, chunk_lens, block_tables, max_blocks_per_seq,
                                          context_lens, num_chunks, num_q_heads, scale, 0, out, num_threads);
}

/* Chunked prefill with a sliding window of W keys (W = 0: none) [P2 sections
 * 4 and 5.2]: row i of chunk c, at position p = chunk_starts[c] + i, sees keys
 * max(0, p - W + 1) .. p. */
static int prefill_problem(problem_t *P, const int32_t *chunk_starts, const int32_t *chunk_lens,
                           const int32_t *context_lens, int32_t num_chunks, int32_t num_threads);

int oracle_paged_attn_prefill_window(const uint16_t *q, int32_t dtype, const uint16_t *k_cache,
                                     const uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_dim, const int32_t *chunk_starts,
                                     const int32_t *chunk_lens, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_chunks,
                                     int32_t num_q_heads, double scale, int32_t window, double *out,
                                     int32_t num_threads) {
  if (window < 0) return -4;
  problem_t P = {q, dtype, k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.window = window;
  return prefill_problem(&P, chunk_starts, chunk_lens, context_lens, num_chunks, num_threads);
}

/* The same chunked prefill on the int8 pool [P2 section 5]: keys and values
 * are the dequantised fp32 numbers of KV8Cache.read. */
int oracle_paged_attn_prefill_q8(const uint16_t *q, int32_t dtype, const int8_t *k_cache, const int8_t *v_cache,
                                 const float *k_scale, const float *v_scale, int64_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                 const int32_t *chunk_starts, const int32_t *chunk_lens,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_chunks, int32_t num_q_heads,
                                 double scale, double *out, int32_t num_threads) {
  problem_t P = {q, dtype, NULL, NULL, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.k8 = k_cache;
  P.v8 = v_cache;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  return prefill_problem(&P, chunk_starts, chunk_lens, context_lens, num_chunks, num_threads);
}

/* The same chunked prefill on the fp8 (E4M3) pool [P2 sections 5.1, 5.4]:
 * keys and values are the e4m3 numbers times their scales, as in the fp8 decode. */
int oracle_paged_attn_prefill_f8(const uint16_t *q, int32_t dtype, const uint8_t *k_cache, const uint8_t *v_cache,
                                 const float *k_scale, const float *v_scale, int64_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                 const int32_t *chunk_starts, const int32_t *chunk_lens,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_chunks, int32_t num_q_heads,
                                 double scale, double *out, int32_t num_threads) {
  problem_t P = {q, dtype, NULL, NULL, num_blocks, block_size, num_kv_heads, head_dim,
                 block_tables, max_blocks_per_seq, num_q_heads, scale, out};
  P.k8 = (const int8_t *)k_cache;
  P.v8 = (const int8_t *)v_cache;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  P.fp8 = 1;
  return prefill_problem(&P, chunk_starts, chunk_lens, context_lens, num_chunks, num_threads);
}

static int prefill_problem(problem_t *P, const int32_t *chunk_starts, const int32_t *chunk_lens,
                           const int32_t *context_lens, int32_t num_chunks, int32_t num_threads) {
  const int32_t max_blocks_per_seq = P->max_blocks_per_seq, block_size = P->block_size;
  int32_t *row0 = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_chunks > 0 ? num_chunks : 1));
  int rc = 0;
  int32_t acc = 0;
  for (int32_t c = 0; c < num_chunks; ++c) {
    row0[c] = acc;
    acc += chunk_lens[c];
    if (chunk_lens[c] < 1 || chunk_starts[c] < 0 ||
        context_lens[c] != chunk_starts[c] + chunk_lens[c] ||
        context_lens[c] > max_blocks_per_seq * block_size)
      rc = -4;
  }
  if (rc == 0) {
    P->num_groups = num_chunks;
    P->group_row0 = row0;
    P->group_nrows = chunk_lens;
    P->group_pos0 = chunk_starts;
    rc = run_problem(P, num_threads);
  }
  free(row0);
  return rc;
}
