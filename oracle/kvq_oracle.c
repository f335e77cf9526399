/*
 * kvq_oracle.c -- plain CPU oracle for the FP8 paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark load this code.  It
 * shares no source, header, table or helper with the CUDA library; it is
 * written from the method's definition so that the two can be compared.
 *
 * Method sources (page titles, sections):
 *   "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV"
 *     section 10.4.1  M_KV = 2 * L * B * Hkv * S * dh * bytes
 *     section 10.4.2  write K_q = quant(K / sK); read K^ = sK * K_q;
 *                     P = softmax(Q K^T / sqrt(dh) + mask), O = P V^
 *     section 10.4.5  FP8 path: store cast_fp8(K / sK), compute with
 *                     cast_float(K_fp8) * sK
 *     section 10.4.3  per-token scales: one scale per token along dh, so a
 *                     new token is quantized on its own and appended
 *   "vLLM FP8 quantized KV cache guide" (per-tensor scales of shape [1],
 *     per-head k/v scales of shape [num_kv_heads]; fp8 = fp8_e4m3;
 *     cache storage is uint8 with FP8 bit semantics; fp8_per_token_head)
 *
 * FP8 bit layouts are not printed on the pages; the oracle takes the OCP
 * 8-bit floating point formats: E4M3 (bias 7, no infinities, NaN = S.1111.111,
 * largest finite 448) and E5M2 (bias 15, IEEE-style inf/NaN, largest finite
 * 57344).  Rounding is round-to-nearest-even; finite overflow and +-inf
 * saturate to +-max ("satfinite"); NaN encodes as 0x7F.
 *
 * Every floating-point step is written so that it can be checked by eye:
 * the encoder works on the exact integer significand of the fp32 input,
 * the decoder returns exact float64 values, attention is float64 throughout.
 * Compile with -O2 -fno-fast-math -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { KVQO_BF16 = 0, KVQO_E4M3 = 1, KVQO_E5M2 = 2 };
enum { KVQO_PER_TENSOR = 0, KVQO_PER_HEAD = 1, KVQO_PER_TOKEN_HEAD = 2 };

/* ------------------------------------------------------------------------ */
/* bf16 <-> f32 (bf16 is the top half of an IEEE binary32)                   */
/* ------------------------------------------------------------------------ */

float kvqo_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even from binary32 to bfloat16, written out on the bits:
 * keep the top 16 bits, look at the 16 dropped bits. NaN stays a quiet NaN
 * with its sign; infinities stay infinities. */
uint16_t kvqo_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t keep = u >> 16, drop = u & 0xFFFFu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

/* ------------------------------------------------------------------------ */
/* FP8 encode: exact integer rounding of the binary32 input                  */
/* ------------------------------------------------------------------------ */

/* Encodes binary32 x into the FP8 format `fmt` (E4M3 or E5M2).
 * Write the magnitude as v = S * 2^P with an integer significand S < 2^24.
 * Let L = floor(log2 v).  The target quantum at v is 2^(max(L, emin) - mbits)
 * (emin = 1 - bias is the exponent of the smallest normal; below it the
 * quantum stays that of the subnormal range).  q = v / quantum is rounded to
 * the nearest integer, ties to even; a rounding carry that reaches
 * 2^(mbits+1) moves to the next binade.  Results above the largest finite
 * value saturate.  Signed zero keeps its sign. */
uint8_t kvqo_encode(int fmt, float x) {
  const int mbits = (fmt == KVQO_E4M3) ? 3 : 2;
  const int bias = (fmt == KVQO_E4M3) ? 7 : 15;
  const uint8_t maxmag = (fmt == KVQO_E4M3) ? 0x7E : 0x7B;
  uint32_t u;
  memcpy(&u, &x, 4);
  const uint8_t s = (uint8_t)((u >> 24) & 0x80u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return 0x7F;                   /* NaN             */
  if (a == 0x7F800000u) return (uint8_t)(s | maxmag); /* +-inf saturates */
  if (a == 0) return s;                               /* +-0             */

  const uint32_t fe = a >> 23, frac = a & 0x7FFFFFu;
  uint64_t S;
  int P;
  if (fe != 0) {
    S = (uint64_t)(frac | 0x800000u);
    P = (int)fe - 150; /* (1.f) * 2^(fe-127) = S * 2^(fe-127-23) */
  } else {
    S = frac;
    P = -149; /* binary32 subnormal: frac * 2^-149 */
  }
  int bitlen = 0;
  for (uint64_t t = S; t; t >>= 1) bitlen++;
  const int L = P + bitlen - 1;
  const int emin = 1 - bias;
  int Eq = (L > emin) ? L : emin;
  const int shift = P - (Eq - mbits); /* q_exact = S * 2^shift */

  uint64_t q;
  if (shift >= 0) {
    q = S << shift;
  } else {
    const int r = -shift;
    if (r > 62) {
      q = 0; /* S < 2^24, so S * 2^-r < 1/2: rounds to zero */
    } else {
      const uint64_t whole = S >> r;
      const uint64_t rem = S & ((1ull << r) - 1ull);
      const uint64_t half = 1ull << (r - 1);
      q = whole;
      if (rem > half || (rem == half && (whole & 1ull))) q += 1ull;
    }
  }
  if (q >> (mbits + 1)) { /* carry: 2^(mbits+1) -> 2^mbits one binade up */
    q >>= 1;
    Eq += 1;
  }
  int efield, mfield;
  if (q >= (1ull << mbits)) {
    efield = Eq + bias;
    mfield = (int)(q - (1ull << mbits));
  } else {
    efield = 0;
    mfield = (int)q;
  }
  if (fmt == KVQO_E4M3) {
    if (efield > 15 || (efield == 15 && mfield == 7)) return (uint8_t)(s | maxmag);
  } else {
    if (efield > 30) return (uint8_t)(s | maxmag);
  }
  return (uint8_t)(s | (efield << mbits) | mfield);
}

/* ------------------------------------------------------------------------ */
/* FP8 decode: exact float64 value of a code                                 */
/* ------------------------------------------------------------------------ */

double kvqo_decode(int fmt, uint8_t c) {
  const int neg = c >> 7;
  double v;
  if (fmt == KVQO_E4M3) {
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    v = e ? ldexp(8.0 + m, e - 10) : ldexp((double)m, -9);
  } else {
    const int e = (c >> 2) & 31, m = c & 3;
    if (e == 31) {
      if (m) return NAN;
      return neg ? -INFINITY : INFINITY;
    }
    v = e ? ldexp(4.0 + m, e - 17) : ldexp((double)m, -16);
  }
  return neg ? -v : v;
}

/* Array forms, used by the exhaustive codec pins. */
void kvqo_encode_f32_array(int fmt, const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvqo_encode(fmt, x[i]);
}

void kvqo_decode_array(int fmt, const uint8_t* c, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvqo_decode(fmt, c[i]);
}

/* Quantize one bf16 value with scale s: the two roundings of the FP8 write,
 * first the IEEE binary32 quotient x / s, then RNE-satfinite to FP8. */
static uint8_t quantize_bf16(int fmt, uint16_t xb, float s) {
  const float x = kvqo_bf16_to_f32(xb);
  const float quotient = x / s;
  return kvqo_encode(fmt, quotient);
}

void kvqo_quantize_bf16_array(int fmt, const uint16_t* x, float s, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = quantize_bf16(fmt, x[i], s);
}

/* ------------------------------------------------------------------------ */
/* Write: quantize and scatter into the paged cache                          */
/* ------------------------------------------------------------------------ */

/* Cache layout [num_blocks][num_kv_heads][block_size][head_dim]; elements are
 * uint8 FP8 codes, or bf16 bit patterns when fmt == KVQO_BF16 (a layer that
 * is skipped from quantization keeps the model dtype and is copied as is).
 * Inputs k, v are bf16 [num_tokens][num_kv_heads][head_dim] with a token
 * stride of `token_stride` elements.  Token t goes to slot slot_mapping[t]:
 * block slot / block_size, offset slot % block_size.  A negative slot is a
 * padding token and is skipped; a slot past the cache is skipped and counted.
 * Returns the number of tokens skipped for an out-of-range slot. */
int64_t kvqo_write(const uint16_t* k, const uint16_t* v, int64_t token_stride,
                   const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                   int head_dim, void* k_cache, void* v_cache, int64_t num_blocks,
                   int block_size, const float* k_scale, const float* v_scale,
                   int granularity, int fmt, int nthreads) {
  int64_t bad = 0;
  const int64_t capacity = num_blocks * (int64_t)block_size;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(nthreads)
#endif
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      bad += 1;
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t src = t * token_stride + (int64_t)h * head_dim;
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      if (fmt == KVQO_BF16) {
        memcpy((uint16_t*)k_cache + dst, k + src, (size_t)head_dim * 2);
        memcpy((uint16_t*)v_cache + dst, v + src, (size_t)head_dim * 2);
        continue;
      }
      const float sk = k_scale[granularity == KVQO_PER_HEAD ? h : 0];
      const float sv = v_scale[granularity == KVQO_PER_HEAD ? h : 0];
      for (int d = 0; d < head_dim; ++d) {
        ((uint8_t*)k_cache)[dst + d] = quantize_bf16(fmt, k[src + d], sk);
        ((uint8_t*)v_cache)[dst + d] = quantize_bf16(fmt, v[src + d], sv);
      }
    }
  }
  return bad;
}

/* Per-(token, KV head) scale of one row of head_dim bf16 values: the largest
 * magnitude among its finite values over the format's largest finite value
 * (binary32 division), or 1 when that is 0 -- the row's largest value then
 * lands on the format's largest code. */
static float token_head_scale(const uint16_t* x, int head_dim, int fmt) {
  float amax = 0.0f;
  for (int d = 0; d < head_dim; ++d) {
    const float a = fabsf(kvqo_bf16_to_f32(x[d]));
    if (isfinite(a) && a > amax) amax = a;
  }
  const float fmt_max = (fmt == KVQO_E4M3) ? 448.0f : 57344.0f;
  const float s = amax / fmt_max;
  return s > 0.0f ? s : 1.0f;
}

/* Write with per-(token, KV head) scales ("10.4 KV Cache quantization",
 * section 10.4.3, per-token granularity; vLLM's fp8_per_token_head): every
 * row gets its own scale from its own values, stored beside the page in
 * k_scale_cache / v_scale_cache [num_blocks][num_kv_heads][block_size]
 * (binary32), and its codes are cast_fp8(x / s) as for the other
 * granularities.  FP8 formats only.  Returns the bad-slot count. */
int64_t kvqo_write_token_head(const uint16_t* k, const uint16_t* v, int64_t token_stride,
                              const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                              int head_dim, uint8_t* k_cache, uint8_t* v_cache,
                              int64_t num_blocks, int block_size, float* k_scale_cache,
                              float* v_scale_cache, int fmt, int nthreads) {
  int64_t bad = 0;
  const int64_t capacity = num_blocks * (int64_t)block_size;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(nthreads)
#endif
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      bad += 1;
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t src = t * token_stride + (int64_t)h * head_dim;
      const int64_t row = (blk * num_kv_heads + h) * block_size + off;
      const float sk = token_head_scale(k + src, head_dim, fmt);
      const float sv = token_head_scale(v + src, head_dim, fmt);
      k_scale_cache[row] = sk;
      v_scale_cache[row] = sv;
      for (int d = 0; d < head_dim; ++d) {
        k_cache[row * head_dim + d] = quantize_bf16(fmt, k[src + d], sk);
        v_cache[row * head_dim + d] = quantize_bf16(fmt, v[src + d], sv);
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over the dequantized cache, float64                      */
/* ------------------------------------------------------------------------ */

/* Dequantized cache element: cast_float(code) * s (exact in float64), or the
 * bf16 value itself in bf16 mode. */
static double cache_value(const void* cache, int64_t idx, int fmt, double s) {
  if (fmt == KVQO_BF16) return (double)kvqo_bf16_to_f32(((const uint16_t*)cache)[idx]);
  return kvqo_decode(fmt, ((const uint8_t*)cache)[idx]) * s;
}

/* Scale of KV head g for the token in block blk at offset off: one per
 * tensor, one per KV head, or -- per (token, KV head) -- the one stored
 * beside the page, [num_blocks][num_kv_heads][block_size]. */
static double scale_at(const float* s, int granularity, int num_kv_heads, int block_size,
                       int64_t blk, int g, int off) {
  if (granularity == KVQO_PER_TOKEN_HEAD)
    return (double)s[(blk * num_kv_heads + g) * block_size + off];
  return (double)s[granularity == KVQO_PER_HEAD ? g : 0];
}

/* Query element d of head h as the attention uses it: the bf16 value, or --
 * with a q scale (the FP8-domain mode) -- the query quantized to the cache's
 * FP8 format with the head's scale and restored, dec(enc(fp32(q) / sQ)) * sQ,
 * the division a binary32 one as for the cache write ("vLLM FP8 quantized KV
 * cache guide", FlashAttention 3 note: the query is quantized to FP8 like K
 * and V). */
static double query_value(uint16_t qb, int fmt, const float* q_scale, int q_per_head, int h) {
  const float x = kvqo_bf16_to_f32(qb);
  if (!q_scale) return (double)x;
  const float sq = q_scale[q_per_head ? h : 0];
  const float quotient = x / sq;
  return kvqo_decode(fmt, kvqo_encode(fmt, quotient)) * (double)sq;
}

/* One query row qrow of head h of sequence b that attends to the tokens
 * [lo, L) of the sequence, lo = L - window when a positive window is shorter
 * than L (the window keeps the newest tokens, the query's own included).
 * x_t = (sum_d q_d * K^_{t,d}) / sqrt(dh); p = softmax(x); O = sum_t p_t V^_t.
 * Query head h reads KV head h / (Hq / Hkv).  Returns 0, or -1 when the
 * block table or length is out of range. */
static int attend_row(const uint16_t* qrow, int L, const void* kc, const void* vc,
                      const int32_t* block_tables, int max_blocks_per_seq, int num_q_heads,
                      int num_kv_heads, int head_dim, int64_t num_blocks, int block_size,
                      const float* k_scale, const float* v_scale, int granularity, int fmt,
                      const float* q_scale, int q_per_head, int window, int b, int h,
                      double* out, double* scores) {
  const int group = num_q_heads / num_kv_heads;
  const int g = h / group;
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (L <= 0) return L < 0 ? -1 : 0;
  if (L > max_blocks_per_seq * block_size) return -1;
  const int lo = (window > 0 && L > window) ? L - window : 0;
  const double inv_sqrt_dh = 1.0 / sqrt((double)head_dim);

  double xmax = -INFINITY;
  for (int t = lo; t < L; ++t) {
    const int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
    if (blk < 0 || blk >= num_blocks) return -1;
    const int64_t base = (((int64_t)blk * num_kv_heads + g) * block_size + t % block_size) * head_dim;
    const double sk = (fmt == KVQO_BF16)
                          ? 1.0
                          : scale_at(k_scale, granularity, num_kv_heads, block_size, blk, g,
                                     t % block_size);
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d)
      dot += query_value(qrow[d], fmt, q_scale, q_per_head, h) * cache_value(kc, base + d, fmt, sk);
    const double x = dot * inv_sqrt_dh;
    scores[t - lo] = x;
    if (x > xmax) xmax = x;
  }
  double denom = 0.0;
  for (int t = lo; t < L; ++t) {
    const double p = exp(scores[t - lo] - xmax);
    scores[t - lo] = p;
    denom += p;
  }
  for (int t = lo; t < L; ++t) {
    const int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
    const int64_t base = (((int64_t)blk * num_kv_heads + g) * block_size + t % block_size) * head_dim;
    const double sv = (fmt == KVQO_BF16)
                          ? 1.0
                          : scale_at(v_scale, granularity, num_kv_heads, block_size, blk, g,
                                     t % block_size);
    const double p = scores[t - lo];
    for (int d = 0; d < head_dim; ++d) out[d] += p * cache_value(vc, base + d, fmt, sv);
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= denom;
  return 0;
}

/* All pairs (pairs == NULL: out is [num_seqs][num_q_heads][head_dim]) or a
 * list of (b, h) pairs (pairs is int32 [npairs][2]; out is [npairs][head_dim]).
 * Returns the number of pairs whose inputs were out of range. */
int64_t kvqo_decode_attn(const uint16_t* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int64_t num_blocks, int block_size,
                         const float* k_scale, const float* v_scale, int granularity, int fmt,
                         const float* q_scale, int q_per_head,
                         int window, const int32_t* pairs, int64_t npairs, double* out,
                         int nthreads) {
  const int64_t n = pairs ? npairs : (int64_t)num_seqs * num_q_heads;
  int max_len = 0;
  for (int b = 0; b < num_seqs; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  int64_t bad = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(+ : bad)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n; ++i) {
      int b, h;
      if (pairs) {
        b = pairs[2 * i];
        h = pairs[2 * i + 1];
      } else {
        b = (int)(i / num_q_heads);
        h = (int)(i % num_q_heads);
      }
      /* the decode query is the sequence's last token: it attends to [lo, L) */
      if (attend_row(q + ((int64_t)b * num_q_heads + h) * head_dim, seq_lens[b], k_cache,
                     v_cache, block_tables, max_blocks_per_seq, num_q_heads, num_kv_heads,
                     head_dim, num_blocks, block_size, k_scale, v_scale, granularity, fmt,
                     q_scale, q_per_head, window, b, h, out + i * head_dim, scores))
        bad += 1;
    }
    free(scores);
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Prefill / prefix-hit attention: several new query tokens per sequence      */
/* ------------------------------------------------------------------------ */

/* "10.4 KV Cache quantization", section 10.4.2: the prefill and prefix-hit
 * paths read the same quantized cache as the decode.  Sequence b holds
 * L_b = seq_lens[b] tokens in the cache, the last n_b = cu_q[b+1] - cu_q[b]
 * of them new; query row cu_q[b] + j (j < n_b) is the token at position
 * pos = L_b - n_b + j and attends causally to the tokens [lo, pos], lo as
 * for the decode with L = pos + 1 (a sliding window keeps the newest
 * `window` of them).  With n_b = 1 this is the decode.  q and out are
 * [total_q][Hq][dh].  pairs (int32 [npairs][2] of (query row, head)) picks
 * rows; NULL takes all.  Returns the number of rows with out-of-range
 * inputs (n_b > L_b, a bad length or block id). */
int64_t kvqo_prefill_attn(const uint16_t* q, const int32_t* cu_q, const void* k_cache,
                          const void* v_cache, const int32_t* block_tables,
                          int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int64_t num_blocks,
                          int block_size, const float* k_scale, const float* v_scale,
                          int granularity, int fmt, const float* q_scale, int q_per_head,
                          int window, const int32_t* pairs, int64_t npairs, double* out,
                          int nthreads) {
  const int64_t total_q = cu_q[num_seqs];
  const int64_t n = pairs ? npairs : total_q * num_q_heads;
  int max_len = 0;
  for (int b = 0; b < num_seqs; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  int64_t bad = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(+ : bad)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
    for (int64_t i = 0; i < n; ++i) {
      int64_t row;
      int h;
      if (pairs) {
        row = pairs[2 * i];
        h = pairs[2 * i + 1];
      } else {
        row = i / num_q_heads;
        h = (int)(i % num_q_heads);
      }
      int b = 0; /* the sequence holding query row `row` */
      while (b + 1 < num_seqs && cu_q[b + 1] <= row) ++b;
      const int64_t nb_q = cu_q[b + 1] - cu_q[b];
      const int64_t pos = (int64_t)seq_lens[b] - nb_q + (row - cu_q[b]);
      double* o = out + i * head_dim;
      if (nb_q > seq_lens[b] || pos < 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        bad += 1;
        continue;
      }
      if (attend_row(q + (row * num_q_heads + h) * head_dim, (int)(pos + 1), k_cache, v_cache,
                     block_tables, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                     num_blocks, block_size, k_scale, v_scale, granularity, fmt, q_scale,
                     q_per_head, window, b, h, o, scores))
        bad += 1;
    }
    free(scores);
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Unfused path: materialise a bf16 cache from the FP8 cache                 */
/* ------------------------------------------------------------------------ */

/* The "independent dequant kernel" of the unfused path: every code c of KV
 * head h becomes bf16(fp32(cast_float(c) * s_h)), s_h the tensor's, the
 * head's or the (token, head)'s scale.  The product of an FP8
 * value (at most 4 significant bits) and a binary32 scale is exact in
 * float64, so the float cast below is the single binary32 rounding of the
 * product, followed by RNE to bf16. */
void kvqo_dequant(const uint8_t* src, uint16_t* dst, int64_t num_blocks, int num_kv_heads,
                  int block_size, int head_dim, const float* scale, int granularity, int fmt) {
  const int64_t per_head = (int64_t)block_size * head_dim;
  for (int64_t blk = 0; blk < num_blocks; ++blk) {
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t base = (blk * num_kv_heads + h) * per_head;
      for (int64_t i = 0; i < per_head; ++i) {
        const double s = scale_at(scale, granularity, num_kv_heads, block_size, blk, h,
                                  (int)(i / head_dim));
        const float prod = (float)(kvqo_decode(fmt, src[base + i]) * s);
        dst[base + i] = kvqo_f32_to_bf16(prod);
      }
    }
  }
}

int kvqo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
