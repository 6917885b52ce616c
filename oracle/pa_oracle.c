/*
 * Plain CPU oracle for paged decode attention and its companion cache ops.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no code, header or constant with the CUDA
 * library.
 *
 * Every routine is the plain definition written out, in float64, with no
 * blocking, fusion or reordering beyond what that definition states:
 *
 *  - Addressing. Token position p of a sequence lives in logical block
 *    p / BS at offset p % BS; the block table maps the logical block to a
 *    physical block ("How Paged Attention and Continuous Batching Actually
 *    Work", §Paged attention: virtual memory for the KV cache -- divide to
 *    find the logical block, look up the physical block, multiply out, add
 *    the offset; the printed formula itself is lost, this is its prose).
 *    Cache layout is [num_blocks][num_kv_heads][BS][head_dim].
 *  - Decode attention. score_i = (q . k_i) * scale, scale = 1/sqrt(d)
 *    ("Paged Attention as a Memory Manager", §How the Kernel Executes Paged
 *    Attention); weights = softmax over all past tokens i < L (decode is the
 *    last position, so the causal mask admits every cached token;
 *    "PagedAttention and continuous batching", §Attention kernel
 *    modification); output = sum_i w_i v_i. The running (online) softmax of
 *    the pages is mathematically this same function, so the oracle uses the
 *    textbook two-pass form over K/V reassembled contiguously.
 *  - GQA: query head h reads KV head h / (Hq / Hkv).
 *  - KV write: the new token's K/V row is copied to the slot named by the
 *    slot mapping ("How Paged Attention ...", §One step, end to end).
 *  - Copy-on-write: the whole content of the source block is copied to the
 *    fresh block ("Paged Attention as a Memory Manager", §Prefix Caching and
 *    Copy-on-Write).
 *
 * bf16 values are widened to double exactly (the bf16 bit pattern is the
 * top half of an IEEE float).
 *
 * 8-bit KV cache ("PagedAttention" glossary page, §What paging costs: paging
 * combines with 8-bit KV quantisation, which halves the bytes per block).
 * The pages fix no format; this oracle follows the reading the library
 * implements: FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals, no infinities, S.1111.111 is NaN, largest finite 448)
 * with one dequantisation scale per KV head for K and one for V:
 *  - write: code = E4M3(x / scale[h]), the division in float32 and the
 *    conversion round-to-nearest-even, saturating finite values (and
 *    infinities) to +-448, NaN to 0x7F;
 *  - read: value = decode(code) * scale[h], in double;
 *  - layout: K as the bf16 cache, [block][head][offset][d]; V transposed
 *    inside each (block, head) tile in sub-tiles of W = min(16, BS) keys,
 *    [block][head][offset / W][d][offset % W] (one [d][BS] sub-tile for
 *    BS <= 16, two [d][16] sub-tiles at BS = 32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_OUT_OF_RANGE 2
#define ORACLE_NO_MEMORY 3

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 code -> value (exact in double). */
static double e4m3_to_double(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* float32 -> E4M3, round to nearest even, saturating to the largest finite
 * value; NaN -> 0x7F. Works on the exact value of the float. */
static uint8_t e4m3_from_float(float xf) {
  const double x = (double)xf;
  if (x != x) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  /* candidates on the grid of this binade: the spacing is 2^(e-3) for a
   * normal value with exponent e, 2^-9 below 2^-6 */
  int e;
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  const int ue = e - 1; /* unbiased exponent of a */
  const double spacing = ue < -6 ? ldexp(1.0, -9) : ldexp(1.0, ue - 3);
  const double k = a / spacing; /* exact: a power-of-two division */
  double r = floor(k);
  const double frac = k - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  const double v = r * spacing; /* the rounded magnitude */
  if (v >= 448.0 + 32.0) return sign | 0x7E; /* would be 480: saturate */
  /* encode v */
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9)); /* subnormal (or 0) */
  int ve;
  (void)frexp(v, &ve);
  const int vue = ve - 1;
  const int man = (int)(v / ldexp(1.0, vue - 3)) - 8;
  return sign | (uint8_t)(((vue + 7) << 3) | man);
}

uint8_t oracle_e4m3_from_float(float x) { return e4m3_from_float(x); }
double oracle_e4m3_to_double(uint8_t c) { return e4m3_to_double(c); }

/* Address of (physical block, kv head, offset in block) in a cache array. */
static size_t cache_row(int64_t blk, int32_t kv_head, int32_t off, int32_t num_kv_heads,
                        int32_t block_size, int32_t head_dim) {
  return (((size_t)blk * (size_t)num_kv_heads + (size_t)kv_head) * (size_t)block_size +
          (size_t)off) * (size_t)head_dim;
}

/*
 * Decode attention for one (sequence b, query head h).
 * out_row: head_dim doubles. lse_out (nullable): log sum_i exp(score_i).
 * Returns ORACLE_OK or an error code.
 */
/* Byte offset of V element (off, c) inside its (block, head) tile of the
 * E4M3 cache: sub-tile off / W, row c, column off % W, W = min(16, BS). */
static size_t vt_offset(int32_t off, int32_t c, int32_t block_size, int32_t head_dim) {
  const int32_t w = block_size < 16 ? block_size : 16;
  return (size_t)(off / w) * (size_t)w * head_dim + (size_t)c * w + (size_t)(off % w);
}

/* Element c of row (blk, head, off) of K and of V, as double, for a bf16
 * cache (fp8 == 0) or an E4M3 cache with per-head scales (fp8 == 1). */
static void kv_element(const void* k_cache, const void* v_cache, int fp8, const float* k_scale,
                       const float* v_scale, int64_t blk, int32_t g, int32_t off, int32_t c,
                       int32_t num_kv_heads, int32_t block_size, int32_t head_dim, double* k,
                       double* v) {
  const size_t row = cache_row(blk, g, off, num_kv_heads, block_size, head_dim);
  if (!fp8) {
    *k = bf16_bits_to_double(((const uint16_t*)k_cache)[row + c]);
    *v = bf16_bits_to_double(((const uint16_t*)v_cache)[row + c]);
    return;
  }
  /* V is transposed inside its (block, head) tile (sub-tiles of 16 keys) */
  const size_t tile = ((size_t)blk * num_kv_heads + g) * (size_t)block_size * head_dim;
  *k = e4m3_to_double(((const uint8_t*)k_cache)[row + c]) * (double)k_scale[g];
  *v = e4m3_to_double(((const uint8_t*)v_cache)[tile + vt_offset(off, c, block_size, head_dim)]) *
       (double)v_scale[g];
}

/* qrow: this query's head_dim bf16 values; L: the number of cached tokens it
 * attends to (the first L of sequence b). */
static int decode_one(const uint16_t* qrow, int32_t L, const void* k_cache, const void* v_cache,
                      int fp8, const float* k_scale, const float* v_scale,
                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                      int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t num_blocks, double scale,
                      int32_t b, int32_t h, double* out_row, double* lse_out) {
  const int32_t group = num_q_heads / num_kv_heads;
  const int32_t g = h / group;
  if (L < 1) return ORACLE_BAD_ARG;
  if ((L + block_size - 1) / block_size > max_blocks_per_seq) return ORACLE_OUT_OF_RANGE;

  /* 1. Reassemble this sequence's K and V contiguously, token by token. */
  double* K = (double*)malloc(sizeof(double) * (size_t)L * (size_t)head_dim);
  double* V = (double*)malloc(sizeof(double) * (size_t)L * (size_t)head_dim);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  if (!K || !V || !s) {
    free(K); free(V); free(s);
    return ORACLE_NO_MEMORY;
  }
  int rc = ORACLE_OK;
  for (int32_t t = 0; t < L && rc == ORACLE_OK; ++t) {
    const int32_t logical = t / block_size;
    const int32_t off = t % block_size;
    const int64_t blk = block_tables[(size_t)b * (size_t)max_blocks_per_seq + (size_t)logical];
    if (blk < 0 || blk >= num_blocks) {
      rc = ORACLE_OUT_OF_RANGE;
      break;
    }
    for (int32_t c = 0; c < head_dim; ++c)
      kv_element(k_cache, v_cache, fp8, k_scale, v_scale, blk, g, off, c, num_kv_heads,
                 block_size, head_dim, &K[(size_t)t * head_dim + c], &V[(size_t)t * head_dim + c]);
  }
  if (rc == ORACLE_OK) {
    /* 2. Scores. */
    for (int32_t t = 0; t < L; ++t) {
      double dot = 0.0;
      for (int32_t c = 0; c < head_dim; ++c)
        dot += bf16_bits_to_double(qrow[c]) * K[(size_t)t * head_dim + c];
      s[t] = dot * scale;
    }
    /* 3. Softmax, two passes: max, then normalised exponentials. */
    double m = s[0];
    for (int32_t t = 1; t < L; ++t)
      if (s[t] > m) m = s[t];
    double denom = 0.0;
    for (int32_t t = 0; t < L; ++t) {
      s[t] = exp(s[t] - m);
      denom += s[t];
    }
    /* 4. Weighted sum of V. */
    for (int32_t c = 0; c < head_dim; ++c) out_row[c] = 0.0;
    for (int32_t t = 0; t < L; ++t) {
      const double w = s[t] / denom;
      for (int32_t c = 0; c < head_dim; ++c) out_row[c] += w * V[(size_t)t * head_dim + c];
    }
    if (lse_out) *lse_out = m + log(denom);
  }
  free(K);
  free(V);
  free(s);
  return rc;
}

/*
 * Paged decode attention over a list of (b, h) units.
 *   q            bf16 bits [num_seqs][num_q_heads][head_dim]
 *   k/v_cache    bf16 bits [num_blocks][num_kv_heads][block_size][head_dim]
 *   block_tables int32 [num_seqs][max_blocks_per_seq]
 *   context_lens int32 [num_seqs]
 *   units        int32 [n_units][2] = (b, h); NULL = every (b, h) in order
 *   out          double [n_units][head_dim] (or [num_seqs][num_q_heads][head_dim])
 *   lse          double [n_units] (nullable)
 * OpenMP parallelises over units; each unit is computed independently.
 */
static int paged_decode(const uint16_t* q, const void* k_cache, const void* v_cache, int fp8,
                        const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, double scale, const int32_t* units, int64_t n_units,
                        double* out, double* lse) {
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
      num_q_heads % num_kv_heads != 0)
    return ORACLE_BAD_ARG;
  const int64_t total = units ? n_units : (int64_t)num_seqs * num_q_heads;
  int rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t u = 0; u < total; ++u) {
    int32_t b, h;
    if (units) {
      b = units[2 * u];
      h = units[2 * u + 1];
    } else {
      b = (int32_t)(u / num_q_heads);
      h = (int32_t)(u % num_q_heads);
    }
    int r = ORACLE_BAD_ARG;
    if (b >= 0 && b < num_seqs && h >= 0 && h < num_q_heads)
      r = decode_one(q + ((size_t)b * num_q_heads + h) * head_dim, context_lens[b], k_cache,
                     v_cache, fp8, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, b, h,
                     out + (size_t)u * head_dim, lse ? lse + u : NULL);
    if (r != ORACLE_OK) {
#pragma omp critical
      rc = r;
    }
  }
  return rc;
}

int oracle_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, double scale, const int32_t* units, int64_t n_units,
                        double* out, double* lse) {
  return paged_decode(q, k_cache, v_cache, 0, NULL, NULL, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, units, n_units, out, lse);
}

/*
 * Decode of query_len new tokens per sequence (the last query_len of its
 * context_lens[b] tokens), causal among themselves: query token i of sequence
 * b attends to the first context_lens[b] - query_len + i + 1 cached tokens.
 *   q, out  [num_seqs][query_len][num_q_heads][head_dim] (bf16 bits / double)
 * Every (b, i, h) is computed; context_lens[b] < query_len is an error.
 */
static int paged_decode_multi(const uint16_t* q, const void* k_cache, const void* v_cache, int fp8,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs, int32_t query_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks, double scale, double* out) {
  if (num_seqs < 0 || query_len < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 ||
      block_size < 1 || num_q_heads % num_kv_heads != 0)
    return ORACLE_BAD_ARG;
  const int64_t total = (int64_t)num_seqs * query_len * num_q_heads;
  int rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t u = 0; u < total; ++u) {
    const int32_t h = (int32_t)(u % num_q_heads);
    const int32_t i = (int32_t)((u / num_q_heads) % query_len);
    const int32_t b = (int32_t)(u / ((int64_t)num_q_heads * query_len));
    const int32_t L = context_lens[b] - query_len + i + 1;
    int r = ORACLE_BAD_ARG;
    if (context_lens[b] >= query_len)
      r = decode_one(q + (size_t)u * head_dim, L, k_cache, v_cache, fp8, k_scale, v_scale,
                     block_tables, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, b, h, out + (size_t)u * head_dim, NULL);
    if (r != ORACLE_OK) {
#pragma omp critical
      rc = r;
    }
  }
  return rc;
}

int oracle_paged_decode_multi(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs, int32_t query_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks, double scale, double* out) {
  return paged_decode_multi(q, k_cache, v_cache, 0, NULL, NULL, block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, query_len, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, out);
}

/* The same over an E4M3 cache (layouts and scales as oracle_paged_decode_fp8 below). */
int oracle_paged_decode_multi_fp8(const uint16_t* q, const uint8_t* k_cache,
                                  const uint8_t* v_cache, const float* k_scale,
                                  const float* v_scale, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t query_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks, double scale, double* out) {
  if (!k_scale || !v_scale) return ORACLE_BAD_ARG;
  return paged_decode_multi(q, k_cache, v_cache, 1, k_scale, v_scale, block_tables,
                            max_blocks_per_seq, context_lens, num_seqs, query_len, num_q_heads,
                            num_kv_heads, head_dim, block_size, num_blocks, scale, out);
}

/* The same decode over an E4M3 cache (k/v_cache uint8, layouts above) with
 * per-KV-head scales k_scale, v_scale (float [num_kv_heads]). */
int oracle_paged_decode_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, double scale, const int32_t* units,
                            int64_t n_units, double* out, double* lse) {
  if (!k_scale || !v_scale) return ORACLE_BAD_ARG;
  return paged_decode(q, k_cache, v_cache, 1, k_scale, v_scale, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, units, n_units, out, lse);
}

/*
 * KV write through the slot mapping: token t's row for every KV head goes
 * to (slot / BS, head, slot % BS). A negative slot means "no write".
 *   k/v_new bf16 bits [num_tokens][num_kv_heads][head_dim]
 */
int oracle_reshape_and_cache(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                             uint16_t* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) return ORACLE_OUT_OF_RANGE;
    const int64_t blk = slot / block_size;
    const int32_t off = (int32_t)(slot % block_size);
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
      const size_t dst = cache_row(blk, h, off, num_kv_heads, block_size, head_dim);
      memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)head_dim);
      memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)head_dim);
    }
  }
  return ORACLE_OK;
}

/*
 * KV write into an E4M3 cache: token t's row of KV head h is quantised with
 * that head's scale (code = E4M3(float32(x) / scale[h])) and stored at
 * (slot / BS, h, slot % BS) -- K as a row, V as a column of its transposed
 * (block, head) tile. A negative slot means "no write".
 */
int oracle_reshape_and_cache_fp8(const uint16_t* k_new, const uint16_t* v_new, uint8_t* k_cache,
                                 uint8_t* v_cache, const int64_t* slot_mapping,
                                 const float* k_scale, const float* v_scale, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_blocks) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) return ORACLE_OUT_OF_RANGE;
    const int64_t blk = slot / block_size;
    const int32_t off = (int32_t)(slot % block_size);
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
      const size_t row = cache_row(blk, h, off, num_kv_heads, block_size, head_dim);
      const size_t tile = ((size_t)blk * num_kv_heads + h) * (size_t)block_size * head_dim;
      for (int32_t c = 0; c < head_dim; ++c) {
        const float kx = (float)bf16_bits_to_double(k_new[src + c]) / k_scale[h];
        const float vx = (float)bf16_bits_to_double(v_new[src + c]) / v_scale[h];
        k_cache[row + c] = e4m3_from_float(kx);
        v_cache[tile + vt_offset(off, c, block_size, head_dim)] = e4m3_from_float(vx);
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Copy-on-write block copy: for each (src, dst) pair, the whole physical
 * block (all KV heads, all slots) of both caches is copied src -> dst.
 *   pairs int32 [num_pairs][2]
 */
int oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int32_t* pairs,
                       int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, int32_t num_blocks) {
  const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
  for (int32_t i = 0; i < num_pairs; ++i) {
    const int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORACLE_OUT_OF_RANGE;
    memmove(k_cache + (size_t)dst * block_elems, k_cache + (size_t)src * block_elems,
            sizeof(uint16_t) * block_elems);
    memmove(v_cache + (size_t)dst * block_elems, v_cache + (size_t)src * block_elems,
            sizeof(uint16_t) * block_elems);
  }
  return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the OpenMP loops use from now on (n >= 1); for timing the oracle
 * on a given number of host cores. The results do not depend on it: every
 * unit is computed independently by one thread. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
