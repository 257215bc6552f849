/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * What it restates (sources are the pages this project is built from):
 *
 *  - "vLLM engine anatomy" (oripoin.cn), section "PagedAttention: paging the
 *    KV cache", Figure 2: the KV cache is cut into fixed physical blocks of 16
 *    tokens; each sequence's block table maps logical block j/16 to a physical
 *    block, and token j sits at offset j%16 of that block.
 *  - same page, same section: shared blocks and block-granular copy-on-write.
 *  - same page, section "Prefill, decode and the three latency metrics": each
 *    processed token's key and value are written into the KV cache; decode
 *    attends over every earlier token.
 *  - same page, section "How much memory does the KV cache need", Table 1:
 *    per-token KV bytes = 2 x element bytes x layers x KV heads x head dim,
 *    and GQA (fewer KV heads than query heads).
 *  - same page, section "Boundaries: FlashAttention ...": FlashAttention
 *    computes exact softmax attention without materialising the score
 *    matrix, so the oracle is the plain definition of softmax attention.
 *  - "vLLM V0 vs V1" (llm.rainlin.net), section 3.1: per step the model runner
 *    builds attention metadata from each request's query length, context
 *    length and block table; V0's scheduler output carries blocks_to_copy.
 *  - "vLLM: a general inference engine" (niuwancheng.cn), section "KV cache
 *    management and prefix caching", the hybrid KV cache manager paragraph:
 *    sliding-window attention layers, whose blocks outside the window can be
 *    released early.  A window of W keys lets the query at position p see
 *    keys max(0, p - W + 1) .. p: its own key and the W - 1 before it.
 *  - "vLLM: a general inference engine" (niuwancheng.cn), KV cache table:
 *    --kv-cache-dtype fp8 stores KV in 1-byte FP8.  The E4M3 "FN" format
 *    (bias 7, no infinities, S.1111.111 = NaN, max 448) is taken from the
 *    OCP 8-bit floating point specification.
 *  - same table: lower-bit KV formats, nvfp4 and int4_per_token_head, whose
 *    accuracy is left to the user to evaluate.  NVFP4 is NVIDIA's published
 *    4-bit format: FP4 E2M1 elements (the OCP Microscaling specification's
 *    E2M1: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; values 0,
 *    0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN), one E4M3 scale per 16
 *    consecutive elements and one fp32 scale per tensor.  int4_per_token_head
 *    is read here as signed 4-bit integers with one fp32 scale per (token,
 *    KV head), chosen at write time as max |x| / 7.
 *
 *  Page layout of the 4-bit formats (one page = one (block, KV head); block
 *  size bs, head dim D): bs * D / 2 bytes of codes, token by token, element
 *  2i in the low nibble of byte i of its token; then the scales: bs fp32
 *  (INT4, one per token) or bs * D / 16 E4M3 bytes (NVFP4, token by token,
 *  one per 16 elements).  Value: INT4 scale * code (two's complement);
 *  NVFP4 tensor_scale * e4m3(block scale) * e2m1(code).
 *
 * Everything is computed in double from the stored bytes; no blocking,
 * fusion or reordering beyond the definitions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element type codes (same numbering as the product header, written out
 * independently here) */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3, ORC_INT4 = 4,
       ORC_NVFP4 = 5 };

static int is_4bit(int dt) { return dt == ORC_INT4 || dt == ORC_NVFP4; }

/* bytes of one (block, KV head) page of a 4-bit cache */
static int64_t page_bytes_4bit(int dt, int bs, int D) {
  const int64_t codes = (int64_t)bs * (D / 2);
  return dt == ORC_INT4 ? codes + 4 * (int64_t)bs : codes + (int64_t)bs * (D / 16);
}

enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 2 };

static int elem_bytes(int dt) {
  switch (dt) {
    case ORC_F32: return 4;
    case ORC_F16: return 2;
    case ORC_BF16: return 2;
    case ORC_E4M3: return 1;
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Exact decoding of the stored formats to double (IEEE 754 binary16,      */
/* bfloat16 = the top half of binary32, OCP FP8 E4M3FN).                   */
/* ---------------------------------------------------------------------- */

double orc_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m/1024 * 2^-14 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

double orc_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133); /* subnormal: m/128 * 2^-126 */
  } else if (e == 255) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  }
  return sign ? -v : v;
}

double orc_e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int m = c & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN; /* the only NaN pattern; no infinities */
  if (e == 0) {
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return sign ? -v : v;
}

/* E2M1 (OCP Microscaling): sign bit 3, exponent bits 2-1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (m * 0.5). */
double orc_e2m1_to_double(uint8_t c) {
  const int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

static double load_elem(const void* base, int64_t i, int dt) {
  switch (dt) {
    case ORC_F32: {
      float f;
      memcpy(&f, (const char*)base + 4 * i, 4);
      return (double)f;
    }
    case ORC_F16: {
      uint16_t h;
      memcpy(&h, (const char*)base + 2 * i, 2);
      return orc_f16_to_double(h);
    }
    case ORC_BF16: {
      uint16_t b;
      memcpy(&b, (const char*)base + 2 * i, 2);
      return orc_bf16_to_double(b);
    }
    case ORC_E4M3:
      return orc_e4m3_to_double(((const uint8_t*)base)[i]);
  }
  return NAN;
}

/* Value of element i as an fp32 number (exact for f32/f16/bf16 inputs). */
static float load_elem_f32(const void* base, int64_t i, int dt) {
  return (float)load_elem(base, i, dt);
}

/*
 * FP8 E4M3FN encoder written from the OCP definition: the result is the
 * finite E4M3 value nearest to y; a tie goes to the code whose last mantissa
 * bit is 0 (round half to even); anything beyond the largest finite value
 * (448) saturates to +-448; NaN maps to the NaN code.  Below 448 the code is
 * found by exhaustive search over the 127 non-negative finite codes, so no
 * rounding trick is involved.  (For |y| < 448 every difference |y| - value
 * that can decide a comparison is exact in double; at and above 448 the
 * answer is the saturated code, decided before any subtraction.)
 */
uint8_t orc_e4m3_encode(float y) {
  if (isnan(y)) return 0x7f;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    double err = fabs(a - orc_e4m3_to_double((uint8_t)c));
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* y = fl32(x / scale): one correctly rounded IEEE binary32 division. */
static float div_f32(float x, float scale) {
  volatile float q = x / scale;
  return q;
}

/* E2M1 code nearest to y, by exhaustive search over the 8 magnitudes; a
 * tie goes to the code whose mantissa bit is 0; |y| beyond 6 saturates to
 * 6; the sign bit follows y's sign (so -0 -> 0x8). */
uint8_t orc_e2m1_encode(float y) {
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  double a = fabs((double)y);
  if (a >= 6.0) return (uint8_t)(sign | 0x7);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 7; ++c) {
    double err = fabs(a - orc_e2m1_to_double((uint8_t)c));
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* INT4 code of y: the integer nearest to y (ties to even), clamped to
 * [-7, 7]. */
int orc_int4_encode(float y) {
  double r = rint((double)y); /* the default rounding mode: ties to even */
  if (r > 7.0) r = 7.0;
  if (r < -7.0) r = -7.0;
  return (int)r;
}

/* Quantise the D values of one (token, KV head), src[0 .. D) of type
 * src_dt, into slot o of a 4-bit page (layout above).  INT4: s = fl32(max |x|
 * / 7), code = int4(fl32(x / s)) (all codes 0 when s = 0).  NVFP4, per block
 * of 16: b = e4m3(fl32(fl32(max |x| / 6) / tensor_scale)), then with
 * r = fl32(e4m3 value of b * tensor_scale) code = e2m1(fl32(x / r)) (all
 * codes 0 when r = 0). */
static void quantize_4bit(const void* src, int64_t src0, int src_dt,
                          uint8_t* page, int o, int bs, int D, int dt,
                          float tensor_scale) {
  uint8_t* codes = page + (int64_t)o * (D / 2);
  for (int i = 0; i < D / 2; ++i) codes[i] = 0;
  if (dt == ORC_INT4) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
      float x = fabsf(load_elem_f32(src, src0 + d, src_dt));
      if (x > amax) amax = x;
    }
    float sc = amax > 0.0f ? div_f32(amax, 7.0f) : 0.0f;
    memcpy(page + (int64_t)bs * (D / 2) + 4 * (int64_t)o, &sc, 4);
    for (int d = 0; d < D; ++d) {
      int c = sc > 0.0f ? orc_int4_encode(div_f32(load_elem_f32(src, src0 + d, src_dt), sc)) : 0;
      codes[d / 2] |= (uint8_t)((c & 0xF) << (4 * (d & 1)));
    }
    return;
  }
  uint8_t* scales = page + (int64_t)bs * (D / 2) + (int64_t)o * (D / 16);
  for (int blk = 0; blk < D / 16; ++blk) {
    float amax = 0.0f;
    for (int d = 16 * blk; d < 16 * blk + 16; ++d) {
      float x = fabsf(load_elem_f32(src, src0 + d, src_dt));
      if (x > amax) amax = x;
    }
    uint8_t b = orc_e4m3_encode(div_f32(div_f32(amax, 6.0f), tensor_scale));
    scales[blk] = b;
    float r = (float)(orc_e4m3_to_double(b) * (double)tensor_scale);
    for (int d = 16 * blk; d < 16 * blk + 16; ++d) {
      uint8_t c = r > 0.0f ? orc_e2m1_encode(div_f32(load_elem_f32(src, src0 + d, src_dt), r)) : 0;
      codes[d / 2] |= (uint8_t)(c << (4 * (d & 1)));
    }
  }
}

/* Value of element i of a cache indexed as [block][head][offset][d] (i =
 * ((block * heads + head) * bs + offset) * D + d), decoded exactly; for the
 * 4-bit formats the element is found in its (block, head) page, and the
 * per-tensor scale is left to the caller. */
static double load_kv(const void* cache, int64_t i, int dt, int bs, int D) {
  if (!is_4bit(dt)) return load_elem(cache, i, dt);
  const int64_t page = i / ((int64_t)bs * D);
  const int o = (int)((i / D) % bs), d = (int)(i % D);
  const uint8_t* pg = (const uint8_t*)cache + page * page_bytes_4bit(dt, bs, D);
  const uint8_t byte = pg[(int64_t)o * (D / 2) + d / 2];
  const int nib = (d & 1) ? (byte >> 4) : (byte & 0xF);
  if (dt == ORC_INT4) {
    float sc;
    memcpy(&sc, pg + (int64_t)bs * (D / 2) + 4 * (int64_t)o, 4);
    return (double)sc * (double)(nib >= 8 ? nib - 16 : nib);
  }
  const uint8_t b = pg[(int64_t)bs * (D / 2) + (int64_t)o * (D / 16) + d / 16];
  return orc_e4m3_to_double(b) * orc_e2m1_to_double((uint8_t)nib);
}

/* ---------------------------------------------------------------------- */
/* reshape_and_cache: write each new token's K and V into its slot.        */
/* Cache layout [num_blocks][num_kv_heads][block_size][head_dim]; slot s   */
/* is block s / block_size, offset s % block_size; a negative slot means   */
/* "padding token, not written".                                           */
/* ---------------------------------------------------------------------- */
int orc_reshape_and_cache(const void* key, const void* value, int kv_dtype,
                          int64_t num_tokens, int64_t key_stride,
                          int64_t value_stride, void* k_cache, void* v_cache,
                          int cache_dtype, int64_t num_blocks, int block_size,
                          int num_kv_heads, int head_dim,
                          const int64_t* slot_mapping, float k_scale,
                          float v_scale) {
  int eb = elem_bytes(cache_dtype);
  if ((eb == 0 && !is_4bit(cache_dtype)) || elem_bytes(kv_dtype) == 0 ||
      kv_dtype == ORC_E4M3)
    return ORC_BAD_ARG;
  if (cache_dtype != kv_dtype && cache_dtype != ORC_E4M3 && !is_4bit(cache_dtype))
    return ORC_BAD_ARG;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t b = slot / block_size;
    int64_t o = slot % block_size;
    if (b >= num_blocks) return ORC_BAD_INDEX;
    if (is_4bit(cache_dtype)) {
      const int64_t pb = page_bytes_4bit(cache_dtype, block_size, head_dim);
      for (int h = 0; h < num_kv_heads; ++h) {
        uint8_t* kp = (uint8_t*)k_cache + (b * num_kv_heads + h) * pb;
        uint8_t* vp = (uint8_t*)v_cache + (b * num_kv_heads + h) * pb;
        quantize_4bit(key, t * key_stride + (int64_t)h * head_dim, kv_dtype, kp,
                      (int)o, block_size, head_dim, cache_dtype, k_scale);
        quantize_4bit(value, t * value_stride + (int64_t)h * head_dim, kv_dtype,
                      vp, (int)o, block_size, head_dim, cache_dtype, v_scale);
      }
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_dim; ++d) {
        int64_t src_k = t * key_stride + (int64_t)h * head_dim + d;
        int64_t src_v = t * value_stride + (int64_t)h * head_dim + d;
        int64_t dst =
            ((b * num_kv_heads + h) * (int64_t)block_size + o) * head_dim + d;
        if (cache_dtype == ORC_E4M3) {
          float xk = load_elem_f32(key, src_k, kv_dtype);
          float xv = load_elem_f32(value, src_v, kv_dtype);
          ((uint8_t*)k_cache)[dst] = orc_e4m3_encode(div_f32(xk, k_scale));
          ((uint8_t*)v_cache)[dst] = orc_e4m3_encode(div_f32(xv, v_scale));
        } else {
          memcpy((char*)k_cache + dst * eb, (const char*)key + src_k * eb, eb);
          memcpy((char*)v_cache + dst * eb, (const char*)value + src_v * eb, eb);
        }
      }
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* copy_blocks: for each (src, dst) pair copy the whole physical block     */
/* (all KV heads, all offsets) of K and of V from src to dst.              */
/* ---------------------------------------------------------------------- */
int orc_copy_blocks(void* k_cache, void* v_cache, int cache_dtype,
                    int64_t num_blocks, int block_size, int num_kv_heads,
                    int head_dim, const int64_t* block_mapping,
                    int64_t num_pairs) {
  int eb = elem_bytes(cache_dtype);
  if (eb == 0 && !is_4bit(cache_dtype)) return ORC_BAD_ARG;
  int64_t block_bytes =
      is_4bit(cache_dtype)
          ? num_kv_heads * page_bytes_4bit(cache_dtype, block_size, head_dim)
          : (int64_t)num_kv_heads * block_size * head_dim * eb;
  for (int64_t p = 0; p < num_pairs; ++p) {
    int64_t src = block_mapping[2 * p], dst = block_mapping[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
      return ORC_BAD_INDEX;
    for (int64_t i = 0; i < block_bytes; ++i) {
      ((char*)k_cache)[dst * block_bytes + i] =
          ((char*)k_cache)[src * block_bytes + i];
      ((char*)v_cache)[dst * block_bytes + i] =
          ((char*)v_cache)[src * block_bytes + i];
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Paged attention for one scheduler step.                                 */
/*                                                                         */
/* Request r owns query tokens [qsl[r], qsl[r+1]) (n_r of them) and has    */
/* L_r = seq_lens[r] keys in the cache, this step's tokens included.       */
/* Query i of request r is the token at absolute position L_r - n_r + i;   */
/* it sees keys 0 .. L_r - n_r + i (causal within the chunk; a decode      */
/* query, n_r = 1, sees all L_r keys).  Query head h reads KV head         */
/* h / (Hq / Hkv).  Key j is stored in block block_tables[r][j / bs] at    */
/* offset j % bs.                                                          */
/*                                                                         */
/*   s_j = scale * sum_d q[d] * k_j[d]                                     */
/*   out = sum_j exp(s_j - max s) v_j / sum_j exp(s_j - max s)             */
/*                                                                         */
/* with k_j = k_scale * stored value (k_scale = 1 unless FP8), likewise v. */
/*                                                                         */
/* With a sliding window of W > 0 keys the query at position p sees only   */
/* keys max(0, p - W + 1) .. p; W = 0 means no window.                     */
/* ---------------------------------------------------------------------- */
static int first_visible_key(int position, int window) {
  if (window <= 0) return 0;
  int first = position - window + 1;
  return first > 0 ? first : 0;
}

typedef struct {
  const void* q;
  int q_dtype;
  const void* k_cache;
  const void* v_cache;
  int cache_dtype;
  int64_t num_blocks;
  int block_size, num_q_heads, num_kv_heads, head_dim;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int num_seqs;
  double scale, k_scale, v_scale;
  int window;
  double* out;
  /* work distribution */
  int64_t next_item;
  pthread_mutex_t lock;
  int status;
} attn_job;

static int attend_one(attn_job* J, int r, int h) {
  const int D = J->head_dim, bs = J->block_size;
  const int group = J->num_q_heads / J->num_kv_heads;
  const int g = h / group;
  const int n = J->query_start_loc[r + 1] - J->query_start_loc[r];
  const int L = J->seq_lens[r];
  if (n == 0) return ORC_OK;
  if (n < 0 || L < n) return ORC_BAD_ARG;
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  double* qv = (double*)malloc(sizeof(double) * (size_t)D);
  if (!s || !qv) {
    free(s);
    free(qv);
    return ORC_BAD_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const int64_t t = J->query_start_loc[r] + i;
    const int visible = L - n + i + 1; /* keys 0 .. L-n+i */
    const int first = first_visible_key(L - n + i, J->window);
    for (int d = 0; d < D; ++d)
      qv[d] = load_elem(J->q, (t * J->num_q_heads + h) * (int64_t)D + d,
                        J->q_dtype);
    double smax = -INFINITY;
    for (int j = first; j < visible; ++j) {
      int32_t b = J->block_tables[(int64_t)r * J->max_blocks_per_seq + j / bs];
      if (b < 0 || b >= J->num_blocks || j / bs >= J->max_blocks_per_seq) {
        free(s);
        free(qv);
        return ORC_BAD_INDEX;
      }
      int64_t base = (((int64_t)b * J->num_kv_heads + g) * bs + j % bs) * D;
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += qv[d] * (J->k_scale * load_kv(J->k_cache, base + d,
                                             J->cache_dtype, bs, D));
      s[j] = J->scale * dot;
      if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    for (int j = first; j < visible; ++j) {
      s[j] = exp(s[j] - smax);
      denom += s[j];
    }
    double* o = J->out + (t * J->num_q_heads + h) * (int64_t)D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = first; j < visible; ++j) {
      int32_t b = J->block_tables[(int64_t)r * J->max_blocks_per_seq + j / bs];
      int64_t base = (((int64_t)b * J->num_kv_heads + g) * bs + j % bs) * D;
      for (int d = 0; d < D; ++d)
        o[d] += s[j] * (J->v_scale *
                        load_kv(J->v_cache, base + d, J->cache_dtype, bs, D));
    }
    for (int d = 0; d < D; ++d) o[d] /= denom;
  }
  free(s);
  free(qv);
  return ORC_OK;
}

static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  const int64_t total = (int64_t)J->num_seqs * J->num_q_heads;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int64_t item = J->next_item++;
    int failed = J->status != ORC_OK;
    pthread_mutex_unlock(&J->lock);
    if (item >= total || failed) break;
    int st = attend_one(J, (int)(item / J->num_q_heads),
                        (int)(item % J->num_q_heads));
    if (st != ORC_OK) {
      pthread_mutex_lock(&J->lock);
      if (J->status == ORC_OK) J->status = st;
      pthread_mutex_unlock(&J->lock);
    }
  }
  return NULL;
}

/* out: [num_tokens][num_q_heads][head_dim] doubles, num_tokens = qsl[B].
 * Rows of tokens that belong to no request are left untouched. */
int orc_paged_attention(const void* q, int q_dtype, const void* k_cache,
                        const void* v_cache, int cache_dtype,
                        int64_t num_blocks, int block_size, int num_q_heads,
                        int num_kv_heads, int head_dim,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* seq_lens,
                        const int32_t* query_start_loc, int num_seqs,
                        double scale, double k_scale, double v_scale,
                        double* out, int num_threads, int window) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || elem_bytes(q_dtype) == 0 ||
      (elem_bytes(cache_dtype) == 0 && !is_4bit(cache_dtype)) ||
      (is_4bit(cache_dtype) && head_dim % 16 != 0) || window < 0)
    return ORC_BAD_ARG;
  attn_job J;
  memset(&J, 0, sizeof J);
  J.q = q;
  J.q_dtype = q_dtype;
  J.k_cache = k_cache;
  J.v_cache = v_cache;
  J.cache_dtype = cache_dtype;
  J.num_blocks = num_blocks;
  J.block_size = block_size;
  J.num_q_heads = num_q_heads;
  J.num_kv_heads = num_kv_heads;
  J.head_dim = head_dim;
  J.block_tables = block_tables;
  J.max_blocks_per_seq = max_blocks_per_seq;
  J.seq_lens = seq_lens;
  J.query_start_loc = query_start_loc;
  J.num_seqs = num_seqs;
  J.scale = scale;
  J.k_scale = (cache_dtype == ORC_E4M3 || cache_dtype == ORC_NVFP4) ? k_scale : 1.0;
  J.v_scale = (cache_dtype == ORC_E4M3 || cache_dtype == ORC_NVFP4) ? v_scale : 1.0;
  J.window = window;
  J.out = out;
  J.next_item = 0;
  J.status = ORC_OK;
  pthread_mutex_init(&J.lock, NULL);
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 512) num_threads = 512;
  pthread_t th[512];
  int started = 0;
  for (int i = 1; i < num_threads; ++i)
    if (pthread_create(&th[started], NULL, attn_worker, &J) == 0) ++started;
  attn_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.status;
}

/*
 * One output row (request r, query i, head h) on its own: the same
 * definition as above for a single row, used to check sampled outputs of
 * very large steps without computing the whole step.
 */
int orc_paged_attention_row(const void* q, int q_dtype, const void* k_cache,
                            const void* v_cache, int cache_dtype,
                            int64_t num_blocks, int block_size,
                            int num_q_heads, int num_kv_heads, int head_dim,
                            const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int r, int i,
                            int h, double scale, double k_scale,
                            double v_scale, double* out_row, int window) {
  const int D = head_dim, bs = block_size;
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ORC_BAD_ARG;
  const int g = h / (num_q_heads / num_kv_heads);
  const int n = query_start_loc[r + 1] - query_start_loc[r];
  const int L = seq_lens[r];
  if (i < 0 || i >= n || L < n || window < 0) return ORC_BAD_ARG;
  const double ks = (cache_dtype == ORC_E4M3 || cache_dtype == ORC_NVFP4) ? k_scale : 1.0;
  const double vs = (cache_dtype == ORC_E4M3 || cache_dtype == ORC_NVFP4) ? v_scale : 1.0;
  const int64_t t = query_start_loc[r] + i;
  const int visible = L - n + i + 1;
  const int first = first_visible_key(L - n + i, window);
  double* s = (double*)malloc(sizeof(double) * (size_t)visible);
  if (!s) return ORC_BAD_ARG;
  double smax = -INFINITY;
  for (int j = first; j < visible; ++j) {
    int32_t b = block_tables[(int64_t)r * max_blocks_per_seq + j / bs];
    if (b < 0 || b >= num_blocks) {
      free(s);
      return ORC_BAD_INDEX;
    }
    int64_t base = (((int64_t)b * num_kv_heads + g) * bs + j % bs) * D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += load_elem(q, (t * num_q_heads + h) * (int64_t)D + d, q_dtype) *
             (ks * load_kv(k_cache, base + d, cache_dtype, bs, D));
    s[j] = scale * dot;
    if (s[j] > smax) smax = s[j];
  }
  double denom = 0.0;
  for (int j = first; j < visible; ++j) {
    s[j] = exp(s[j] - smax);
    denom += s[j];
  }
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  for (int j = first; j < visible; ++j) {
    int32_t b = block_tables[(int64_t)r * max_blocks_per_seq + j / bs];
    int64_t base = (((int64_t)b * num_kv_heads + g) * bs + j % bs) * D;
    for (int d = 0; d < D; ++d)
      out_row[d] += s[j] * (vs * load_kv(v_cache, base + d, cache_dtype, bs, D));
  }
  for (int d = 0; d < D; ++d) out_row[d] /= denom;
  free(s);
  return ORC_OK;
}

/* Per-token KV bytes (Table 1): 2 (K and V) x element bytes x layers x KV
 * heads x head dim. */
int64_t orc_kv_bytes_per_token(int64_t elem_bytes_, int64_t layers,
                               int64_t kv_heads, int64_t head_dim) {
  return 2 * elem_bytes_ * layers * kv_heads * head_dim;
}
