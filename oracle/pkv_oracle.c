/*
 * pkv_oracle.c -- CPU oracle for decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the timed CPU
 * baseline of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Everything here is the plain definition of what the pages describe, written
 * for a reader to check by eye: no blocking, no fusion, no reordering.
 * Floating point is fp64 except where the method itself fixes a precision
 * (the FP8 quantiser's scale and quotient are fp32, because the stored code is
 * an integer decided by that fp32 value).
 *
 * Sources (page title, section):
 *   [LC]  "长上下文优化：注意力稀疏化与 KV Cache 管理" (plumephp.com,
 *         llm-long-context-optimization): KV-size formula; sliding-window mask
 *         |i-j| <= window; StreamingKVCache (sinks + recent window);
 *         H2OEviction (update_scores / select); logical->physical block table.
 *   [PA]  "KV Cache 与 PagedAttention：显存复用与长上下文推理" (plumephp.com,
 *         ai-kv-cache-paged-attention): 16-token blocks, global free pool,
 *         per-request block table, Block{bid, refcount} + copy_on_write,
 *         FP8 (E4M3) / INT8 KV with per-token or per-channel scaling.
 *   [SO]  "系统优化" (threethreeliu.top, knowledge-inference-optimization-
 *         memory): sliding window / StreamingLLM keep-set, H2O evict_tokens.
 *
 * Where the pages are silent or garbled, the reading taken is stated next to
 * the code that adopts it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_BLOCK 16 /* [PA] PagedAttention design: fixed blocks of 16 tokens by default */

enum { KV_FP32 = 0, KV_BF16 = 1, KV_FP8 = 2, KV_INT8 = 3 };
enum { MASK_FULL = 0, MASK_SLIDING = 1, MASK_SINK_WINDOW = 2 };

/* ------------------------------------------------------------------------- */
/* Input element decoding (bytes -> value).                                   */
/* ------------------------------------------------------------------------- */

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16; /* bf16 is the top half of an fp32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 ([PA] quantisation section: FP8 E4M3 KV with per-token scales).   */
/* Encoding follows the OCP 8-bit floating point specification, E4M3 variant: */
/* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,      */
/* S.1111.111 is NaN, largest finite magnitude 448 = 1.75 * 2^8.              */
/* ------------------------------------------------------------------------- */

double oracle_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    mag = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* Round-to-nearest-even of q >= 0 to an integer (q is exact in double). */
static int round_half_even(double q) {
  double fl = floor(q);
  double rem = q - fl;
  int n = (int)fl;
  if (rem > 0.5 || (rem == 0.5 && (n & 1))) n++;
  return n;
}

/* fp32 -> E4M3, round to nearest even, saturating to +-448 ("satfinite"):
 * every finite or infinite magnitude above 448 becomes 448; NaN -> 0x7F.
 * The sign of zero is kept. */
uint8_t oracle_e4m3_encode(float x) {
  uint8_t sign;
  double a;
  if (isnan(x)) return 0x7F;
  sign = signbit(x) ? 0x80 : 0x00;
  a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: spacing 2^-9; m == 8 lands exactly on the smallest
     * normal (exponent field 1, mantissa 0), whose bit pattern is also 8. */
    int m = round_half_even(a * 512.0);
    return (uint8_t)(sign | m);
  }
  {
    int ex, e, m, ef;
    (void)frexp(a, &ex); /* a = f * 2^ex with f in [0.5, 1) */
    e = ex - 1;          /* a = (1 + m/8) * 2^e */
    m = round_half_even((ldexp(a, -e) - 1.0) * 8.0);
    if (m == 8) {
      m = 0;
      e += 1;
    }
    ef = e + 7;
    return (uint8_t)(sign | (ef << 3) | m);
  }
}

/* Per-token quantisation of one (token, kv_head) row of D bf16 values.
 * Reading adopted: scale s = absmax / 448 in fp32 (s = 1 when absmax == 0),
 * code_d = E4M3(x_d / s) with the quotient rounded to fp32 first. */
void oracle_quantize_row_bf16(const uint16_t* x, int D, uint8_t* codes, float* scale) {
  float amax = 0.0f, s;
  int d;
  for (d = 0; d < D; d++) {
    float v = fabsf(bf16_bits_to_float(x[d]));
    if (v > amax) amax = v;
  }
  s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
  for (d = 0; d < D; d++) {
    float q = bf16_bits_to_float(x[d]) / s;
    codes[d] = oracle_e4m3_encode(q);
  }
  *scale = s;
}

/* fp32 -> symmetric INT8: round to nearest, ties to even, then clamp to
 * [-127, 127] (-128 is never produced, so the code range is symmetric). */
int8_t oracle_int8_encode(float x) {
  double a = fabs((double)x);
  int n;
  if (a != a) return 0;
  if (a > 127.0) a = 127.0;
  n = round_half_even(a);
  if (n > 127) n = 127;
  return (int8_t)(x < 0.0f ? -n : n);
}

/* Per-token INT8 quantisation of one (token, kv_head) row of D bf16 values
 * ([PA] KV quantisation, FP16 -> INT8 with per-token scaling).  Reading
 * adopted: symmetric, s = absmax / 127 in fp32 (s = 1 when absmax == 0),
 * code_d = INT8(x_d / s) with the quotient rounded to fp32 first. */
void oracle_quantize_row_int8(const uint16_t* x, int D, int8_t* codes, float* scale) {
  float amax = 0.0f, s;
  int d;
  for (d = 0; d < D; d++) {
    float v = fabsf(bf16_bits_to_float(x[d]));
    if (v > amax) amax = v;
  }
  s = (amax == 0.0f) ? 1.0f : amax / 127.0f;
  for (d = 0; d < D; d++) {
    float q = bf16_bits_to_float(x[d]) / s;
    codes[d] = oracle_int8_encode(q);
  }
  *scale = s;
}

/* Per-channel scaling ([PA] KV quantisation: "per-channel / per-token"
 * scaling).  Reading adopted: every (kv head, channel d) has a fixed scale
 * c_d > 0 chosen by the caller, and the per-token scale is kept on top of
 * it: the row is first divided by its channel scales, y_d = x_d / c_d in
 * fp32, then quantised per token exactly as above (s = absmax(y) / qmax,
 * code_d = Q(y_d / s)).  The value a code stands for is code_d * s * c_d.
 * c = NULL means c_d = 1 (y = x exactly: the per-token scheme). */
void oracle_quantize_row_channel(const uint16_t* x, int D, const float* c, int kv_dtype, void* codes,
                                 float* scale) {
  float amax = 0.0f, s, y;
  const float qmax = kv_dtype == KV_INT8 ? 127.0f : 448.0f;
  int d;
  for (d = 0; d < D; d++) {
    const float v = c ? bf16_bits_to_float(x[d]) / c[d] : bf16_bits_to_float(x[d]);
    if (fabsf(v) > amax) amax = fabsf(v);
  }
  s = (amax == 0.0f) ? 1.0f : amax / qmax;
  for (d = 0; d < D; d++) {
    y = c ? bf16_bits_to_float(x[d]) / c[d] : bf16_bits_to_float(x[d]);
    if (kv_dtype == KV_INT8)
      ((int8_t*)codes)[d] = oracle_int8_encode(y / s);
    else
      ((uint8_t*)codes)[d] = oracle_e4m3_encode(y / s);
  }
  *scale = s;
}

/* ------------------------------------------------------------------------- */
/* Keep-set predicates.                                                       */
/*   FULL:         every j in [0, L).                                         */
/*   SLIDING(W):   [LC] sliding_window_mask keeps |i - j| <= window; decode    */
/*                 queries i = L-1, causal, so j in [L-1-W, L-1] (W+1 keys).   */
/*   SINK_WINDOW:  [LC] StreamingKVCache keeps the first num_sinks and the    */
/*                 last window entries once the total exceeds sinks+window;    */
/*                 otherwise everything.                                       */
/* ------------------------------------------------------------------------- */

int oracle_keep(int L, int mode, int num_sinks, int window, int j) {
  if (j < 0 || j >= L) return 0;
  if (mode == MASK_FULL) return 1;
  if (mode == MASK_SLIDING) {
    int i = L - 1;
    int dist = i - j;
    return dist <= window;
  }
  if (mode == MASK_SINK_WINDOW) {
    if (L <= num_sinks + window) return 1;
    return j < num_sinks || j >= L - window;
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Paged storage. Reading adopted for the in-block layout:                     */
/*   pool[block][kv_head][slot][d], slot = token % 16, block from the table.  */
/* ------------------------------------------------------------------------- */

static size_t pool_index(int block, int Hk, int g, int slot, int D, int d) {
  return (((size_t)block * Hk + g) * ORACLE_BLOCK + slot) * D + d;
}

/* Scatter per-token rows into the pool at the given slots
 * (slot = block * 16 + offset).  src is [T][Hk][D], elem_bytes per element. */
void oracle_scatter(void* pool, int Hk, int D, int elem_bytes, const int64_t* slots,
                    int T, const void* src) {
  int t, g;
  for (t = 0; t < T; t++) {
    int block = (int)(slots[t] / ORACLE_BLOCK), slot = (int)(slots[t] % ORACLE_BLOCK);
    for (g = 0; g < Hk; g++) {
      size_t dst = pool_index(block, Hk, g, slot, D, 0) * (size_t)elem_bytes;
      size_t s = (((size_t)t * Hk + g) * D) * (size_t)elem_bytes;
      memcpy((char*)pool + dst, (const char*)src + s, (size_t)D * elem_bytes);
    }
  }
}

/* Quantised variants (FP8 E4M3 or INT8): quantise each (token, kv_head) row
 * of bf16 and scatter codes and the per-token scale (scale pool layout
 * [block][kv_head][slot]); channel (NULL or [Hk][D]) gives the per-channel
 * scales.  Tokens are independent (distinct slots), so they are spread over
 * the host's cores. */
typedef struct {
  uint8_t* pool;
  float* scale_pool;
  int Hk, D, T, thread_id, n_threads, kv_dtype;
  const int64_t* slots;
  const uint16_t* src;
  const float* channel;
} quantize_job;

static void* quantize_worker(void* arg) {
  quantize_job* q = (quantize_job*)arg;
  int t, g;
  for (t = q->thread_id; t < q->T; t += q->n_threads) {
    int block = (int)(q->slots[t] / ORACLE_BLOCK), slot = (int)(q->slots[t] % ORACLE_BLOCK);
    for (g = 0; g < q->Hk; g++) {
      size_t di = pool_index(block, q->Hk, g, slot, q->D, 0);
      size_t si = ((size_t)block * q->Hk + g) * ORACLE_BLOCK + slot;
      const uint16_t* row = q->src + ((size_t)t * q->Hk + g) * q->D;
      if (q->channel)
        oracle_quantize_row_channel(row, q->D, q->channel + (size_t)g * q->D, q->kv_dtype, q->pool + di,
                                    q->scale_pool + si);
      else if (q->kv_dtype == KV_INT8)
        oracle_quantize_row_int8(row, q->D, (int8_t*)(q->pool + di), q->scale_pool + si);
      else
        oracle_quantize_row_bf16(row, q->D, q->pool + di, q->scale_pool + si);
    }
  }
  return NULL;
}

void oracle_quantize_scatter(uint8_t* pool, float* scale_pool, int Hk, int D, const int64_t* slots, int T,
                             const uint16_t* src, int kv_dtype, const float* channel) {
  long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
  int n = (int)(ncpu > 0 ? ncpu : 1), i;
  quantize_job* jobs;
  pthread_t* th;
  if (n > 64) n = 64;
  if (T < 4096) n = 1;
  jobs = (quantize_job*)malloc(sizeof(quantize_job) * n);
  th = (pthread_t*)malloc(sizeof(pthread_t) * n);
  for (i = 0; i < n; i++) {
    jobs[i].pool = pool;
    jobs[i].scale_pool = scale_pool;
    jobs[i].Hk = Hk;
    jobs[i].D = D;
    jobs[i].T = T;
    jobs[i].thread_id = i;
    jobs[i].n_threads = n;
    jobs[i].slots = slots;
    jobs[i].src = src;
    jobs[i].kv_dtype = kv_dtype;
    jobs[i].channel = channel;
    pthread_create(&th[i], NULL, quantize_worker, &jobs[i]);
  }
  for (i = 0; i < n; i++) pthread_join(th[i], NULL);
  free(jobs);
  free(th);
}

/* Copy rows (all kv heads, K, V and scales) from slot src[t] to slot dst[t]. */
void oracle_copy_rows(void* k_pool, void* v_pool, float* k_scale, float* v_scale, int Hk, int D, int elem_bytes,
                      const int64_t* src, const int64_t* dst, int n) {
  int t, g;
  for (t = 0; t < n; t++) {
    int sb = (int)(src[t] / ORACLE_BLOCK), so = (int)(src[t] % ORACLE_BLOCK);
    int db = (int)(dst[t] / ORACLE_BLOCK), dso = (int)(dst[t] % ORACLE_BLOCK);
    for (g = 0; g < Hk; g++) {
      size_t si = pool_index(sb, Hk, g, so, D, 0), di = pool_index(db, Hk, g, dso, D, 0);
      memcpy((char*)k_pool + di * elem_bytes, (char*)k_pool + si * elem_bytes, (size_t)D * elem_bytes);
      memcpy((char*)v_pool + di * elem_bytes, (char*)v_pool + si * elem_bytes, (size_t)D * elem_bytes);
      if (k_scale && v_scale) {
        k_scale[((size_t)db * Hk + g) * ORACLE_BLOCK + dso] = k_scale[((size_t)sb * Hk + g) * ORACLE_BLOCK + so];
        v_scale[((size_t)db * Hk + g) * ORACLE_BLOCK + dso] = v_scale[((size_t)sb * Hk + g) * ORACLE_BLOCK + so];
      }
    }
  }
}

/* Copy one whole physical block (all kv heads, all slots, K, V and scales):
 * [PA] copy-on-write, where the fresh block receives the shared block's data. */
void oracle_copy_block(void* k_pool, void* v_pool, float* k_scale, float* v_scale, int Hk,
                       int D, int elem_bytes, int src, int dst) {
  size_t blk = (size_t)Hk * ORACLE_BLOCK * D * elem_bytes;
  memcpy((char*)k_pool + (size_t)dst * blk, (char*)k_pool + (size_t)src * blk, blk);
  memcpy((char*)v_pool + (size_t)dst * blk, (char*)v_pool + (size_t)src * blk, blk);
  if (k_scale && v_scale) {
    size_t sb = (size_t)Hk * ORACLE_BLOCK;
    memcpy(k_scale + (size_t)dst * sb, k_scale + (size_t)src * sb, sb * sizeof(float));
    memcpy(v_scale + (size_t)dst * sb, v_scale + (size_t)src * sb, sb * sizeof(float));
  }
}

/* ------------------------------------------------------------------------- */
/* Decode attention: the plain definition, gathered through the block table.  */
/* For sequence b, query head h, kv head g = h / G ([LC] GQA: a group of      */
/* query heads shares one KV head; reading: contiguous groups):               */
/*   K_j = dequant(pool[table[b][j/16]][g][j%16][:])                          */
/*   s_j = scale * <q_h, K_j>        for j in keep(b)                        */
/*   lse = ln sum_j exp(s_j),  out = sum_j exp(s_j - lse) V_j                */
/* Empty keep-set: out = 0, lse = -inf.                                       */
/* ------------------------------------------------------------------------- */

typedef struct {
  int n_seqs, H, Hk, D, kv_dtype, q_dtype;
  const void *k_pool, *v_pool;
  const float *k_scale, *v_scale;
  const float *k_channel, *v_channel; /* per-channel scales [Hk][D], or NULL */
  const int32_t* tables;
  int max_blocks;
  const int32_t* lens;
  const void* q;
  double scale;
  int mask_mode, num_sinks, window;
  double *out, *lse, *logits;
  int logits_stride;
  int n_threads, thread_id;
  int bad_block; /* set when a kept token's table entry is not a valid block */
  int num_blocks;
} decode_job;

/* The value element d of a pool slot stands for: FP8 / INT8 code times the
 * token's scale (times the channel's scale when the pool has them). */
static double kv_value(const decode_job* jb, const void* pool, const float* scl, const float* channel,
                       int block, int g, int slot, int d) {
  size_t i = pool_index(block, jb->Hk, g, slot, jb->D, d);
  if (jb->kv_dtype == KV_FP32) return (double)((const float*)pool)[i];
  if (jb->kv_dtype == KV_BF16) return bf16_bits_to_double(((const uint16_t*)pool)[i]);
  {
    size_t si = ((size_t)block * jb->Hk + g) * ORACLE_BLOCK + slot;
    double c = channel ? (double)channel[(size_t)g * jb->D + d] : 1.0;
    if (jb->kv_dtype == KV_INT8) return (double)((const int8_t*)pool)[i] * (double)scl[si] * c;
    return oracle_e4m3_decode(((const uint8_t*)pool)[i]) * (double)scl[si] * c;
  }
}

static double q_value(const decode_job* jb, int b, int h, int d) {
  size_t i = ((size_t)b * jb->H + h) * jb->D + d;
  if (jb->q_dtype == KV_FP32) return (double)((const float*)jb->q)[i];
  return bf16_bits_to_double(((const uint16_t*)jb->q)[i]);
}

static void decode_one(decode_job* jb, int b, int h) {
  int G = jb->H / jb->Hk, g = h / G, D = jb->D, L = jb->lens[b];
  double* o = jb->out + ((size_t)b * jb->H + h) * D;
  double* s = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
  double m = -INFINITY, sum = 0.0, lse;
  int j, d, any = 0;
  for (d = 0; d < D; d++) o[d] = 0.0;
  for (j = 0; j < L; j++) {
    int block, slot;
    double dot = 0.0;
    if (!oracle_keep(L, jb->mask_mode, jb->num_sinks, jb->window, j)) continue;
    block = jb->tables[(size_t)b * jb->max_blocks + j / ORACLE_BLOCK];
    slot = j % ORACLE_BLOCK;
    if (block < 0 || block >= jb->num_blocks) {
      jb->bad_block = 1;
      s[j] = -INFINITY;
      continue;
    }
    for (d = 0; d < D; d++)
      dot += q_value(jb, b, h, d) * kv_value(jb, jb->k_pool, jb->k_scale, jb->k_channel, block, g, slot, d);
    s[j] = jb->scale * dot;
    if (jb->logits) jb->logits[((size_t)b * jb->H + h) * jb->logits_stride + j] = s[j];
    if (s[j] > m) m = s[j];
    any = 1;
  }
  if (!any) {
    jb->lse[(size_t)b * jb->H + h] = -INFINITY;
    free(s);
    return;
  }
  for (j = 0; j < L; j++)
    if (oracle_keep(L, jb->mask_mode, jb->num_sinks, jb->window, j)) sum += exp(s[j] - m);
  lse = m + log(sum);
  jb->lse[(size_t)b * jb->H + h] = lse;
  for (j = 0; j < L; j++) {
    int block, slot;
    double p;
    if (!oracle_keep(L, jb->mask_mode, jb->num_sinks, jb->window, j)) continue;
    block = jb->tables[(size_t)b * jb->max_blocks + j / ORACLE_BLOCK];
    slot = j % ORACLE_BLOCK;
    if (block < 0 || block >= jb->num_blocks) continue;
    p = exp(s[j] - lse);
    for (d = 0; d < D; d++)
      o[d] += p * kv_value(jb, jb->v_pool, jb->v_scale, jb->v_channel, block, g, slot, d);
  }
  free(s);
}

static void* decode_worker(void* arg) {
  decode_job* jb = (decode_job*)arg;
  int pairs = jb->n_seqs * jb->H, p;
  for (p = jb->thread_id; p < pairs; p += jb->n_threads) decode_one(jb, p / jb->H, p % jb->H);
  return NULL;
}

/* Returns 0, or 1 when some kept token pointed at an invalid block.
 * k_channel / v_channel: per-channel scales [Hk][D] of an FP8 / INT8 pool, or
 * NULL. */
int oracle_decode(int n_seqs, int H, int Hk, int D, int kv_dtype, const void* k_pool,
                  const void* v_pool, const float* k_scale, const float* v_scale, int num_blocks,
                  const int32_t* tables, int max_blocks, const int32_t* lens, int q_dtype,
                  const void* q, double scale, int mask_mode, int num_sinks, int window,
                  double* out, double* lse, double* logits, int logits_stride, int n_threads,
                  const float* k_channel, const float* v_channel) {
  decode_job base, *jobs;
  pthread_t* th;
  int t, bad = 0;
  if (n_threads < 1) n_threads = 1;
  base.n_seqs = n_seqs;
  base.H = H;
  base.Hk = Hk;
  base.D = D;
  base.kv_dtype = kv_dtype;
  base.q_dtype = q_dtype;
  base.k_pool = k_pool;
  base.v_pool = v_pool;
  base.k_scale = k_scale;
  base.v_scale = v_scale;
  base.k_channel = k_channel;
  base.v_channel = v_channel;
  base.tables = tables;
  base.max_blocks = max_blocks;
  base.lens = lens;
  base.q = q;
  base.scale = scale;
  base.mask_mode = mask_mode;
  base.num_sinks = num_sinks;
  base.window = window;
  base.out = out;
  base.lse = lse;
  base.logits = logits;
  base.logits_stride = logits_stride;
  base.n_threads = n_threads;
  base.bad_block = 0;
  base.num_blocks = num_blocks;
  jobs = (decode_job*)malloc(sizeof(decode_job) * n_threads);
  th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
  for (t = 0; t < n_threads; t++) {
    jobs[t] = base;
    jobs[t].thread_id = t;
    pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
  }
  for (t = 0; t < n_threads; t++) {
    pthread_join(th[t], NULL);
    bad |= jobs[t].bad_block;
  }
  free(jobs);
  free(th);
  return bad;
}

/* ------------------------------------------------------------------------- */
/* H2O ([LC] H2OEviction).                                                    */
/* update_scores: attention weights [heads, q_len, kv_len] are summed over the */
/* query axis and averaged over heads, then accumulated into the running       */
/* scores.  Reading: the running scores are zero-extended to the current      */
/* kv_len before the add (the page's slice-add assumes the opposite length    */
/* order); masked positions have weight 0; the mean is over all query heads.  */
/* Decode has q_len = 1, so the weight of (h, j) is exp(s_hj - lse_h).        */
/* ------------------------------------------------------------------------- */

void oracle_h2o_update(int n_seqs, int H, const int32_t* lens, const double* logits,
                       int logits_stride, const double* lse, int mask_mode, int num_sinks,
                       int window, double* acc, int acc_stride) {
  int b, h, j;
  for (b = 0; b < n_seqs; b++) {
    int L = lens[b];
    for (j = 0; j < L; j++) {
      double cur = 0.0;
      if (!oracle_keep(L, mask_mode, num_sinks, window, j)) continue;
      for (h = 0; h < H; h++) {
        double w = exp(logits[((size_t)b * H + h) * logits_stride + j] - lse[(size_t)b * H + h]);
        cur += w; /* sum over the single decode query, then over heads */
      }
      acc[(size_t)b * acc_stride + j] += cur / (double)H; /* mean over heads */
    }
  }
}

/* select: keep = budget - recent.  The last `recent` positions are always
 * kept; the rest of the budget goes to the highest accumulated scores among
 * positions [0, L - recent).  Result sorted ascending, no duplicates.
 * Readings: L <= budget (or fewer candidates than keep) keeps everything;
 * ties between equal scores go to the lower position. */
typedef struct {
  double score;
  int pos;
} scored_pos;

static int cmp_desc_score_asc_pos(const void* a, const void* b) {
  const scored_pos* x = (const scored_pos*)a;
  const scored_pos* y = (const scored_pos*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

int oracle_h2o_select(int L, int budget, int recent, const double* scores, int32_t* keep_out) {
  int keep = budget - recent, ncand = L - recent, n = 0, j;
  unsigned char* chosen;
  scored_pos* c;
  if (L <= 0) return 0;
  if (L <= budget || ncand <= keep) {
    for (j = 0; j < L; j++) keep_out[n++] = j;
    return n;
  }
  chosen = (unsigned char*)calloc((size_t)L, 1);
  c = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)ncand);
  for (j = 0; j < ncand; j++) {
    c[j].score = scores[j];
    c[j].pos = j;
  }
  qsort(c, (size_t)ncand, sizeof(scored_pos), cmp_desc_score_asc_pos);
  for (j = 0; j < keep; j++) chosen[c[j].pos] = 1;
  for (j = ncand; j < L; j++) chosen[j] = 1; /* recent window */
  for (j = 0; j < L; j++)
    if (chosen[j]) keep_out[n++] = j;
  free(c);
  free(chosen);
  return n;
}

/* The combined cache rule ([PA] KV compression, the combination of initial
 * tokens, a recent window and high-attention tokens, with sink 4, window 256
 * and 512 - 4 - 256 heavy hitters): position p of a length-L sequence stays
 * when p < sinks, when p is one of the last `window` positions, or when its
 * accumulated score is among the `heavy` highest of ALL L positions.
 * Readings: the ranking spans every position, as the printed rule ranks the
 * whole score array, so a heavy hitter that is also a sink or recent counts
 * once and the kept set can be smaller than sinks + window + heavy; ties go
 * to the lower position.  Result ascending; returns its size. */
int oracle_policy_select(int L, int sinks, int window, int heavy, const double* scores, int32_t* keep_out) {
  unsigned char* heavy_hit;
  scored_pos* c;
  int j, n = 0;
  if (L <= 0) return 0;
  heavy_hit = (unsigned char*)calloc((size_t)L, 1);
  c = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)L);
  for (j = 0; j < L; j++) {
    c[j].score = scores[j];
    c[j].pos = j;
  }
  qsort(c, (size_t)L, sizeof(scored_pos), cmp_desc_score_asc_pos);
  for (j = 0; j < heavy && j < L; j++) heavy_hit[c[j].pos] = 1;
  for (j = 0; j < L; j++) {
    const int is_sink = j < sinks, is_recent = j >= L - window;
    if (is_sink || is_recent || heavy_hit[j]) keep_out[n++] = j;
  }
  free(c);
  free(heavy_hit);
  return n;
}

/* ------------------------------------------------------------------------- */
/* Block allocator replay ([PA] PagedAttention design, three runtime         */
/* components; Block{bid, refcount}; copy_on_write).                          */
/* Readings adopted:                                                          */
/*  - the free pool starts as a Fisher-Yates shuffle of [0, NB) driven by     */
/*    splitmix64(seed) (identity order when seed == 0), or an explicit order; */
/*  - allocation takes the front of the free pool; a freed block goes back to */
/*    the front (last freed, first reused);                                   */
/*  - a sequence id is the smallest id not in use;                            */
/*  - appending token position p of a sequence: p % 16 == 0 takes a new      */
/*    block; otherwise, if the last block is shared (refcount > 1), it is     */
/*    copied to a fresh block first (copy-on-write), the old block's count    */
/*    drops by one and the table points at the copy;                          */
/*  - sequences are processed in the order given; an append that cannot get   */
/*    every block it needs changes nothing;                                   */
/*  - fork shares every block (count + 1); free drops every count by one and  */
/*    returns blocks that reach zero, in ascending logical order;             */
/*  - streaming eviction frees every block wholly outside the sink + window  */
/*    keep-set (entry becomes -1), in ascending logical order;                */
/*  - truncation frees blocks past the new length, in ascending order; it is  */
/*    refused when the new last block is partial and was evicted.             */
/* ------------------------------------------------------------------------- */

typedef struct {
  int NB, max_seqs, max_blocks;
  int32_t* refcount; /* per physical block */
  int32_t* free_stack;
  int free_top; /* front of the free pool is free_stack[free_top - 1] */
  int32_t* tables;
  int32_t* lens;
  unsigned char* active;
  /* CPU swap space: NH host blocks with their own counts and free pool; a
   * swapped-out sequence keeps its length, its device table row is empty
   * and its blocks are named by host_tables. */
  int NH;
  int32_t* host_refcount;
  int32_t* host_free_stack;
  int host_free_top;
  int32_t* host_tables;
  unsigned char* swapped;
} oracle_alloc;

static uint64_t splitmix64_next(uint64_t* state) {
  uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* The raw generator stream (checked against the generator's published test
 * vector, since the free-pool order depends on it). */
void oracle_splitmix64(uint64_t seed, int n, uint64_t* out) {
  uint64_t st = seed;
  int i;
  for (i = 0; i < n; i++) out[i] = splitmix64_next(&st);
}

oracle_alloc* oracle_alloc_create(int NB, int max_seqs, int max_blocks, uint64_t seed,
                                  const int32_t* order) {
  oracle_alloc* a = (oracle_alloc*)calloc(1, sizeof(oracle_alloc));
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NB > 0 ? NB : 1));
  int i;
  a->NB = NB;
  a->max_seqs = max_seqs;
  a->max_blocks = max_blocks;
  a->refcount = (int32_t*)calloc((size_t)(NB > 0 ? NB : 1), sizeof(int32_t));
  a->free_stack = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NB > 0 ? NB : 1));
  a->tables = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_seqs * max_blocks);
  a->lens = (int32_t*)calloc((size_t)max_seqs, sizeof(int32_t));
  a->active = (unsigned char*)calloc((size_t)max_seqs, 1);
  for (i = 0; i < max_seqs * max_blocks; i++) a->tables[i] = -1;
  a->NH = 0;
  a->host_refcount = (int32_t*)calloc(1, sizeof(int32_t));
  a->host_free_stack = (int32_t*)calloc(1, sizeof(int32_t));
  a->host_free_top = 0;
  a->host_tables = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_seqs * max_blocks);
  for (i = 0; i < max_seqs * max_blocks; i++) a->host_tables[i] = -1;
  a->swapped = (unsigned char*)calloc((size_t)max_seqs, 1);
  if (order) {
    for (i = 0; i < NB; i++) perm[i] = order[i];
  } else {
    uint64_t st = seed;
    for (i = 0; i < NB; i++) perm[i] = i;
    if (seed != 0) {
      for (i = NB - 1; i >= 1; i--) {
        int j = (int)(splitmix64_next(&st) % (uint64_t)(i + 1));
        int32_t tmp = perm[i];
        perm[i] = perm[j];
        perm[j] = tmp;
      }
    }
  }
  /* front of the pool = perm[0]: push in reverse so it ends on top */
  a->free_top = 0;
  for (i = NB - 1; i >= 0; i--) a->free_stack[a->free_top++] = perm[i];
  free(perm);
  return a;
}

void oracle_alloc_destroy(oracle_alloc* a) {
  if (!a) return;
  free(a->refcount);
  free(a->free_stack);
  free(a->tables);
  free(a->lens);
  free(a->active);
  free(a->host_refcount);
  free(a->host_free_stack);
  free(a->host_tables);
  free(a->swapped);
  free(a);
}

static oracle_alloc* alloc_clone(const oracle_alloc* a) {
  oracle_alloc* c = (oracle_alloc*)calloc(1, sizeof(oracle_alloc));
  size_t nb = (size_t)(a->NB > 0 ? a->NB : 1), nt = (size_t)a->max_seqs * a->max_blocks;
  *c = *a;
  c->refcount = (int32_t*)malloc(sizeof(int32_t) * nb);
  c->free_stack = (int32_t*)malloc(sizeof(int32_t) * nb);
  c->tables = (int32_t*)malloc(sizeof(int32_t) * nt);
  c->lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)a->max_seqs);
  c->active = (unsigned char*)malloc((size_t)a->max_seqs);
  memcpy(c->refcount, a->refcount, sizeof(int32_t) * nb);
  memcpy(c->free_stack, a->free_stack, sizeof(int32_t) * nb);
  memcpy(c->tables, a->tables, sizeof(int32_t) * nt);
  memcpy(c->lens, a->lens, sizeof(int32_t) * (size_t)a->max_seqs);
  memcpy(c->active, a->active, (size_t)a->max_seqs);
  {
    size_t nh = (size_t)(a->NH > 0 ? a->NH : 1);
    c->host_refcount = (int32_t*)malloc(sizeof(int32_t) * nh);
    c->host_free_stack = (int32_t*)malloc(sizeof(int32_t) * nh);
    c->host_tables = (int32_t*)malloc(sizeof(int32_t) * nt);
    c->swapped = (unsigned char*)malloc((size_t)a->max_seqs);
    memcpy(c->host_refcount, a->host_refcount, sizeof(int32_t) * nh);
    memcpy(c->host_free_stack, a->host_free_stack, sizeof(int32_t) * nh);
    memcpy(c->host_tables, a->host_tables, sizeof(int32_t) * nt);
    memcpy(c->swapped, a->swapped, (size_t)a->max_seqs);
  }
  return c;
}

/* A live sequence whose blocks are on the device (device-side operations
 * refuse a swapped-out sequence). */
static int dev_seq(const oracle_alloc* a, int s) {
  return s >= 0 && s < a->max_seqs && a->active[s] && !a->swapped[s];
}

static void alloc_swap(oracle_alloc* a, oracle_alloc* c) {
  oracle_alloc tmp = *a;
  *a = *c;
  *c = tmp;
}

static int take_block(oracle_alloc* a) {
  int b;
  if (a->free_top == 0) return -1;
  b = a->free_stack[--a->free_top];
  a->refcount[b] = 1;
  return b;
}

static void drop_block(oracle_alloc* a, int b) {
  a->refcount[b] -= 1;
  if (a->refcount[b] == 0) a->free_stack[a->free_top++] = b;
}

int oracle_alloc_seq_add(oracle_alloc* a) {
  int s;
  for (s = 0; s < a->max_seqs; s++) {
    if (!a->active[s]) {
      a->active[s] = 1;
      a->lens[s] = 0;
      return s;
    }
  }
  return -1;
}

/* Appends T tokens to each listed sequence, writing slots[i*T + t] and the
 * copy-on-write (src, dst) pairs.  Returns 0, -1 when out of blocks (state
 * unchanged), -2 for an invalid argument. */
int oracle_alloc_append(oracle_alloc* a, int n, const int32_t* seq_ids, int T, int64_t* slots,
                        int32_t* cow_pairs, int* n_cow) {
  oracle_alloc* w;
  int i, t, ncow = 0;
  for (i = 0; i < n; i++) {
    int k;
    if (!dev_seq(a, seq_ids[i])) return -2;
    for (k = 0; k < i; k++)
      if (seq_ids[k] == seq_ids[i]) return -2;
    if ((a->lens[seq_ids[i]] + T + ORACLE_BLOCK - 1) / ORACLE_BLOCK > a->max_blocks) return -2;
  }
  w = alloc_clone(a); /* work on a copy; keep it only if everything fits */
  for (i = 0; i < n; i++) {
    int s = seq_ids[i];
    int32_t* row = w->tables + (size_t)s * w->max_blocks;
    for (t = 0; t < T; t++) {
      int p = w->lens[s];
      int lb = p / ORACLE_BLOCK;
      if (p % ORACLE_BLOCK == 0) {
        int b = take_block(w);
        if (b < 0) {
          oracle_alloc_destroy(w);
          return -1;
        }
        row[lb] = b;
      } else if (row[lb] < 0) {
        /* the block holding position p was evicted: nothing to append into */
        oracle_alloc_destroy(w);
        return -2;
      } else if (w->refcount[row[lb]] > 1) {
        int old = row[lb];
        int b = take_block(w);
        if (b < 0) {
          oracle_alloc_destroy(w);
          return -1;
        }
        w->refcount[old] -= 1;
        row[lb] = b;
        if (cow_pairs) {
          cow_pairs[2 * ncow] = old;
          cow_pairs[2 * ncow + 1] = b;
        }
        ncow++;
      }
      if (slots) slots[(size_t)i * T + t] = (int64_t)row[lb] * ORACLE_BLOCK + p % ORACLE_BLOCK;
      w->lens[s] = p + 1;
    }
  }
  alloc_swap(a, w);
  oracle_alloc_destroy(w);
  if (n_cow) *n_cow = ncow;
  return 0;
}

int oracle_alloc_fork(oracle_alloc* a, int src) {
  int dst, lb, nblk;
  if (!dev_seq(a, src)) return -2;
  dst = oracle_alloc_seq_add(a);
  if (dst < 0) return -1;
  nblk = (a->lens[src] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  for (lb = 0; lb < nblk; lb++) {
    int b = a->tables[(size_t)src * a->max_blocks + lb];
    a->tables[(size_t)dst * a->max_blocks + lb] = b;
    if (b >= 0) a->refcount[b] += 1;
  }
  a->lens[dst] = a->lens[src];
  return dst;
}

int oracle_alloc_truncate(oracle_alloc* a, int s, int new_len) {
  int lb, keep_blk, nblk;
  if (!dev_seq(a, s) || new_len < 0 || new_len > a->lens[s]) return -2;
  keep_blk = (new_len + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  /* a partial last block must still be present, or later appends would have
   * nowhere to go */
  if (new_len % ORACLE_BLOCK != 0 && a->tables[(size_t)s * a->max_blocks + keep_blk - 1] < 0)
    return -2;
  for (lb = keep_blk; lb < nblk; lb++) {
    int32_t* e = a->tables + (size_t)s * a->max_blocks + lb;
    if (*e >= 0) drop_block(a, *e);
    *e = -1;
  }
  a->lens[s] = new_len;
  return 0;
}

static int take_host_block(oracle_alloc* a) {
  int b;
  if (a->host_free_top == 0) return -1;
  b = a->host_free_stack[--a->host_free_top];
  a->host_refcount[b] = 1;
  return b;
}

static void drop_host_block(oracle_alloc* a, int b) {
  a->host_refcount[b] -= 1;
  if (a->host_refcount[b] == 0) a->host_free_stack[a->host_free_top++] = b;
}

int oracle_alloc_free(oracle_alloc* a, int s) {
  int r;
  if (s >= 0 && s < a->max_seqs && a->active[s] && a->swapped[s]) {
    /* a swapped-out sequence gives back its host blocks, ascending */
    int lb, nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    for (lb = 0; lb < nblk; lb++) {
      int32_t* e = a->host_tables + (size_t)s * a->max_blocks + lb;
      if (*e >= 0) drop_host_block(a, *e);
      *e = -1;
    }
    a->swapped[s] = 0;
    a->lens[s] = 0;
    a->active[s] = 0;
    return 0;
  }
  r = oracle_alloc_truncate(a, s, 0);
  if (r) return r;
  a->active[s] = 0;
  return 0;
}

/* CPU swap ([PA] the block allocator manages the pool in blocks and can swap
 * them out to CPU RAM; [LC] CPU offloading keeps inactive requests' KV in host
 * memory and loads it back when needed).  Readings adopted:
 *  - the host pool holds NH blocks; it starts in ascending order, allocation
 *    takes its front and a released host block goes back to the front;
 *  - swap-out of a list of sequences: every listed sequence's blocks, in list
 *    order and ascending logical order, get host blocks -- a device block that
 *    several listed sequences share is copied once and its host block is
 *    shared as many times; then every device block is released (same
 *    order) and the device table rows become empty;
 *  - swap-in is the mirror image: device blocks from the front of the device
 *    pool (a host block shared by several listed sequences becomes one device
 *    block shared as many times), then the host blocks are released;
 *  - either call changes nothing when the destination pool lacks blocks
 *    (returns -1), and refuses (-2) a sequence that is not live, already in
 *    the requested place, or listed twice;
 *  - a swapped-out sequence keeps its length; every device-side operation
 *    refuses it; freeing it releases its host blocks. */
int oracle_alloc_set_swap_space(oracle_alloc* a, int NH) {
  int i;
  for (i = 0; i < a->max_seqs; i++)
    if (a->swapped[i]) return -2;
  free(a->host_refcount);
  free(a->host_free_stack);
  a->NH = NH;
  a->host_refcount = (int32_t*)calloc((size_t)(NH > 0 ? NH : 1), sizeof(int32_t));
  a->host_free_stack = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NH > 0 ? NH : 1));
  a->host_free_top = 0;
  for (i = NH - 1; i >= 0; i--) a->host_free_stack[a->host_free_top++] = i;
  return 0;
}

/* pairs_out receives (device block, host block) copies (swap-out) or (host
 * block, device block) copies (swap-in); returns the number of pairs. */
static int swap_move(oracle_alloc* a, int n, const int32_t* seq_ids, int out, int32_t* pairs_out) {
  int i, k, lb, npairs = 0, need = 0;
  int32_t* map;
  int src_n = out ? a->NB : a->NH;
  for (i = 0; i < n; i++) {
    int s = seq_ids[i];
    if (s < 0 || s >= a->max_seqs || !a->active[s] || a->swapped[s] != (out ? 0 : 1)) return -2;
    for (k = 0; k < i; k++)
      if (seq_ids[k] == s) return -2;
  }
  map = (int32_t*)malloc(sizeof(int32_t) * (size_t)(src_n > 0 ? src_n : 1));
  for (i = 0; i < src_n; i++) map[i] = -1;
  for (i = 0; i < n; i++) {
    int s = seq_ids[i], nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    const int32_t* row = (out ? a->tables : a->host_tables) + (size_t)s * a->max_blocks;
    for (lb = 0; lb < nblk; lb++)
      if (row[lb] >= 0 && map[row[lb]] < 0) {
        map[row[lb]] = 0;
        need++;
      }
  }
  if (need > (out ? a->host_free_top : a->free_top)) {
    free(map);
    return -1;
  }
  for (i = 0; i < src_n; i++) map[i] = -1;
  for (i = 0; i < n; i++) {
    int s = seq_ids[i], nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int32_t* from = (out ? a->tables : a->host_tables) + (size_t)s * a->max_blocks;
    int32_t* to = (out ? a->host_tables : a->tables) + (size_t)s * a->max_blocks;
    for (lb = 0; lb < nblk; lb++) {
      int b = from[lb];
      if (b < 0) {
        to[lb] = -1;
        continue;
      }
      if (map[b] < 0) {
        map[b] = out ? take_host_block(a) : take_block(a);
        pairs_out[2 * npairs] = b;
        pairs_out[2 * npairs + 1] = map[b];
        npairs++;
      } else if (out) {
        a->host_refcount[map[b]] += 1;
      } else {
        a->refcount[map[b]] += 1;
      }
      to[lb] = map[b];
    }
  }
  for (i = 0; i < n; i++) {
    int s = seq_ids[i], nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int32_t* from = (out ? a->tables : a->host_tables) + (size_t)s * a->max_blocks;
    for (lb = 0; lb < nblk; lb++) {
      if (from[lb] >= 0) {
        if (out)
          drop_block(a, from[lb]);
        else
          drop_host_block(a, from[lb]);
      }
      from[lb] = -1;
    }
    a->swapped[s] = out ? 1 : 0;
  }
  free(map);
  return npairs;
}

int oracle_alloc_swap_out(oracle_alloc* a, int n, const int32_t* seq_ids, int32_t* pairs_out) {
  return swap_move(a, n, seq_ids, 1, pairs_out);
}

int oracle_alloc_swap_in(oracle_alloc* a, int n, const int32_t* seq_ids, int32_t* pairs_out) {
  return swap_move(a, n, seq_ids, 0, pairs_out);
}

int oracle_alloc_swapped(const oracle_alloc* a, int s) { return a->swapped[s]; }
int oracle_alloc_host_refcount(const oracle_alloc* a, int b) { return a->host_refcount[b]; }
int oracle_alloc_num_host_free(const oracle_alloc* a) { return a->host_free_top; }

/* Copies the host table row of a swapped-out sequence (ceil(len/16) entries). */
int oracle_alloc_host_table(const oracle_alloc* a, int s, int32_t* out) {
  int nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK, lb;
  for (lb = 0; lb < nblk; lb++) out[lb] = a->host_tables[(size_t)s * a->max_blocks + lb];
  return nblk;
}

/* Block copies between a device pool and a host pool of the same layout:
 * pairs[2i] -> pairs[2i+1] (K, V and, when present, the scales). */
void oracle_copy_blocks_between(const void* src_k, const void* src_v, const float* src_ks, const float* src_vs,
                                void* dst_k, void* dst_v, float* dst_ks, float* dst_vs, int Hk, int D,
                                int elem_bytes, const int32_t* pairs, int n) {
  size_t blk = (size_t)Hk * ORACLE_BLOCK * D * elem_bytes, sb = (size_t)Hk * ORACLE_BLOCK;
  int i;
  for (i = 0; i < n; i++) {
    size_t s = (size_t)pairs[2 * i], d = (size_t)pairs[2 * i + 1];
    memcpy((char*)dst_k + d * blk, (const char*)src_k + s * blk, blk);
    memcpy((char*)dst_v + d * blk, (const char*)src_v + s * blk, blk);
    if (src_ks && dst_ks) {
      memcpy(dst_ks + d * sb, src_ks + s * sb, sb * sizeof(float));
      memcpy(dst_vs + d * sb, src_vs + s * sb, sb * sizeof(float));
    }
  }
}

int oracle_alloc_evict(oracle_alloc* a, int s, int num_sinks, int window) {
  int L, lb, nblk;
  if (!dev_seq(a, s) || num_sinks < 0 || window < 1) return -2;
  L = a->lens[s];
  if (L <= num_sinks + window) return 0;
  nblk = (L + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  for (lb = 0; lb < nblk; lb++) {
    int32_t* e = a->tables + (size_t)s * a->max_blocks + lb;
    int lo = lb * ORACLE_BLOCK, hi = lo + ORACLE_BLOCK, j, needed = 0;
    if (*e < 0) continue;
    for (j = lo; j < hi && j < L; j++)
      if (oracle_keep(L, MASK_SINK_WINDOW, num_sinks, window, j)) needed = 1;
    if (!needed) {
      drop_block(a, *e);
      *e = -1;
    }
  }
  return 0;
}

/* H2O compaction (the cache keeps only the selected tokens): for each listed
 * sequence, counts[i] fresh blocks' worth of slots are taken from the front
 * of the free pool (all sequences first, in list order, blocks in logical
 * order); then every old block of every listed sequence is released (list
 * order, ascending logical order); the new table is the fresh blocks and the
 * length is counts[i].  new_blocks receives the fresh ids, concatenated.
 * Returns 0, -1 when out of blocks (state unchanged), -2 for invalid input. */
int oracle_alloc_compact(oracle_alloc* a, int n, const int32_t* seq_ids, const int32_t* counts,
                         int32_t* new_blocks) {
  oracle_alloc* w;
  int i, k, total = 0, pos = 0;
  for (i = 0; i < n; i++) {
    if (!dev_seq(a, seq_ids[i])) return -2;
    if (counts[i] < 0 || counts[i] > a->lens[seq_ids[i]]) return -2;
    for (k = 0; k < i; k++)
      if (seq_ids[k] == seq_ids[i]) return -2;
    total += (counts[i] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  }
  if (total > a->free_top) return -1;
  w = alloc_clone(a);
  for (i = 0; i < n; i++) {
    int nb = (counts[i] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    for (k = 0; k < nb; k++) new_blocks[pos++] = take_block(w);
  }
  for (i = 0; i < n; i++) {
    int s = seq_ids[i], lb, nold = (w->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    for (lb = 0; lb < nold; lb++) {
      int32_t* e = w->tables + (size_t)s * w->max_blocks + lb;
      if (*e >= 0) drop_block(w, *e);
      *e = -1;
    }
  }
  pos = 0;
  for (i = 0; i < n; i++) {
    int s = seq_ids[i], nb = (counts[i] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    for (k = 0; k < nb; k++) w->tables[(size_t)s * w->max_blocks + k] = new_blocks[pos++];
    w->lens[s] = counts[i];
  }
  alloc_swap(a, w);
  oracle_alloc_destroy(w);
  return 0;
}

int oracle_alloc_len(const oracle_alloc* a, int s) { return a->lens[s]; }

/* Copies the table row of s (ceil(len/16) entries) into out; returns count. */
int oracle_alloc_table(const oracle_alloc* a, int s, int32_t* out) {
  int nblk = (a->lens[s] + ORACLE_BLOCK - 1) / ORACLE_BLOCK, lb;
  for (lb = 0; lb < nblk; lb++) out[lb] = a->tables[(size_t)s * a->max_blocks + lb];
  return nblk;
}

int oracle_alloc_refcount(const oracle_alloc* a, int b) { return a->refcount[b]; }
int oracle_alloc_num_free(const oracle_alloc* a) { return a->free_top; }

/* Free pool from front to back (for invariant checks). */
int oracle_alloc_free_list(const oracle_alloc* a, int32_t* out) {
  int i;
  for (i = 0; i < a->free_top; i++) out[i] = a->free_stack[a->free_top - 1 - i];
  return a->free_top;
}
