/*
 * Plain fp64 CPU oracle for paged-KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it. It shares no code, header or constant with the
 * CUDA library; the two meet only through seeded host arrays.
 *
 * What it computes. The pages describe a nano-vLLM style engine whose KV block
 * manager hands out fixed-size cache blocks ("How lunaryes/nano-vllm works",
 * Components: KV Block Manager; Connections: Scheduler -> KV Block Manager
 * "allocates cached blocks"), whose model runner sets an execution context for
 * the layers (same page, Connections: Model Runner -> Execution Context), whose
 * CUDA memory budget holds a "paged KV cache" (nano-vllm-rs README, "GGUF
 * Models") with a configurable block size (same README, "Notes":
 * NANO_VLLM_KVCACHE_BLOCK_SIZE), which supports prefix caching
 * (nano-vllm-sansho README, "Key Features") and decodes with a q=1 attention
 * kernel (same README, "Sansho Serving Roofline Anchors"). The pages never
 * write the attention formula down, so this file is the plain textbook
 * definition that a paged kernel must reproduce:
 *
 *   slot(t)          = block_table[s][pos / bs] * bs + pos % bs
 *   cache[slot(t)]   = k[t], v[t]                       (slot -1: skipped)
 *   z_p              = scale * <q, k_p>                 (keys gathered by table)
 *   M = max_p z_p,   L = sum_p exp(z_p - M)
 *   out              = sum_p exp(z_p - M) v_p / L,      lse = M + ln L
 *
 * with decode attending to every key p < context_len and prefill query i of a
 * segment (Lq new tokens at the end of Lk keys) attending to p <= Lk - Lq + i.
 *
 * Sliding window. The serving target of the nano-vllm-sansho README ("Sansho
 * Fork") is an SWA-256 export: sliding-window attention with a window of 256.
 * The page does not spell the mask out; the reading taken is the plain one: a
 * query at position i attends to the last `window` positions up to itself,
 * keys p with i - window < p <= i (window 0: no window).
 *
 * Readings where the pages are silent (layout [num_blocks, block_size, H_kv,
 * D] row-major; q head h uses KV head h / (H_q / H_kv); -1 marks both a
 * skipped slot and an unused block-table entry; bottom-right causal alignment
 * when a prefix is cached) are the library's documented conventions.
 *
 * Everything is computed in double precision from bf16 inputs that are widened
 * exactly. No blocking, no online softmax, no reordering: one query row at a
 * time, keys in logical order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_BLOCK 2
#define ORACLE_NO_MEMORY 3

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Slot mapping: the cache slot that the block manager assigns to token t of
 * sequence seq_of_token[t] at logical position pos_of_token[t].
 * A position whose block-table entry is -1 has no slot: -1 is written.
 */
int oracle_slot_mapping(const int32_t *block_tables, int32_t max_blocks,
                        int32_t num_seqs, const int32_t *seq_of_token,
                        const int32_t *pos_of_token, int64_t num_tokens,
                        int32_t block_size, int32_t *slot_out) {
  if (block_size <= 0 || max_blocks <= 0) return ORACLE_BAD_ARG;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int32_t s = seq_of_token[t], pos = pos_of_token[t];
    if (s < 0 || s >= num_seqs || pos < 0) return ORACLE_BAD_ARG;
    int32_t logical_block = pos / block_size;
    if (logical_block >= max_blocks) return ORACLE_BAD_ARG;
    int32_t block = block_tables[(int64_t)s * max_blocks + logical_block];
    slot_out[t] = block < 0 ? -1 : block * block_size + pos % block_size;
  }
  return ORACLE_OK;
}

/*
 * KV store: copy token rows into their slots, bit for bit.
 * row_elems = H_kv * D elements per token. Slots of -1 are skipped; any other
 * slot outside [0, num_slots) is rejected before anything is written.
 */
int oracle_kv_store(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                    uint16_t *v_cache, const int32_t *slot_mapping,
                    int64_t num_tokens, int64_t row_elems, int64_t num_slots) {
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < -1 || slot >= num_slots) return ORACLE_BAD_ARG;
  }
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    memcpy(k_cache + slot * row_elems, k + t * row_elems,
           (size_t)row_elems * sizeof(uint16_t));
    memcpy(v_cache + slot * row_elems, v + t * row_elems,
           (size_t)row_elems * sizeof(uint16_t));
  }
  return ORACLE_OK;
}

/* Shape of the cache and of the head grouping, shared by the attention calls. */
typedef struct {
  const uint16_t *k_cache, *v_cache;
  const int32_t *block_tables;
  int32_t max_blocks, block_size;
  int64_t num_blocks;
  int32_t H_q, H_kv, D;
} cache_view;

/* Physical cache row of logical key p of sequence s, or -1 if the table entry
 * is outside the pool. */
static int64_t gather_row(const cache_view *c, int32_t s, int64_t p) {
  int64_t logical_block = p / c->block_size;
  if (logical_block >= c->max_blocks) return -1;
  int64_t block = c->block_tables[(int64_t)s * c->max_blocks + logical_block];
  if (block < 0 || block >= c->num_blocks) return -1;
  return block * c->block_size + p % c->block_size;
}

/* First key a query sees when its keys end at n_keys (the query sits at
 * position n_keys - 1): 0, or the start of its window. */
static int64_t window_start(int64_t n_keys, int32_t window) {
  if (window <= 0 || n_keys <= window) return 0;
  return n_keys - window;
}

/*
 * One query row (query head h of sequence s) against logical keys
 * [first, n_keys). z holds n_keys doubles of scratch (indexed by key). Returns
 * ORACLE_BAD_BLOCK if a needed table entry is outside the pool.
 */
static int attend_row(const cache_view *c, const uint16_t *q_row, int32_t s,
                      int32_t h, int64_t first, int64_t n_keys, double scale, double *z,
                      double *out_row, double *lse_out) {
  const int32_t g = h / (c->H_q / c->H_kv);
  const int32_t D = c->D;
  for (int64_t p = first; p < n_keys; ++p) {
    int64_t row = gather_row(c, s, p);
    if (row < 0) return ORACLE_BAD_BLOCK;
    const uint16_t *k_row = c->k_cache + (row * c->H_kv + g) * D;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d) dot += bf16_to_f64(q_row[d]) * bf16_to_f64(k_row[d]);
    z[p] = scale * dot;
  }
  double M = -INFINITY;
  for (int64_t p = first; p < n_keys; ++p)
    if (z[p] > M) M = z[p];
  double L = 0.0;
  for (int64_t p = first; p < n_keys; ++p) {
    z[p] = exp(z[p] - M); /* z now holds the unnormalised weights */
    L += z[p];
  }
  for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
  for (int64_t p = first; p < n_keys; ++p) {
    int64_t row = gather_row(c, s, p);
    const uint16_t *v_row = c->v_cache + (row * c->H_kv + g) * D;
    for (int32_t d = 0; d < D; ++d) out_row[d] += z[p] * bf16_to_f64(v_row[d]);
  }
  for (int32_t d = 0; d < D; ++d) out_row[d] /= L;
  *lse_out = M + log(L);
  return ORACLE_OK;
}

static int check_heads(int32_t H_q, int32_t H_kv, int32_t D, int32_t bs) {
  if (H_q <= 0 || H_kv <= 0 || D <= 0 || bs <= 0) return 0;
  return H_q % H_kv == 0;
}

/*
 * Decode: one query token per sequence, attending to every cached key
 * p < context_lens[s] (the query's own K/V are already stored at p = ctx - 1),
 * or to the last `window` of them.
 * q [S, H_q, D] bf16; out [S, H_q, D] f64; lse [S, H_q] f64.
 */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache,
                  const uint16_t *v_cache, const int32_t *block_tables,
                  int32_t max_blocks, const int32_t *context_lens,
                  int32_t num_seqs, int32_t H_q, int32_t H_kv, int32_t D,
                  int32_t block_size, int64_t num_blocks, double scale,
                  int32_t window, double *out, double *lse) {
  if (!check_heads(H_q, H_kv, D, block_size) || window < 0) return ORACLE_BAD_ARG;
  int64_t max_ctx = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (context_lens[s] <= 0) return ORACLE_BAD_ARG;
    if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
  }
  cache_view c = {k_cache, v_cache, block_tables, max_blocks, block_size,
                  num_blocks, H_q, H_kv, D};
  int status = ORACLE_OK;
  const int64_t rows = (int64_t)num_seqs * H_q;
#pragma omp parallel
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!z) {
#pragma omp critical
      status = ORACLE_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
      if (!z) continue;
      int32_t s = (int32_t)(r / H_q), h = (int32_t)(r % H_q);
      int rc = attend_row(&c, q + r * D, s, h, window_start(context_lens[s], window),
                          context_lens[s], scale, z, out + r * D, lse + r);
      if (rc != ORACLE_OK) {
#pragma omp critical
        status = rc;
      }
    }
    free(z);
  }
  return status;
}

/*
 * Prefill over a paged cache. Segment s owns query tokens
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) and keys [0, Lk) with
 * Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s]; its Lq queries are the last Lq
 * positions of the Lk, so query i attends to keys p <= Lk - Lq + i (with a
 * window, only the last `window` of those). Keys are always read from the
 * cache (the caller stored them first).
 * q [T_q, H_q, D] bf16; out [T_q, H_q, D] f64; lse [T_q, H_q] f64.
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *cu_seqlens_q,
                   const int32_t *cu_seqlens_k, const int32_t *block_tables,
                   int32_t max_blocks, int32_t num_seqs, int32_t H_q,
                   int32_t H_kv, int32_t D, int32_t block_size,
                   int64_t num_blocks, double scale, int32_t window, double *out,
                   double *lse) {
  if (!check_heads(H_q, H_kv, D, block_size) || window < 0) return ORACLE_BAD_ARG;
  int64_t max_k = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t Lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    int64_t Lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
    if (Lq < 0 || Lk < Lq) return ORACLE_BAD_ARG;
    if (Lk > max_k) max_k = Lk;
  }
  cache_view c = {k_cache, v_cache, block_tables, max_blocks, block_size,
                  num_blocks, H_q, H_kv, D};
  const int64_t total_q = cu_seqlens_q[num_seqs] - cu_seqlens_q[0];
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)(max_k > 0 ? max_k : 1));
    if (!z) {
#pragma omp critical
      status = ORACLE_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < total_q * H_q; ++r) {
      if (!z) continue;
      int64_t t = cu_seqlens_q[0] + r / H_q; /* global query token */
      int32_t h = (int32_t)(r % H_q);
      int32_t s = 0;
      while (t >= cu_seqlens_q[s + 1]) ++s;
      int64_t Lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
      int64_t Lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
      int64_t i = t - cu_seqlens_q[s];
      int64_t n_keys = Lk - Lq + i + 1;
      int rc = attend_row(&c, q + (t * H_q + h) * D, s, h, window_start(n_keys, window),
                          n_keys, scale, z, out + (t * H_q + h) * D, lse + t * H_q + h);
      if (rc != ORACLE_OK) {
#pragma omp critical
        status = rc;
      }
    }
    free(z);
  }
  return status;
}

/*
 * Sampled rows, for checks at full size: attention of the listed
 * (sequence, query head, number of keys) rows, where row r reads query
 * q_rows[r] (D bf16 values) and sees keys [0, n_keys[r]), or their last
 * `window`. Used to check a few outputs of very large calls one by one.
 */
int oracle_attend_rows(const uint16_t *q_rows, const int32_t *seq_ids,
                       const int32_t *head_ids, const int64_t *n_keys,
                       int64_t num_rows, const uint16_t *k_cache,
                       const uint16_t *v_cache, const int32_t *block_tables,
                       int32_t max_blocks, int32_t H_q, int32_t H_kv, int32_t D,
                       int32_t block_size, int64_t num_blocks, double scale,
                       int32_t window, double *out, double *lse) {
  if (!check_heads(H_q, H_kv, D, block_size) || window < 0) return ORACLE_BAD_ARG;
  int64_t max_k = 1;
  for (int64_t r = 0; r < num_rows; ++r) {
    if (n_keys[r] <= 0) return ORACLE_BAD_ARG;
    if (n_keys[r] > max_k) max_k = n_keys[r];
  }
  cache_view c = {k_cache, v_cache, block_tables, max_blocks, block_size,
                  num_blocks, H_q, H_kv, D};
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)max_k);
    if (!z) {
#pragma omp critical
      status = ORACLE_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < num_rows; ++r) {
      if (!z) continue;
      int rc = attend_row(&c, q_rows + r * D, seq_ids[r], head_ids[r],
                          window_start(n_keys[r], window), n_keys[r], scale, z,
                          out + r * D, lse + r);
      if (rc != ORACLE_OK) {
#pragma omp critical
        status = rc;
      }
    }
    free(z);
  }
  return status;
}
