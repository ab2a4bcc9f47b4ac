/*
 * pkv.h -- paged-KV-cache attention for GB300 (sm_103a): the C ABI of libpkv.so.
 *
 * The pages describe a nano-vLLM style serving engine whose scheduler asks a
 * KV block manager for cache blocks ("How lunaryes/nano-vllm works",
 * Connections: "Scheduler -> KV Block Manager: allocates cached blocks") and
 * whose model runner sets an execution context before running the Qwen3
 * layers (same page, Connections: "Model Runner -> Execution Context"). This
 * library is the data-parallel hot path inside those layers: writing each
 * step's new K/V rows into the paged cache (the "paged KV cache" of the
 * nano-vllm-rs README, "GGUF Models"), q=1 decode attention (the q=1 decode
 * kernel of the nano-vllm-sansho README, "Sansho Serving Roofline Anchors") and
 * varlen causal prefill attention that also serves prompts whose leading blocks
 * are already cached (prefix caching: nano-vllm-sansho README, "Key Features").
 * Its arguments are that execution context: slot mapping, block tables,
 * context lengths, cumulative sequence lengths.
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout. bf16 everywhere for tensors; row-major, contiguous.
 *   new K/V rows   k, v        [T, H_kv, D]
 *   cache          k_cache     [num_blocks, block_size, H_kv, D]  (same for v_cache)
 *   queries        q           [T_q, H_q, D] (prefill) or [S, H_q, D] (decode)
 *   outputs        out         like q; lse float32 [rows, H_q]
 *   block tables   int32       [S, max_blocks_per_seq]; entry -1 = no block
 * Slot of token at position p of sequence s:
 *   block_tables[s][p / block_size] * block_size + p % block_size.
 * Query head h reads KV head h / (H_q / H_kv).
 * D must be 128, block_size a multiple of 16, H_q / H_kv in {1, 2, 4}.
 *
 * Memory and ownership. Every pointer is caller-owned device memory (except
 * the host pointer flags_out); the library allocates and frees nothing, keeps
 * no per-call state, and returns before the kernels finish. Device buffers
 * must be 16-byte aligned.
 *
 * Streams. `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream). Every call only enqueues work on that stream and never
 * synchronises, so it may be captured into a CUDA graph, except
 * pkv_check_device_errors, which synchronises the stream.
 *
 * Errors. Arguments the host can see are checked before anything is enqueued:
 * PKV_ERR_INVALID_ARG (null pointer, negative size, inconsistent shape),
 * PKV_ERR_UNSUPPORTED (a shape this library has no kernel for),
 * PKV_ERR_WORKSPACE_TOO_SMALL. A failing CUDA call gives PKV_ERR_CUDA and
 * pkv_last_cuda_error() names it (thread-local). Values that live on the device
 * (slots, table entries, lengths) are checked by the kernels: an invalid one
 * skips the access it would have made and raises a bit of the device error
 * word (PKV_DEVERR_*), read with pkv_check_device_errors (which blocks) or
 * pkv_read_device_errors_async (which does not). Outputs that depend on an
 * invalid value are undefined; nothing outside the given buffers is touched.
 *
 * Timeouts are sticky. Every wait inside a kernel is bounded; a kernel that
 * gives up raises PKV_DEVERR_TIMEOUT. From then on every later decode call
 * (fused store included) and prefill call on that device returns PKV_OK but
 * skips all its work, leaving its outputs (and, for the fused call, the cache)
 * untouched, until the word is cleared by pkv_check_device_errors. An engine
 * that runs these calls inside CUDA graphs and never synchronises should
 * append pkv_read_device_errors_async to its step and act on the bit.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,
  PKV_ERR_UNSUPPORTED = 2,
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,
  PKV_ERR_CUDA = 4,
  PKV_ERR_OUT_OF_BLOCKS = 5 /* the block manager has too few free blocks (pkv_blocks.h) */
} pkv_status;

/* Bits of the device error word. */
#define PKV_DEVERR_SLOT 0x1u      /* a slot outside [-1, num_blocks * block_size)      */
#define PKV_DEVERR_BLOCK 0x2u     /* a needed block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT 0x4u   /* context_len <= 0, above max_context_len or above
                                     max_blocks_per_seq * block_size                  */
#define PKV_DEVERR_SEQLENS 0x8u   /* cu_seqlens inconsistent with the host-side maxima  */
#define PKV_DEVERR_TIMEOUT 0x10u  /* a kernel gave up waiting on one of its barriers    */

/*
 * Launch mode, process-wide: with enabled != 0 (the default) every kernel is
 * launched with programmatic stream serialization (programmatic dependent
 * launch), so it may start while the previous kernel on the stream finishes;
 * each kernel still waits for that kernel's completion before it reads or
 * writes global memory, so results and ordering are unchanged. 0 launches
 * them the classic way.
 */
void pkv_set_programmatic_launch(int32_t enabled);

/* Name of a status code (static string). */
const char *pkv_status_string(pkv_status status);

/* The CUDA error string of this thread's last PKV_ERR_CUDA, or "" if none. */
const char *pkv_last_cuda_error(void);

/*
 * KV store: the slot-mapping scatter of the new tokens' K/V rows into the
 * paged cache (the engine's KV block manager hands out the cache slots: "How
 * lunaryes/nano-vllm works", Components: KV Block Manager, and Connections:
 * "Scheduler -> KV Block Manager: allocates cached blocks"; the cache is the
 * paged KV cache of the nano-vllm-rs README, "GGUF Models").
 * k_cache[slot_mapping[t]] = k[t] and v_cache[slot_mapping[t]] = v[t]
 * for every t with slot_mapping[t] >= 0 (all H_kv * D values of the row, bit
 * for bit); -1 skips the token (the block manager gave it no slot, as for
 * tokens of a cached prefix). Two tokens with the same non-negative slot in one
 * call race. A slot below -1 or at/above num_blocks * block_size is skipped
 * and raises PKV_DEVERR_SLOT.
 *   k, v           device bf16 [num_tokens, num_kv_heads, head_dim]
 *   k_cache,v_cache device bf16 [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping   device int32 [num_tokens]
 * num_tokens == 0 is a no-op. Here head_dim may be any value with
 * num_kv_heads * head_dim * 2 a multiple of 16 bytes.
 */
pkv_status pkv_kv_store(const void *k, const void *v, void *k_cache, void *v_cache,
                        const int32_t *slot_mapping, int32_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int64_t num_blocks, void *stream);

/*
 * Bytes of device workspace that pkv_paged_decode_attn needs for these sizes on
 * the current device (0 on invalid sizes or without a device). The workspace
 * holds the partial results of the (sequence, KV head) pairs whose keys are
 * split between CTAs; its size depends on the heads and on the device's SM
 * count, not on context length or on the number of sequences. The caller
 * allocates it once and may reuse it for every call with sizes no larger than
 * these; it needs no initialisation. Calls that share a workspace must be
 * ordered (same stream).
 */
size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_context_len);

/*
 * Paged decode attention, one query token per sequence (q=1 decode).
 * For sequence s, query head h and KV head g = h / (H_q / H_kv):
 *   z_p   = scale * <q[s,h], k_cache[slot(s, p), g]>   for p < context_lens[s]
 *   out   = sum_p exp(z_p - M) v_cache[slot(s,p), g] / sum_p exp(z_p - M)
 *   lse   = M + ln sum_p exp(z_p - M),   M = max_p z_p      (natural log)
 * The query's own K/V must already be in the cache (store first, then attend,
 * on the same stream). Split-K over the context ("flash decoding"): partial
 * results go to the workspace and a second kernel merges them.
 *   q              device bf16 [num_seqs, num_q_heads, head_dim]
 *   block_tables   device int32 [num_seqs, max_blocks_per_seq]
 *   context_lens   device int32 [num_seqs], each in [1, max_context_len]
 *   max_context_len host int: an upper bound of context_lens (sizes the grid)
 *   scale          the logit scale (usually 1/sqrt(head_dim))
 *   sliding_window 0: every key; W > 0: only the last W keys up to the
 *                  query's own, p >= context_lens[s] - W (sliding-window
 *                  attention: the SWA-256 serving target of the
 *                  nano-vllm-sansho README, "Sansho Fork"); blocks wholly
 *                  before the window are not read. Negative: PKV_ERR_INVALID_ARG.
 *   out            device bf16 [num_seqs, num_q_heads, head_dim]
 *   lse            device float32 [num_seqs, num_q_heads], or NULL
 *   workspace      device, >= pkv_decode_workspace_size(...) bytes, 16-byte aligned
 * num_seqs is at most 1024.
 * Rows whose context_len is invalid raise PKV_DEVERR_CONTEXT and are not written.
 */
pkv_status pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t max_context_len,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                 float scale, int32_t sliding_window, void *out, float *lse,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Fused decode step: the KV store of each sequence's new token and paged decode
 * attention in one kernel (the engine's per-layer decode work, one launch).
 * Equivalent to pkv_kv_store(k_new, v_new, k_cache, v_cache, slot_mapping,
 * num_seqs, ...) followed by pkv_paged_decode_attn(...) on the same stream:
 * the new token of sequence s is the one at logical position
 * context_lens[s] - 1, its K/V rows k_new[s], v_new[s] are written to
 * slot_mapping[s] (-1: not written) and used as that key by the attention.
 *   k_new, v_new   device bf16 [num_seqs, num_kv_heads, head_dim]
 *   slot_mapping   device int32 [num_seqs]
 * Other arguments, the workspace and the error behaviour are those of
 * pkv_paged_decode_attn; an invalid slot raises PKV_DEVERR_SLOT (not written;
 * the attention still uses the new rows).
 *   flags          0, or PKV_DECODE_STABLE_INPUTS: the caller guarantees that
 *                  k_cache and v_cache (except the rows this call stores),
 *                  block_tables and context_lens are written neither by the
 *                  kernel enqueued just before this call nor by any earlier one
 *                  that may still be running (with programmatic dependent
 *                  launch a kernel of this library lets the next one start
 *                  before it ends). The call then reads them, and starts
 *                  streaming K/V, while the previous kernel finishes; q,
 *                  k_new, v_new and slot_mapping are still read only after it
 *                  has completed. This holds in a decode step whose tables and
 *                  lengths are set before the step and whose layers each have
 *                  their own caches.
 */
#define PKV_DECODE_STABLE_INPUTS 0x1u
pkv_status pkv_paged_decode_attn_store(const void *k_new, const void *v_new,
                                       const int32_t *slot_mapping, const void *q,
                                       void *k_cache, void *v_cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t max_context_len,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int64_t num_blocks, float scale, int32_t sliding_window,
                                       void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * Tuning knob of the decode launch, process-wide (not thread-safe against
 * concurrent launches): ctas = number of persistent CTAs (0 = one per SM, the
 * default); variant = launch shape (0 = default: head groups of 8 KV heads and
 * three TMA stages per CTA when the KV heads split into groups of 8, else the
 * shape of variant 2; 1 = head groups of up to 8 KV heads, two stages; 2 =
 * head groups of up to 4 KV heads, two stages, two CTAs per SM). Results do
 * not depend on either, beyond rounding.
 * A non-default ctas changes pkv_decode_workspace_size.
 */
void pkv_decode_set_config(int32_t ctas, int32_t variant);

/*
 * Decode attention for callers that cannot allocate device memory.
 * (An addition of this library: the pages have no counterpart.)
 * Some callers of decode cannot call cudaMalloc where they run: a plugin inside
 * a host framework whose allocator owns the whole device pool, a deployment
 * that forbids dynamic allocation after start-up, a latency-critical loop where
 * an allocation may synchronise the device. This call computes exactly what
 * pkv_paged_decode_attn computes, with the same arguments except the
 * workspace: its scratch is a static device array of
 * PKV_DECODE_NOALLOC_SCRATCH_BYTES inside libpkv.so, present on every GPU that
 * loads the library until the process exits. It calls no cudaMalloc, cudaFree
 * or other allocator.
 *   - Sizes whose pkv_decode_workspace_size exceeds that limit are rejected with
 *     PKV_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is kept for the life of the
 *     process: a cudaDeviceReset of that device afterwards is not supported.
 *   - Without a usable device the call returns PKV_ERR_CUDA (with
 *     pkv_last_cuda_error set); sizes that no decode call accepts return
 *     PKV_ERR_INVALID_ARG.
 *   - Every call on a device shares that device's one array, which keeps the
 *     last call's contents; nothing in it needs to start at zero. Calls that
 *     can overlap on the GPU (for example on two streams with no ordering
 *     between them) race on the array: the caller must order them.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
pkv_status pkv_paged_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables,
                                         int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t max_context_len,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int64_t num_blocks, float scale,
                                         int32_t sliding_window, void *out, float *lse,
                                         void *stream);

/*
 * Bytes of device workspace that pkv_paged_prefill_attn needs (currently 0 for
 * every size: the prefill kernel keeps all its state on chip).
 */
size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t max_seqlen_q);

/*
 * Varlen causal prefill attention over the paged cache, with prefix caching
 * (nano-vllm-sansho README, "Key Features": prefix caching; "How
 * lunaryes/nano-vllm works", Connections: the block manager allocates cached
 * blocks, which a later prompt with the same leading tokens reads instead of
 * recomputing them).
 * Segment s has Lq = cu_seqlens_q[s+1] - cu_seqlens_q[s] query tokens
 * (rows cu_seqlens_q[s] .. of q) and Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s]
 * keys, read through block_tables[s]; the queries are the last Lq of the Lk
 * positions, so query i sees keys p <= Lk - Lq + i (bottom-right causal;
 * Lq == Lk is plain causal attention, Lq < Lk serves a prompt whose first
 * Lk - Lq tokens are cached). Keys are always read from the cache: store the
 * prompt's new K/V first, on the same stream. Lq == 0 writes nothing.
 * Output and lse as in decode, for every query row. With sliding_window
 * W > 0 query i sees only keys Lk - Lq + i - W < p <= Lk - Lq + i (the last W
 * positions up to its own); KV tiles wholly before a CTA's windows are not
 * read. Negative: PKV_ERR_INVALID_ARG.
 *   q              device bf16 [total_q, num_q_heads, head_dim]
 *   cu_seqlens_q/k device int32 [num_seqs + 1], non-decreasing, from 0
 *   max_seqlen_q/k host ints: upper bounds of Lq and Lk (size the grid)
 *   out            device bf16 [total_q, num_q_heads, head_dim]
 *   lse            device float32 [total_q, num_q_heads], or NULL
 *   workspace      may be NULL when pkv_prefill_workspace_size returns 0
 * Segments with Lq > Lk, Lq > max_seqlen_q, Lk > max_seqlen_k or Lk beyond
 * the table raise PKV_DEVERR_SEQLENS and are not written.
 */
pkv_status pkv_paged_prefill_attn(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                  int32_t max_seqlen_k, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, float scale, int32_t sliding_window,
                                  void *out, float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Synchronise `stream`, then return in *flags_out the OR of the device error
 * words of every kernel of this library on the current device, and clear
 * them. It blocks the host; it is also the only way to clear the words, and
 * so to end the skip that a PKV_DEVERR_TIMEOUT starts.
 */
pkv_status pkv_check_device_errors(void *stream, uint32_t *flags_out);

/*
 * Non-blocking readout of the device error words: enqueues on `stream` a
 * one-thread kernel that writes the OR of the error words of every kernel of
 * this library on the current device into *host_flags, in stream order after
 * the work enqueued before it. The words are not cleared. host_flags must be
 * page-locked host memory (cudaHostAlloc, cudaMallocHost or cudaHostRegister)
 * that the device can write; other memory gives PKV_ERR_INVALID_ARG. The value
 * is there once that kernel has completed (for example after an event
 * recorded behind it). Capturable; make the first call on a device (which
 * looks up the words' addresses) before any stream capture.
 */
pkv_status pkv_read_device_errors_async(uint32_t *host_flags, void *stream);

/*
 * Raise bits of the device error words from the host, in stream order, as a
 * kernel that met the condition would. For tests of an engine's error
 * handling, for instance of the skip that follows PKV_DEVERR_TIMEOUT, without
 * making any kernel wait or fault. Bits outside PKV_DEVERR_* give
 * PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_raise_device_errors(uint32_t flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
