// Host-side interface between the C ABI (api.cu) and the kernel translation
// units. Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// ---------------------------------------------------------------- KV store
struct KvStoreArgs {
  const void *k, *v;
  void *k_cache, *v_cache;
  const int32_t *slot_mapping;
  int32_t num_tokens;
  int32_t row_vec16;      // 16-byte vectors per token row (H_kv * D * 2 / 16)
  int64_t num_slots;      // num_blocks * block_size
};
cudaError_t launch_kv_store(const KvStoreArgs &a, cudaStream_t stream);
cudaError_t take_kv_store_errors(cudaStream_t stream, uint32_t *flags);

// ---------------------------------------------------------------- decode
constexpr int kDecodeChunk = 32;          // keys per chunk (one TMA round per warp)
constexpr int kDecodeMinChunksPerSplit = 2;

struct DecodeArgs {
  const void *q;
  const int32_t *block_tables;
  const int32_t *context_lens;
  void *out;
  float *lse;
  float *ws_o;            // [S, H_q, J, D] per-split normalised partial outputs
  float *ws_lse;          // [S, H_q, J] per-split log2-sum-exp
  int32_t max_blocks;
  int32_t max_context_len;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t num_blocks;
  int32_t chunks_per_split; // keys per split = chunks_per_split * kDecodeChunk
  int32_t num_splits;       // J = ceil(max_context_len / keys per split)
  float scale_log2;         // scale * log2(e)
};
// Plan: how many chunks per split for these sizes on a GPU with num_sms SMs.
int32_t decode_chunks_per_split(const DecodeArgs &a, int num_sms, int32_t override_chunks);
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, cudaStream_t stream);
cudaError_t take_decode_errors(cudaStream_t stream, uint32_t *flags);

// ---------------------------------------------------------------- prefill
struct PrefillArgs {
  const int32_t *cu_seqlens_q, *cu_seqlens_k;
  const int32_t *block_tables;
  void *out;
  float *lse;
  int32_t max_blocks;
  int32_t num_seqs, total_q, max_seqlen_q, max_seqlen_k;
  int32_t num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t num_blocks;
  float scale_log2;
};
cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t stream);
cudaError_t take_prefill_errors(cudaStream_t stream, uint32_t *flags);

}  // namespace pkv
