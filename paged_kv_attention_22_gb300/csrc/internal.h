// Host-side interface between the C ABI (api.cu) and the kernel translation
// units. Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Record a failed CUDA call as this thread's last error (pkv_last_cuda_error)
// and return PKV_ERR_CUDA.
pkv_status cuda_fail(cudaError_t e, const char *where);

// SM count of the current device (cached per device); PKV_ERR_CUDA, with the
// error recorded, without a usable device or on a GPU older than sm_100.
pkv_status current_sm_count(int *sms);

// Launch with programmatic stream serialization (programmatic dependent
// launch), so a kernel's launch and prologue overlap the previous kernel's
// tail. Process-wide switch, on by default.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

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
// Device address of the kernel file's error word on the current device.
cudaError_t kv_store_error_word(uint32_t **word);

// ---------------------------------------------------------------- decode
constexpr int kDecodeChunk = 16;          // keys per unit (one TMA box of all heads of a group)
constexpr int kDecodeMaxSeqs = 1024;      // sequences per call (chunk prefix lives in smem)
constexpr int kDecodeMaxGroupHeads = 8;   // KV heads per CTA head group

// Launch shapes of the decode kernel (process-wide knob):
//   0  head groups of up to 8 KV heads, 3 TMA stages where they fit, 1 CTA/SM
//   1  head groups of up to 8 KV heads, 2 stages, 1 CTA/SM
//   2  head groups of up to 4 KV heads, 2 stages, 2 CTAs/SM
constexpr int kDecodeNumVariants = 3;
inline int decode_variant_group_max(int variant) { return variant == 2 ? 4 : 8; }
inline int decode_variant_ctas_per_sm(int variant) { return variant == 2 ? 2 : 1; }

// KV heads per CTA head group: the largest divisor of H_kv that is <= group_max.
inline int decode_group_heads(int num_kv_heads, int group_max = kDecodeMaxGroupHeads) {
  for (int d = group_max; d > 1; --d)
    if (num_kv_heads % d == 0) return d;
  return 1;
}

struct DecodeArgs {
  const void *k_new, *v_new;     // fused store: new rows [S, H_kv, D], or null
  void *k_cache_w, *v_cache_w;   // fused store: caches to write
  const int32_t *slot_mapping;   // fused store: slot of each sequence's new token
  const void *q;
  const int32_t *block_tables;
  const int32_t *context_lens;
  void *out;
  float *lse;
  float *ws_o;            // [2 grid, HG, G, D] partial outputs of pieces cut by CTA ranges
  float *ws_ml;           // [2 grid, HG, G, 2] their (max, sum), base 2
  int32_t max_blocks;
  int32_t max_context_len;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t num_blocks;
  int32_t grid;             // CTAs (persistent; one per SM by default)
  int32_t variant;          // launch shape (see kDecodeNumVariants)
  int32_t window;           // sliding window in keys (0: none)
  bool stable_inputs;       // caches, tables and lengths may be read before the wait
  float scale_log2;         // scale * log2(e)
};
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, const CUtensorMap &q_map,
                          const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                          cudaStream_t stream);
cudaError_t take_decode_errors(cudaStream_t stream, uint32_t *flags);
cudaError_t decode_error_word(uint32_t **word);

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
  int32_t window;  // sliding window in keys (0: none)
  int32_t box_rows;  // rows per K/V TMA box: prefill_box_rows(block_size)
  int32_t num_sms;   // SMs of the device (persistent grid)
  float scale_log2;
};
// Work items of one prefill call (row tiles x head pairs x sequences) are
// indexed with 32-bit integers, with headroom for the per-CTA walk.
constexpr int64_t kMaxPrefillItems = (int64_t{1} << 31) - (int64_t{1} << 20);
// Rows per K/V box of the prefill kernel: the largest of 128, 64, 32, 16 that
// divides the block size, so that a box never crosses a cache block and a
// 128-key tile takes as few copies as the block size allows.
inline int32_t prefill_box_rows(int32_t block_size) {
  int32_t r = 128;
  while (block_size % r != 0) r >>= 1;
  return r;
}
cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t stream);
cudaError_t take_prefill_errors(cudaStream_t stream, uint32_t *flags);
cudaError_t prefill_error_word(uint32_t **word);

}  // namespace pkv
