// The C ABI of libpkv.so (declared in include/pkv.h): argument checks, launch
// planning, TMA descriptor encoding and error reporting around the kernels.
// Allocates nothing; every call only enqueues work on the caller's stream.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "internal.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

}  // namespace

namespace pkv {

pkv_status cuda_fail(cudaError_t e, const char *where) {
  snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%s)", where,
           cudaGetErrorName(e), cudaGetErrorString(e));
  return PKV_ERR_CUDA;
}

}  // namespace pkv

namespace {

using pkv::cuda_fail;

pkv_status cu_fail(CUresult r, const char *where) {
  snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: CUresult %d", where,
           static_cast<int>(r));
  return PKV_ERR_CUDA;
}

// ---------------------------------------------------------------- device facts

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

}  // namespace

namespace pkv {

pkv_status current_sm_count(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    int major = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major < 10) {
      snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
               "device %d has compute capability %d.x; this library is built for sm_103a", dev,
               major);
      return PKV_ERR_CUDA;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  *sms = n;
  return PKV_OK;
}

}  // namespace pkv

namespace {

using pkv::current_sm_count;

// ---------------------------------------------------------------- TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

pkv_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
      g_encode_err = cudaErrorNotSupported;
    if (g_encode_err == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (g_encode == nullptr) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled entry point");
  *fn = g_encode;
  return PKV_OK;
}

// A 3-D bf16 view [rows, heads, dim] (dim innermost, contiguous) with a box of
// box_dim x box_heads x box_rows.
pkv_status encode_rows_map(CUtensorMap *map, const void *base, int64_t rows, int32_t heads,
                           int32_t dim, uint32_t box_dim, uint32_t box_heads, uint32_t box_rows,
                           bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  pkv_status st = get_encoder(&enc);
  if (st != PKV_OK) return st;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(dim) * 2,
                           static_cast<cuuint64_t>(dim) * 2 * static_cast<cuuint64_t>(heads)};
  cuuint32_t box[3] = {box_dim, box_heads, box_rows};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cu_fail(r, "cuTensorMapEncodeTiled");
  return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int32_t> g_pdl{1};

// Tuning overrides of the decode launch (0 = automatic / default).
std::atomic<int32_t> g_decode_ctas{0};
std::atomic<int32_t> g_decode_variant{0};

constexpr float kLog2e = 1.4426950408889634f;

// Sizes shared by the attention calls.
pkv_status check_attention_shape(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t num_blocks, int32_t max_blocks) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int32_t G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  // cache rows are addressed with 32-bit TMA coordinates
  if (num_blocks * static_cast<int64_t>(block_size) > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Decode workspace layout: per-CTA partial (max, sum) [2 grid, HG, G, 2], then
// partial outputs [2 grid, HG, G, D].
struct DecodeWorkspace {
  size_t ml_offset, o_offset, total;
};

int32_t decode_grid_ctas(int sms, int variant) {
  const int32_t o = g_decode_ctas.load(std::memory_order_relaxed);
  return o > 0 ? (o > 65535 ? 65535 : o) : sms * pkv::decode_variant_ctas_per_sm(variant);
}

bool decode_workspace_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int sms, DecodeWorkspace *w) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return false;
  // the largest slots x heads of any launch variant: 2 per CTA, each holding a
  // head group's G query heads
  int64_t slot_heads = 0;
  for (int v = 0; v < pkv::kDecodeNumVariants; ++v) {
    const int64_t sh = 2 * static_cast<int64_t>(decode_grid_ctas(sms, v)) *
                       pkv::decode_group_heads(num_kv_heads, pkv::decode_variant_group_max(v));
    if (sh > slot_heads) slot_heads = sh;
  }
  const int64_t G = num_q_heads / num_kv_heads;
  w->ml_offset = 0;
  w->o_offset =
      align_up(w->ml_offset + static_cast<size_t>(slot_heads * G * 2) * sizeof(float), 256);
  w->total = w->o_offset + static_cast<size_t>(slot_heads * G * head_dim) * sizeof(float);
  return true;
}

}  // namespace

namespace pkv {
bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }
}  // namespace pkv

extern "C" {

void pkv_set_programmatic_launch(int32_t enabled) {
  g_pdl.store(enabled != 0 ? 1 : 0, std::memory_order_relaxed);
}

const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
  }
  return "PKV_ERR_UNKNOWN";
}

const char *pkv_last_cuda_error(void) { return g_last_cuda_error; }

pkv_status pkv_kv_store(const void *k, const void *v, void *k_cache, void *v_cache,
                        const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int64_t num_blocks, void *stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (k_cache == nullptr || v_cache == nullptr) return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && (k == nullptr || v == nullptr || slot_mapping == nullptr))
    return PKV_ERR_INVALID_ARG;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
  if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  pkv::KvStoreArgs a;
  a.k = k;
  a.v = v;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.row_vec16 = static_cast<int32_t>(row_bytes / 16);
  a.num_slots = num_blocks * block_size;
  cudaError_t e = pkv::launch_kv_store(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_store launch");
  return PKV_OK;
}

size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_context_len) {
  (void)max_context_len;  // the layout depends on the grid, not on context length
  int sms = 0;
  if (current_sm_count(&sms) != PKV_OK) return 0;
  DecodeWorkspace w;
  if (!decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, sms, &w)) return 0;
  return w.total;
}

void pkv_decode_set_config(int32_t ctas, int32_t variant) {
  g_decode_ctas.store(ctas < 0 ? 0 : ctas, std::memory_order_relaxed);
  g_decode_variant.store(variant < 0 || variant >= pkv::kDecodeNumVariants ? 0 : variant,
                         std::memory_order_relaxed);
}

}  // extern "C"

namespace {

// Shared by the plain and the fused-store decode entry points; k_new == nullptr
// for the plain one.
pkv_status decode_common(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                         const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, float scale,
                         int32_t sliding_window, void *out, float *lse, void *workspace,
                         size_t workspace_bytes, uint32_t flags, void *stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_tables == nullptr ||
      context_lens == nullptr || out == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs <= 0 || max_context_len <= 0 || !std::isfinite(scale) || sliding_window < 0)
    return PKV_ERR_INVALID_ARG;
  pkv_status st = check_attention_shape(num_q_heads, num_kv_heads, head_dim, block_size,
                                        num_blocks, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  if (num_seqs > pkv::kDecodeMaxSeqs) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
  if (workspace == nullptr) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != PKV_OK) return st;
  DecodeWorkspace w;
  decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, sms, &w);
  if (workspace_bytes < w.total) return PKV_ERR_WORKSPACE_TOO_SMALL;

  pkv::DecodeArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache_w = const_cast<void *>(k_cache);
  a.v_cache_w = const_cast<void *>(v_cache);
  a.slot_mapping = slot_mapping;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.lse = lse;
  a.ws_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + w.ml_offset);
  a.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + w.o_offset);
  a.max_blocks = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = static_cast<int32_t>(num_blocks);
  // variant 0 picks the shape from the head count: groups of 8 KV heads, one
  // CTA per SM, where the heads split into groups of 8; otherwise groups of
  // up to 4 with two CTAs per SM, which keeps more warps streaming per SM
  a.variant = g_decode_variant.load(std::memory_order_relaxed);
  if (a.variant == 0 && pkv::decode_group_heads(num_kv_heads, 8) < 8) a.variant = 2;
  a.grid = decode_grid_ctas(sms, a.variant);
  a.window = sliding_window;
  a.stable_inputs = (flags & PKV_DECODE_STABLE_INPUTS) != 0 && pkv::pdl_enabled();
  a.scale_log2 = scale * kLog2e;

  // one box = 16 token rows of a head group (K, V), the group's q rows, or
  // the group's rows of one new token
  CUtensorMap kmap, vmap, qmap, knmap, vnmap;
  const int64_t rows = num_blocks * block_size;
  const uint32_t G = static_cast<uint32_t>(num_q_heads / num_kv_heads);
  const uint32_t HG = static_cast<uint32_t>(
      pkv::decode_group_heads(num_kv_heads, pkv::decode_variant_group_max(a.variant)));
  if ((st = encode_rows_map(&kmap, k_cache, rows, num_kv_heads, head_dim, 128, HG,
                            pkv::kDecodeChunk, false)) != PKV_OK)
    return st;
  if ((st = encode_rows_map(&vmap, v_cache, rows, num_kv_heads, head_dim, 128, HG,
                            pkv::kDecodeChunk, false)) != PKV_OK)
    return st;
  if ((st = encode_rows_map(&qmap, q, num_seqs, num_q_heads, head_dim, 128, HG * G, 1, false)) !=
      PKV_OK)
    return st;
  if (k_new != nullptr) {
    if ((st = encode_rows_map(&knmap, k_new, num_seqs, num_kv_heads, head_dim, 128, HG, 1,
                              false)) != PKV_OK)
      return st;
    if ((st = encode_rows_map(&vnmap, v_new, num_seqs, num_kv_heads, head_dim, 128, HG, 1,
                              false)) != PKV_OK)
      return st;
  } else {
    knmap = qmap;  // unused without the fused store
    vnmap = qmap;
  }
  cudaError_t e =
      pkv::launch_decode(a, kmap, vmap, qmap, knmap, vnmap, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PKV_OK;
}

}  // namespace

namespace {

// The device error words of the three kernel files on one device.
struct ErrorWords {
  uint32_t *w[3];
};
std::mutex g_words_mutex;
ErrorWords g_words[kMaxDevices];
bool g_words_set[kMaxDevices] = {};

// Addresses of the error words on the current device, looked up once per
// device and process.
pkv_status error_words(ErrorWords *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
  std::lock_guard<std::mutex> lock(g_words_mutex);
  if (!g_words_set[dev]) {
    ErrorWords w;
    if ((e = pkv::kv_store_error_word(&w.w[0])) != cudaSuccess ||
        (e = pkv::decode_error_word(&w.w[1])) != cudaSuccess ||
        (e = pkv::prefill_error_word(&w.w[2])) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress (device error words)");
    g_words[dev] = w;
    g_words_set[dev] = true;
  }
  *out = g_words[dev];
  return PKV_OK;
}

// A one-thread launch in stream order (no programmatic dependent launch: it
// starts after the previous kernel on the stream has completed).
template <typename... KArgs, typename... Args>
cudaError_t launch_one_thread(void (*kernel)(KArgs...), void *stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One thread: *dst = the OR of the three words (dst may be a mapped host word).
__global__ void read_errors_kernel(ErrorWords w, uint32_t *dst) {
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) v |= *reinterpret_cast<volatile uint32_t *>(w.w[i]);
  *reinterpret_cast<volatile uint32_t *>(dst) = v;
}

// One thread: OR `bits` into each of the three words.
__global__ void raise_errors_kernel(ErrorWords w, uint32_t bits) {
#pragma unroll
  for (int i = 0; i < 3; ++i) atomicOr(w.w[i], bits);
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t max_context_len,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                 float scale, int32_t sliding_window, void *out, float *lse,
                                 void *workspace, size_t workspace_bytes, void *stream) {
  return decode_common(nullptr, nullptr, nullptr, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_q_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, scale, sliding_window,
                       out, lse, workspace, workspace_bytes, 0u, stream);
}

pkv_status pkv_paged_decode_attn_store(const void *k_new, const void *v_new,
                                       const int32_t *slot_mapping, const void *q,
                                       void *k_cache, void *v_cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t max_context_len,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int64_t num_blocks, float scale, int32_t sliding_window,
                                       void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, uint32_t flags, void *stream) {
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PKV_ERR_INVALID_ARG;
  if ((flags & ~PKV_DECODE_STABLE_INPUTS) != 0) return PKV_ERR_INVALID_ARG;
  return decode_common(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_q_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, scale, sliding_window,
                       out, lse, workspace, workspace_bytes, flags, stream);
}

size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t max_seqlen_q) {
  (void)num_seqs;
  (void)max_seqlen_q;
  return 0;
}

pkv_status pkv_paged_prefill_attn(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                  int32_t max_seqlen_k, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, float scale, int32_t sliding_window,
                                  void *out, float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (k_cache == nullptr || v_cache == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr || block_tables == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      !std::isfinite(scale) || sliding_window < 0)
    return PKV_ERR_INVALID_ARG;
  if (max_seqlen_q > max_seqlen_k) return PKV_ERR_INVALID_ARG;
  pkv_status st = check_attention_shape(num_q_heads, num_kv_heads, head_dim, block_size,
                                        num_blocks, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  if (total_q > 0 && (q == nullptr || out == nullptr)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != PKV_OK) return st;

  pkv::PrefillArgs a;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.block_tables = block_tables;
  a.out = out;
  a.lse = lse;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = static_cast<int32_t>(num_blocks);
  a.window = sliding_window;
  a.num_sms = sms;
  a.scale_log2 = scale * kLog2e;
  {
    // the kernel indexes its work items with 32-bit integers
    const int32_t G = num_q_heads / num_kv_heads;
    const int64_t rows_per_item = G >= 2 ? 128 : 256;
    const int64_t n_items = (max_seqlen_q + rows_per_item - 1) / rows_per_item *
                            (G >= 2 ? num_q_heads / 2 : num_q_heads) * num_seqs;
    if (n_items > pkv::kMaxPrefillItems) return PKV_ERR_UNSUPPORTED;
  }

  CUtensorMap qmap, kmap, vmap;
  const int64_t rows = num_blocks * block_size;
  if ((st = encode_rows_map(&qmap, q, total_q, num_q_heads, head_dim, 64, 1, 128, true)) != PKV_OK)
    return st;
  a.box_rows = pkv::prefill_box_rows(block_size);
  const uint32_t box = static_cast<uint32_t>(a.box_rows);
  if ((st = encode_rows_map(&kmap, k_cache, rows, num_kv_heads, head_dim, 64, 1, box, true)) != PKV_OK)
    return st;
  if ((st = encode_rows_map(&vmap, v_cache, rows, num_kv_heads, head_dim, 64, 1, box, true)) != PKV_OK)
    return st;
  cudaError_t e = pkv::launch_prefill(a, qmap, kmap, vmap, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return PKV_OK;
}

pkv_status pkv_read_device_errors_async(uint32_t *host_flags, void *stream) {
  if (host_flags == nullptr) return PKV_ERR_INVALID_ARG;
  // only page-locked host memory with a device mapping is written by the
  // kernel; anything else is rejected before a launch
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host_flags);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaPointerGetAttributes (host_flags)");
      (void)cudaGetLastError();  // an argument error: leave no pending runtime error behind
    }
    return PKV_ERR_INVALID_ARG;
  }
  uint32_t *dst = static_cast<uint32_t *>(attr.devicePointer);
  ErrorWords w;
  pkv_status st = error_words(&w);
  if (st != PKV_OK) return st;
  if ((e = launch_one_thread(read_errors_kernel, stream, w, dst)) != cudaSuccess)
    return cuda_fail(e, "error readout launch");
  return PKV_OK;
}

pkv_status pkv_raise_device_errors(uint32_t flags, void *stream) {
  if ((flags & ~(PKV_DEVERR_SLOT | PKV_DEVERR_BLOCK | PKV_DEVERR_CONTEXT | PKV_DEVERR_SEQLENS |
                 PKV_DEVERR_TIMEOUT)) != 0)
    return PKV_ERR_INVALID_ARG;
  ErrorWords w;
  pkv_status st = error_words(&w);
  if (st != PKV_OK) return st;
  if (flags == 0) return PKV_OK;
  const cudaError_t e = launch_one_thread(raise_errors_kernel, stream, w, flags);
  if (e != cudaSuccess) return cuda_fail(e, "error raise launch");
  return PKV_OK;
}

pkv_status pkv_check_device_errors(void *stream, uint32_t *flags_out) {
  if (flags_out == nullptr) return PKV_ERR_INVALID_ARG;
  *flags_out = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if ((e = pkv::take_kv_store_errors(s, flags_out)) != cudaSuccess)
    return cuda_fail(e, "kv_store error word");
  if ((e = pkv::take_decode_errors(s, flags_out)) != cudaSuccess)
    return cuda_fail(e, "decode error word");
  if ((e = pkv::take_prefill_errors(s, flags_out)) != cudaSuccess)
    return cuda_fail(e, "prefill error word");
  return PKV_OK;
}

}  // extern "C"
