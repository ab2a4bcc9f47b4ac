// Paged decode attention without a caller-supplied workspace.
//
// The split-K decode call needs scratch memory for its per-split partial
// results. pkv_paged_decode_attn takes that scratch from the caller. Some
// callers cannot allocate device memory where they run: a plugin inside a host
// framework whose allocator owns the whole device pool and refuses foreign
// allocations, a deployment that forbids dynamic allocation after start-up, or
// a latency-critical loop where cudaMalloc/cudaFree may synchronise the device.
// This entry point serves them from a fixed array of static device memory that
// belongs to this file, so it calls no allocator at all.
#include <mutex>

#include "pkv.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = PKV_DECODE_NOALLOC_SCRATCH_BYTES;

// Present on every GPU that loads this library, for the life of the process.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device and process (a later cudaDeviceReset of that device is not supported:
// the address kept here would outlive the context it belongs to). In host code
// the array's name is only a host-side stand-in, so the kernels must be given
// this address, never the name.
pkv_status scratch_for_current_device(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return pkv::cuda_fail(cudaErrorInvalidDevice, "device index");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "cudaGetSymbolAddress (decode scratch)");
    if (p == nullptr)
      return pkv::cuda_fail(cudaErrorInvalidSymbol, "cudaGetSymbolAddress (decode scratch)");
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t max_context_len,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, float scale, int32_t sliding_window, void *out,
    float *lse, void *stream) {
  // the scratch size depends on the device: without a usable one this is a
  // CUDA error (recorded for pkv_last_cuda_error), not an argument error
  int sms = 0;
  pkv_status st = pkv::current_sm_count(&sms);
  if (st != PKV_OK) return st;
  const size_t need =
      pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len);
  if (need == 0) return PKV_ERR_INVALID_ARG;  // sizes no decode call accepts
  if (need > kScratchBytes) return PKV_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != PKV_OK) return st;
  // Nothing in the scratch needs to start at zero: every partial result the
  // call reads back, it writes first.
  return pkv_paged_decode_attn(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                               max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, sliding_window, out, lse, scratch,
                               kScratchBytes, stream);
}
