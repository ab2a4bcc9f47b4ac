// KV store: scatter each new token's K and V rows into the cache slot that the
// block manager assigned to it (the slot mapping of the engine's execution
// context; "How lunaryes/nano-vllm works", Connections: Scheduler -> KV Block
// Manager, Model Runner -> Execution Context).
//
// A pure copy, bound by HBM bandwidth: one warp per token, each lane moving
// 16-byte vectors of the K row and then of the V row, so a token row (2 KiB
// for 8 KV heads x 128 dims) is read and written as fully coalesced 512-byte
// warp transactions with several loads in flight per lane.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

static __device__ uint32_t g_kv_store_errors;

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kVecPerLane = 8;  // loads in flight per lane per pass

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    kv_store_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                    const int32_t *__restrict__ slot_mapping, int32_t num_tokens,
                    int32_t row_vec, int64_t num_slots) {
  griddep_wait();  // inputs written by the previous kernel are visible from here on
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t t = warp; t < num_tokens; t += nwarps) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < -1 || slot >= num_slots) {
      if (lane == 0) atomicOr(&g_kv_store_errors, kErrSlot);
      continue;
    }
    const uint4 *ks = k + t * row_vec;
    const uint4 *vs = v + t * row_vec;
    uint4 *kd = k_cache + slot * row_vec;
    uint4 *vd = v_cache + slot * row_vec;
    // K and V rows interleaved: kVecPerLane/2 vectors of each per pass
    for (int base = 0; base < row_vec; base += 32 * (kVecPerLane / 2)) {
      uint4 rk[kVecPerLane / 2], rv[kVecPerLane / 2];
#pragma unroll
      for (int i = 0; i < kVecPerLane / 2; ++i) {
        const int idx = base + i * 32 + lane;
        if (idx < row_vec) {
          rk[i] = ld_stream(ks + idx);
          rv[i] = ld_stream(vs + idx);
        }
      }
#pragma unroll
      for (int i = 0; i < kVecPerLane / 2; ++i) {
        const int idx = base + i * 32 + lane;
        if (idx < row_vec) {
          kd[idx] = rk[i];
          vd[idx] = rv[i];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_store(const KvStoreArgs &a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int64_t blocks_needed = (static_cast<int64_t>(a.num_tokens) + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int grid = static_cast<int>(blocks_needed < 65535 * 8 ? blocks_needed : 65535 * 8);
  return launch_pdl(kv_store_kernel, dim3(grid), dim3(kWarpsPerBlock * 32), 0, stream,
                    static_cast<const uint4 *>(a.k), static_cast<const uint4 *>(a.v),
                    static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache),
                    a.slot_mapping, a.num_tokens, a.row_vec16, a.num_slots);
}

cudaError_t kv_store_error_word(uint32_t **word) {
  return cudaGetSymbolAddress(reinterpret_cast<void **>(word), g_kv_store_errors);
}

cudaError_t take_kv_store_errors(cudaStream_t stream, uint32_t *flags) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_kv_store_errors, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_kv_store_errors, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  *flags |= v;
  return cudaSuccess;
}

}  // namespace pkv
