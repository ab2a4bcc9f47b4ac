// Varlen causal prefill attention over the paged KV cache, on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Serves both plain prompts (Lq == Lk) and prompts whose leading blocks are
// already cached (prefix caching: "nano-vllm-sansho" README, "Key Features";
// "How lunaryes/nano-vllm works", where the block manager hands out cached
// blocks). Query i of a segment sees keys p <= Lk - Lq + i.
//
// One CTA per (128-query tile, query head, sequence); 6 warps:
//   warp 4  TMA producer: the Q tile once, then K and V tiles of 128 keys as
//           eight 16-row boxes each (a box never crosses a cache block), two
//           stages deep, 128-byte swizzled.
//   warp 5  MMA issuer: S = Q K^T into TMEM (128 lanes x 128 fp32 columns),
//           then O += P V into a second TMEM region; completion is signalled
//           through tcgen05.commit on mbarriers. Before the P.V of the tile
//           that holds the segment's last key it zeroes the V rows past it,
//           so that stale or poisoned rows never meet a zero probability.
//   warps 0-3  one query row per thread (TMEM lane = row): read the S row,
//           mask, online softmax in base 2, rescale the O row in TMEM when the
//           running max moves, write P (bf16) to shared memory in the swizzled
//           K-major layout the MMA reads, and finally normalise O and store
//           the bf16 output and the natural-log lse.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

static __device__ uint32_t g_prefill_errors;

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                       // query rows per CTA
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kBoxRows = 16;                   // rows per K/V TMA box
constexpr int kHalfBytes = 128 * 128;          // 128 rows x 64 bf16 (one swizzle column group)
constexpr int kTileBytes = 2 * kHalfBytes;     // 128 rows x 128 bf16
constexpr int kStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTileBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
constexpr int kPOff = kVOff + kStages * kTileBytes;
constexpr int kBarOff = kPOff + kTileBytes;
// barrier slots (8 bytes each)
constexpr int kBarQ = 0, kBarKFull = 1, kBarVFull = 3, kBarKvEmpty = 5, kBarS = 7, kBarP = 8,
              kBarO = 9, kNumBars = 10;
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kAbortOff = kTmemSlotOff + 8;
constexpr int kSmemBytes = kAbortOff + 8 + 1024;  // + slack for 1024-byte alignment
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;            // S: columns 0-127, O: 128-255
constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);  // A=Q K-major, B=K K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, 0, 1);   // A=P K-major, B=V MN-major
constexpr float kLn2 = 0.693147180559945309f;

struct PrefillParams {
  const int32_t *cu_q, *cu_k, *block_tables;
  __nv_bfloat16 *out;
  float *lse;
  int32_t max_blocks, num_seqs, total_q, max_seqlen_q, max_seqlen_k;
  int32_t num_q_heads, num_kv_heads, block_size, num_blocks, n_qtiles;
  float scale_log2;
};

__device__ __forceinline__ bool wait_(uint32_t bar, uint32_t parity, const volatile int *abort) {
  return mbar_wait(bar, parity, &g_prefill_errors, abort);
}

__device__ __forceinline__ void fail(volatile int *abort) {
  *abort = 1;
  atomicOr(&g_prefill_errors, kErrTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
  const int h = blockIdx.y, s = blockIdx.z;
  const int g = h / (p.num_q_heads / p.num_kv_heads);

  // a CTA gave up waiting (in this or an earlier launch): skip the work until
  // the error word is read and cleared; decided once per CTA
  if (__syncthreads_or(tid == 0 &&
                       (*reinterpret_cast<volatile uint32_t *>(&g_prefill_errors) & kErrTimeout)))
    return;

  const int q0 = p.cu_q[s], q1 = p.cu_q[s + 1];
  const int Lq = q1 - q0, Lk = p.cu_k[s + 1] - p.cu_k[s];
  if (q0 < 0 || Lq < 0 || Lk < Lq || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k ||
      q1 > p.total_q ||
      static_cast<int64_t>(Lk) > static_cast<int64_t>(p.max_blocks) * p.block_size) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) atomicOr(&g_prefill_errors, kErrSeqlens);
    return;
  }
  const int row0 = t * kBM;
  if (row0 >= Lq) return;
  const int diag = Lk - Lq;                        // query i sees keys <= diag + i
  const int last_row = min(Lq, row0 + kBM) - 1;
  const int kv_end = diag + last_row + 1;          // keys this tile needs (<= Lk)
  const int n_tiles = (kv_end + kBN - 1) / kBN;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kQOff, sK = sbase + kKOff, sV = sbase + kVOff, sP = sbase + kPOff;
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile int *abort = reinterpret_cast<volatile int *>(smem + kAbortOff);

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarP), kBM);
    mbar_init(bar(kBarO), 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(sbase + kTmemSlotOff, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kTmemSlotOff);
  const uint32_t tS = tmem, tO = tmem + kBN;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      mbar_arrive_expect_tx(bar(kBarQ), kTileBytes);
      tma_load_3d(sQ, &q_map, bar(kBarQ), 0, h, q0 + row0);
      tma_load_3d(sQ + kHalfBytes, &q_map, bar(kBarQ), 64, h, q0 + row0);
      const int64_t table = static_cast<int64_t>(s) * p.max_blocks;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        if (j >= kStages && !wait_(bar(kBarKvEmpty + st), ((j >> 1) - 1) & 1, abort)) {
          fail(abort);
          break;
        }
        int32_t rows[kBN / kBoxRows];
        uint32_t nbox = 0;
#pragma unroll
        for (int b = 0; b < kBN / kBoxRows; ++b) {
          rows[b] = -1;
          const int key = j * kBN + b * kBoxRows;
          if (key < Lk) {
            const int32_t blk = p.block_tables[table + key / p.block_size];
            if (blk < 0 || blk >= p.num_blocks) {
              atomicOr(&g_prefill_errors, kErrBlock);
            } else {
              rows[b] = blk * p.block_size + key % p.block_size;
              ++nbox;
            }
          }
        }
        const uint32_t bytes = nbox * 2u * kBoxRows * 128u;
        const uint32_t kdst = sK + st * kTileBytes, vdst = sV + st * kTileBytes;
        mbar_arrive_expect_tx(bar(kBarKFull + st), bytes);
#pragma unroll
        for (int b = 0; b < kBN / kBoxRows; ++b) {
          if (rows[b] < 0) continue;
          tma_load_3d(kdst + b * kBoxRows * 128, &k_map, bar(kBarKFull + st), 0, g, rows[b]);
          tma_load_3d(kdst + kHalfBytes + b * kBoxRows * 128, &k_map, bar(kBarKFull + st), 64, g,
                      rows[b]);
        }
        mbar_arrive_expect_tx(bar(kBarVFull + st), bytes);
#pragma unroll
        for (int b = 0; b < kBN / kBoxRows; ++b) {
          if (rows[b] < 0) continue;
          tma_load_3d(vdst + b * kBoxRows * 128, &v_map, bar(kBarVFull + st), 0, g, rows[b]);
          tma_load_3d(vdst + kHalfBytes + b * kBoxRows * 128, &v_map, bar(kBarVFull + st), 64, g,
                      rows[b]);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    bool good = __all_sync(0xffffffffu, wait_(bar(kBarQ), 0, abort));
    auto issue_s = [&](int j) -> bool {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, wait_(bar(kBarKFull + st), (j >> 1) & 1, abort)))
        return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_bf16_ss(tS, smem_desc_sw128(sQ + off, 16, 1024),
                      smem_desc_sw128(sK + st * kTileBytes + off, 16, 1024), kIdescQK, kk > 0);
        }
        mma_commit(bar(kBarS));
      }
      __syncwarp();
      return true;
    };
    auto issue_pv = [&](int j) -> bool {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, wait_(bar(kBarVFull + st), (j >> 1) & 1, abort)))
        return false;
      const int r0 = Lk - j * kBN;  // V rows >= r0 are past the segment's last key
      if (r0 < kBN) {
        const uint32_t vbase = sV + st * kTileBytes;
        const int n16 = (kBN - r0) * 16;  // 16-byte pieces over both column halves
        for (int idx = lane; idx < n16; idx += 32) {
          const int row = r0 + idx / 16, piece = idx % 16;
          const uint32_t addr = vbase + (piece / 8) * kHalfBytes + row * 128 + (piece % 8) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(0u), "r"(0u), "r"(0u),
                       "r"(0u)
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_bf16_ss(tO, smem_desc_sw128(sP + poff, 16, 1024),
                      smem_desc_sw128(sV + st * kTileBytes + kk * 16 * 128, kHalfBytes, 1024),
                      kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarO));
        mma_commit(bar(kBarKvEmpty + st));
      }
      __syncwarp();
      return true;
    };
    if (good) good = issue_s(0);
    for (int j = 1; good && j < n_tiles; ++j) {
      good = __all_sync(0xffffffffu, wait_(bar(kBarP), (j - 1) & 1, abort)) &&
             issue_s(j) && issue_pv(j - 1);
    }
    if (good)
      good = __all_sync(0xffffffffu, wait_(bar(kBarP), (n_tiles - 1) & 1, abort)) &&
             issue_pv(n_tiles - 1);
    if (!good && lane == 0) fail(abort);
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int r = tid;                      // row within the tile == TMEM lane
    const int qi = row0 + r;                // query index within the segment
    const int lim = diag + qi;              // last key this row may see
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool good = true;
    uint32_t x[kBN];
    for (int j = 0; j < n_tiles; ++j) {
      if (!__all_sync(0xffffffffu, wait_(bar(kBarS), j & 1, abort))) {
        good = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        tmem_ld32(tS + lane_off + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
      tmem_wait_ld();
      const int kbase = j * kBN;
      const bool need_mask = (kbase + kBN - 1 > diag + row0) || (kbase + kBN > Lk);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        float v = __uint_as_float(x[c]) * p.scale_log2;
        if (need_mask && (kbase + c > lim || kbase + c >= Lk)) v = -INFINITY;
        x[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        const float pr = fast_exp2(__uint_as_float(x[c]) - m_new);
        rowsum += pr;
        x[c] = __float_as_uint(pr);
      }
      l = l * alpha + rowsum;
      m = m_new;
      if (j > 0) {
        // P.V of the previous tile must be done: it reads the P buffer and
        // accumulates into the O row that is rescaled here
        if (!__all_sync(0xffffffffu, wait_(bar(kBarO), (j - 1) & 1, abort))) {
          good = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle
#pragma unroll
      for (int ch = 0; ch < kBN / 8; ++ch) {
        const uint32_t w0 = pack_bf16x2(__uint_as_float(x[ch * 8 + 0]), __uint_as_float(x[ch * 8 + 1]));
        const uint32_t w1 = pack_bf16x2(__uint_as_float(x[ch * 8 + 2]), __uint_as_float(x[ch * 8 + 3]));
        const uint32_t w2 = pack_bf16x2(__uint_as_float(x[ch * 8 + 4]), __uint_as_float(x[ch * 8 + 5]));
        const uint32_t w3 = pack_bf16x2(__uint_as_float(x[ch * 8 + 6]), __uint_as_float(x[ch * 8 + 7]));
        const uint32_t addr = sP + (ch >> 3) * kHalfBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1),
                     "r"(w2), "r"(w3)
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarP));
    }
    if (__all_sync(0xffffffffu, good && wait_(bar(kBarO), (n_tiles - 1) & 1, abort))) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool store = qi < Lq;
      __nv_bfloat16 *orow = p.out + (static_cast<int64_t>(q0 + qi) * p.num_q_heads + h) * kD;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[i + 0]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
            *reinterpret_cast<uint4 *>(orow + c * 32 + i) = v;
          }
        }
      }
      if (store && p.lse != nullptr)
        p.lse[static_cast<int64_t>(q0 + qi) * p.num_q_heads + h] = (m + log2f(l)) * kLn2;
    } else if (tid == 0) {
      fail(abort);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t stream) {
  if (a.total_q == 0 || a.max_seqlen_q == 0 || a.num_seqs == 0) return cudaSuccess;
  PrefillParams p;
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.block_tables = a.block_tables;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q;
  p.max_seqlen_q = a.max_seqlen_q;
  p.max_seqlen_k = a.max_seqlen_k;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.n_qtiles = (a.max_seqlen_q + kBM - 1) / kBM;
  p.scale_log2 = a.scale_log2;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_qtiles, a.num_q_heads, a.num_seqs);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(q_map, k_map, v_map, p);
  return cudaGetLastError();
}

cudaError_t take_prefill_errors(cudaStream_t stream, uint32_t *flags) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_prefill_errors, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_prefill_errors, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  *flags |= v;
  return cudaSuccess;
}

}  // namespace pkv
