// Paged decode attention, one query token per sequence: the engine's q=1
// decode step ("nano-vllm-sansho" README, "Sansho Serving Roofline Anchors",
// where a q=1 decode kernel runs under CUDA-graph replay and KV traffic is one
// of the costs the crude weight roof ignores).
//
// Split-K ("flash decoding") over the context, on CUDA cores:
//
//   split kernel   grid (split j, KV head g, sequence s). Each of the NW warps of
//                  a CTA streams its own 32-key chunks of the split: lane 0
//                  issues two 16-row TMA boxes for K and two for V per chunk
//                  (a box never crosses a cache block because block_size is a
//                  multiple of 16) into the warp's shared-memory ring, and the
//                  warp computes the G query heads that share KV head g
//                  against the staged rows: logits with one lane group per key
//                  and a transposing butterfly reduction (each lane ends with
//                  one key's logit), a chunk-wise online softmax in base 2,
//                  then P.V with half-warps on alternate keys. The warps'
//                  (max, sum, output) triples are merged in shared memory; a
//                  sequence that needs a single split writes its final bf16
//                  output and lse directly, otherwise the split's normalised
//                  output and log2-sum-exp go to the workspace.
//   merge kernel   grid (query head, sequence): combines the splits of the
//                  sequences that have more than one.
//
// The 2-wide GQA group makes the logits and P.V skinny matrix-vector products,
// so the kernel is bound by HBM bandwidth, not by any tensor-core contraction.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

static __device__ uint32_t g_decode_errors;

namespace {

constexpr int kD = 128;                 // head dim (the only one supported)
constexpr int kChunk = kDecodeChunk;    // 32 keys
constexpr int kBoxRows = 16;            // rows per TMA box
constexpr int kRowBytes = kD * 2;       // 256 bytes of one head's K (or V) row
constexpr int kBoxBytes = kBoxRows * kRowBytes;          // 4 KiB
constexpr int kStageBytes = 2 * kChunk * kRowBytes;      // K + V of a chunk: 16 KiB
constexpr float kLn2 = 0.693147180559945309f;

struct DecodeParams {
  const __nv_bfloat16 *q;
  const int32_t *block_tables;
  const int32_t *context_lens;
  __nv_bfloat16 *out;
  float *lse;
  float *ws_o;
  float *ws_lse;
  int32_t max_blocks, max_context_len, num_q_heads, block_size, num_blocks;
  int32_t keys_per_split, num_splits;
  float scale_log2;
};

template <int G, int NW, int NS>
struct DecodeSmem {
  static constexpr int kStagesOffset = 0;
  static constexpr int kStagesBytes = NW * NS * kStageBytes;
  static constexpr int kProbOffset = kStagesBytes;                     // float [NW][32][G]
  static constexpr int kProbBytes = NW * kChunk * G * 4;
  static constexpr int kCmbOOffset = kProbOffset + kProbBytes;         // float [NW][G][128]
  static constexpr int kCmbOBytes = NW * G * kD * 4;
  static constexpr int kCmbMLOffset = kCmbOOffset + kCmbOBytes;        // float [NW][G][2]
  static constexpr int kCmbMLBytes = NW * G * 2 * 4;
  static constexpr int kBarOffset = (kCmbMLOffset + kCmbMLBytes + 7) & ~7;
  static constexpr int kBarBytes = NW * NS * 8;
  static constexpr int kTotal = kBarOffset + kBarBytes + 128;  // + alignment slack
};

// Issue the TMA copies of chunk c of the split into a stage. Returns nothing;
// the stage's barrier completes when every issued byte has landed (or at once
// if no box could be issued).
__device__ __forceinline__ void issue_chunk(const CUtensorMap *k_map, const CUtensorMap *v_map,
                                            const DecodeParams &p, int s, int g, int key0,
                                            int key_end, uint32_t stage, uint32_t bar,
                                            uint64_t policy) {
  int32_t rows[2];
  uint32_t nbox = 0;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    rows[b] = -1;
    const int kb = key0 + b * kBoxRows;
    if (kb < key_end) {
      const int32_t blk = p.block_tables[static_cast<int64_t>(s) * p.max_blocks + kb / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(&g_decode_errors, kErrBlock);
      } else {
        rows[b] = blk * p.block_size + kb % p.block_size;
        ++nbox;
      }
    }
  }
  mbar_arrive_expect_tx(bar, nbox * 2u * kBoxBytes);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    if (rows[b] >= 0) {
      tma_load_3d_hint(stage + b * kBoxBytes, k_map, bar, 0, g, rows[b], policy);
      tma_load_3d_hint(stage + kChunk * kRowBytes + b * kBoxBytes, v_map, bar, 0, g, rows[b],
                       policy);
    }
  }
}

// One step of the transposing butterfly: lanes whose `bit` of the 8-lane
// sub-index is set keep the upper half of their n partial sums and send the
// lower half; partners do the opposite; both add what they receive.
template <int N>
__device__ __forceinline__ void butterfly_half(float (&x)[N], bool upper, int lane_mask) {
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float send = upper ? x[i] : x[i + N / 2];
    const float keep = upper ? x[i + N / 2] : x[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, lane_mask);
  }
}

template <int G, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
    decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using L = DecodeSmem<G, NW, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                              ~static_cast<uintptr_t>(127));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = blockIdx.x, g = blockIdx.y, s = blockIdx.z;

  // a CTA gave up waiting (in this or an earlier launch): skip the work until
  // the error word is read and cleared; decided once per CTA
  if (__syncthreads_or(threadIdx.x == 0 &&
                       (*reinterpret_cast<volatile uint32_t *>(&g_decode_errors) & kErrTimeout)))
    return;
  const int ctx = p.context_lens[s];
  if (ctx <= 0 || ctx > p.max_context_len ||
      static_cast<int64_t>(ctx) > static_cast<int64_t>(p.max_blocks) * p.block_size) {
    if (j == 0 && threadIdx.x == 0) atomicOr(&g_decode_errors, kErrContext);
    return;
  }
  const int key_begin = j * p.keys_per_split;
  if (key_begin >= ctx) return;  // this split has no keys for this sequence
  const int key_end = min(key_begin + p.keys_per_split, ctx);
  const int nchunks = (key_end - key_begin + kChunk - 1) / kChunk;
  const int nsplits_s = (ctx + p.keys_per_split - 1) / p.keys_per_split;
  const int mine = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;

  const uint32_t stage0 = smem_u32(smem + L::kStagesOffset) + warp * NS * kStageBytes;
  const uint32_t bar0 = smem_u32(smem + L::kBarOffset) + warp * NS * 8;
  float *prob = reinterpret_cast<float *>(smem + L::kProbOffset) + warp * kChunk * G;
  const uint64_t policy = l2_policy_evict_first();

  if (lane == 0) {
    if (warp == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_barrier_init();
#pragma unroll
    for (int i = 0; i < NS; ++i)
      if (i < mine)
        issue_chunk(&k_map, &v_map, p, s, g, key_begin + (warp + i * NW) * kChunk, key_end,
                    stage0 + i * kStageBytes, bar0 + 8 * i, policy);
  }
  __syncwarp();

  // This lane's 16 query dims for each of the G heads, pre-scaled into the
  // base-2 logit domain: dims sub*8 .. sub*8+7 and 64 + sub*8 .. 64 + sub*8+7.
  const int sub = lane & 7, grp = lane >> 3;
  float qf[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 *qrow = reinterpret_cast<const uint4 *>(
        p.q + (static_cast<int64_t>(s) * p.num_q_heads + g * G + h) * kD);
    const uint4 a = qrow[sub], b = qrow[8 + sub];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qf[h][2 * i] = bf16lo(wa[i]) * p.scale_log2;
      qf[h][2 * i + 1] = bf16hi(wa[i]) * p.scale_log2;
      qf[h][8 + 2 * i] = bf16lo(wb[i]) * p.scale_log2;
      qf[h][8 + 2 * i + 1] = bf16hi(wb[i]) * p.scale_log2;
    }
  }

  float m[G], lsum[G], o[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[h][i] = 0.f;
  }
  // key owned by this lane after the butterfly, and this lane's V dims
  const int my_key = 4 * sub + grp;
  const int half = lane >> 4, vcol = lane & 15;
  bool ok = true;

#pragma unroll 1
  for (int it = 0; it < mine; ++it) {
    const int st = it % NS;
    const uint32_t stage = stage0 + st * kStageBytes;
    const bool landed = mbar_wait(bar0 + 8 * st, (it / NS) & 1, &g_decode_errors);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) atomicOr(&g_decode_errors, kErrTimeout);
      ok = false;
      break;
    }
    const int key0 = key_begin + (warp + it * NW) * kChunk;
    const int nvalid = min(kChunk, key_end - key0);
    const uint8_t *kst = smem + L::kStagesOffset + (warp * NS + st) * kStageBytes;
    const uint8_t *vst = kst + kChunk * kRowBytes;

    // ---- logits: pass pp covers keys 4*pp + grp, lane group grp, sub-dims sub
    float part[G][8];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      const uint8_t *krow = kst + (4 * pp + grp) * kRowBytes;
      const uint4 ka = *reinterpret_cast<const uint4 *>(krow + sub * 16);
      const uint4 kb = *reinterpret_cast<const uint4 *>(krow + 128 + sub * 16);
      const uint32_t w[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = fmaf(qf[h][2 * i], bf16lo(w[i]), acc);
          acc = fmaf(qf[h][2 * i + 1], bf16hi(w[i]), acc);
        }
        part[h][pp] = acc;
      }
    }
    // transposing reduction over the 8 lanes of a group: afterwards lane
    // (grp, sub) holds the full logit of key 4*sub + grp
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      butterfly_half<8>(part[h], (sub & 4) != 0, 4);
      float q4[4] = {part[h][0], part[h][1], part[h][2], part[h][3]};
      butterfly_half<4>(q4, (sub & 2) != 0, 2);
      float q2[2] = {q4[0], q4[1]};
      butterfly_half<2>(q2, (sub & 1) != 0, 1);
      sc[h] = my_key < nvalid ? q2[0] : -INFINITY;
    }

    // ---- online softmax over the chunk (base 2)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = sc[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[h], mx);
      const float alpha = fast_exp2(m[h] - m_new);  // 0 on the first chunk
      const float pr = fast_exp2(sc[h] - m_new);    // 0 for masked keys
      lsum[h] = lsum[h] * alpha + pr;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] *= alpha;
      m[h] = m_new;
      prob[my_key * G + h] = pr;
    }
    __syncwarp();

    // ---- P.V: half-warp `half` takes keys 2*pp + half, lane covers 8 dims
#pragma unroll 4
    for (int pp = 0; pp < kChunk / 2; ++pp) {
      const int key = 2 * pp + half;
      if (2 * pp >= nvalid) break;
      if (key < nvalid) {
        const uint4 vv = *reinterpret_cast<const uint4 *>(vst + key * kRowBytes + vcol * 16);
        const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) pr[h] = prob[key * G + h];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v0 = bf16lo(w[i]), v1 = bf16hi(w[i]);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            o[h][2 * i] = fmaf(pr[h], v0, o[h][2 * i]);
            o[h][2 * i + 1] = fmaf(pr[h], v1, o[h][2 * i + 1]);
          }
        }
      }
    }
    // every lane is done with this stage (and with prob) before it is refilled
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && it + NS < mine)
      issue_chunk(&k_map, &v_map, p, s, g, key_begin + (warp + (it + NS) * NW) * kChunk, key_end,
                  stage, bar0 + 8 * st, policy);
  }

  // ---- warp result: fold the two half-warps, reduce the row sums
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[h][i] += __shfl_xor_sync(0xffffffffu, o[h][i], 16);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], off);
  }
  float *cmb_o = reinterpret_cast<float *>(smem + L::kCmbOOffset);
  float *cmb_ml = reinterpret_cast<float *>(smem + L::kCmbMLOffset);
  if (lane < 16) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float4 *dst = reinterpret_cast<float4 *>(cmb_o + (warp * G + h) * kD + vcol * 8);
      dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
      dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      cmb_ml[(warp * G + h) * 2] = ok ? m[h] : -INFINITY;
      cmb_ml[(warp * G + h) * 2 + 1] = ok ? lsum[h] : 0.f;
    }
  }
  __syncthreads();

  // ---- merge the warps; write the final row or this split's partial
  for (int idx = threadIdx.x; idx < G * kD; idx += NW * 32) {
    const int h = idx / kD, d = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, cmb_ml[(w * G + h) * 2]);
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float wm = cmb_ml[(w * G + h) * 2];
      if (wm == -INFINITY) continue;
      const float sc = fast_exp2(wm - M);
      Lsum += cmb_ml[(w * G + h) * 2 + 1] * sc;
      O += cmb_o[(w * G + h) * kD + d] * sc;
    }
    const int qh = g * G + h;
    const int64_t row = static_cast<int64_t>(s) * p.num_q_heads + qh;
    if (nsplits_s == 1) {
      p.out[row * kD + d] = __float2bfloat16_rn(O / Lsum);
      if (d == 0 && p.lse != nullptr) p.lse[row] = (M + log2f(Lsum)) * kLn2;
    } else {
      p.ws_o[(row * p.num_splits + j) * kD + d] = O / Lsum;
      if (d == 0) p.ws_lse[row * p.num_splits + j] = M + log2f(Lsum);
    }
  }
}

__global__ void __launch_bounds__(kD)
    decode_merge_kernel(const DecodeParams p) {
  const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
  const int ctx = p.context_lens[s];
  if (ctx <= 0 || ctx > p.max_context_len ||
      static_cast<int64_t>(ctx) > static_cast<int64_t>(p.max_blocks) * p.block_size)
    return;
  const int n = (ctx + p.keys_per_split - 1) / p.keys_per_split;
  if (n <= 1) return;
  const int64_t row = static_cast<int64_t>(s) * p.num_q_heads + h;
  const float *lse_j = p.ws_lse + row * p.num_splits;
  const float *o_j = p.ws_o + row * p.num_splits * kD;
  float M = -INFINITY;
  for (int jj = 0; jj < n; ++jj) M = fmaxf(M, lse_j[jj]);
  float Lsum = 0.f, O = 0.f;
  for (int jj = 0; jj < n; ++jj) {
    const float w = fast_exp2(lse_j[jj] - M);
    Lsum += w;
    O = fmaf(w, o_j[jj * kD + d], O);
  }
  p.out[row * kD + d] = __float2bfloat16_rn(O / Lsum);
  if (d == 0 && p.lse != nullptr) p.lse[row] = (M + log2f(Lsum)) * kLn2;
}

template <int G, int NW, int NS>
cudaError_t launch_variant(const DecodeArgs &a, const CUtensorMap &k_map,
                           const CUtensorMap &v_map, const DecodeParams &p,
                           cudaStream_t stream) {
  using L = DecodeSmem<G, NW, NS>;
  auto kern = decode_split_kernel<G, NW, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
  kern<<<grid, NW * 32, L::kTotal, stream>>>(k_map, v_map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.num_splits > 1) {
    decode_merge_kernel<<<dim3(a.num_q_heads, a.num_seqs), kD, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

int32_t decode_chunks_per_split(const DecodeArgs &a, int num_sms, int32_t override_chunks) {
  if (override_chunks > 0) {
    return override_chunks < kDecodeMinChunksPerSplit ? kDecodeMinChunksPerSplit
           : override_chunks > 1024                   ? 1024
                                                      : override_chunks;
  }
  // Enough CTAs for about two full waves of 3 resident CTAs per SM, with a
  // multiple of 4 chunks per split (one per warp and round).
  const int64_t chunks_max = (static_cast<int64_t>(a.max_context_len) + kChunk - 1) / kChunk;
  const int64_t pairs = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  const int64_t target = static_cast<int64_t>(num_sms) * 3 * 2;
  int64_t splits = (target + pairs - 1) / pairs;
  if (splits < 1) splits = 1;
  int64_t cps = (chunks_max + splits - 1) / splits;
  cps = (cps + 3) / 4 * 4;
  if (cps < kDecodeMinChunksPerSplit) cps = kDecodeMinChunksPerSplit;
  if (cps > 1024) cps = 1024;
  return static_cast<int32_t>(cps);
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, cudaStream_t stream) {
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.max_blocks = a.max_blocks;
  p.max_context_len = a.max_context_len;
  p.num_q_heads = a.num_q_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.keys_per_split = a.chunks_per_split * kChunk;
  p.num_splits = a.num_splits;
  p.scale_log2 = a.scale_log2;
  const int G = a.num_q_heads / a.num_kv_heads;
  switch (G) {
    case 1: return launch_variant<1, 4, 1>(a, k_map, v_map, p, stream);
    case 2: return launch_variant<2, 4, 1>(a, k_map, v_map, p, stream);
    case 4: return launch_variant<4, 4, 1>(a, k_map, v_map, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_decode_errors(cudaStream_t stream, uint32_t *flags) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_decode_errors, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_decode_errors, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  *flags |= v;
  return cudaSuccess;
}

}  // namespace pkv
