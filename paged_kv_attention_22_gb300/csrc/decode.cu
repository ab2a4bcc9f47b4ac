// Paged decode attention, one query token per sequence: the engine's q=1
// decode step ("nano-vllm-sansho" README, "Sansho Serving Roofline Anchors",
// where a q=1 decode kernel runs under CUDA-graph replay and KV traffic is one
// of the costs the crude weight roof ignores).
//
// One persistent kernel on CUDA cores, bound by HBM bandwidth:
//
//   Work list. The keys of every (sequence s, KV head g) pair are cut into
//   32-key chunks; pairs are listed in (s, g) order, so the whole call is one
//   list of C chunks. The grid holds one CTA per SM with NW warps, and the list
//   is cut into W = min(grid * NW, C) equal contiguous ranges, one per warp:
//   every warp moves the same number of bytes whatever the mix of context
//   lengths, and no wave of CTAs is left half full.
//
//   Streaming. Each warp runs its own NS-deep ring of shared-memory stages:
//   lane 0 issues, per chunk, two 16-row TMA boxes of K and two of V (a box
//   never crosses a cache block since block_size is a multiple of 16) and,
//   for the first chunk of a segment, the pair's G query rows; the warp
//   computes one chunk while the next ones land.
//
//   Math. Logits with one 8-lane group per key and a transposing butterfly
//   reduction (each lane ends with one key's logit), chunk-wise online softmax
//   in base 2, then P.V with half-warps on alternate keys; the G query heads
//   of a KV head share every staged byte.
//
//   Merge. A pair that lies inside one warp's range is finished by that warp.
//   A pair cut by range boundaries leaves one (max, sum, output) partial per
//   warp in the workspace: the first segment of warp w goes to slot 2w, its
//   last segment (if different) to slot 2w+1. Each such warp then bumps the
//   pair's arrival counter, and the last one to arrive merges the partials and
//   writes the row. Nothing waits on another CTA. The counters are zeroed on
//   the stream right before the kernel.
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
constexpr int kKVBytes = 2 * kChunk * kRowBytes;         // K + V of a chunk: 16 KiB
constexpr float kLn2 = 0.693147180559945309f;

struct DecodeParams {
  const int32_t *block_tables;
  const int32_t *context_lens;
  __nv_bfloat16 *out;
  float *lse;
  float *ws_o;
  float *ws_ml;
  uint32_t *ws_cnt;
  int32_t max_blocks, max_context_len, num_seqs, num_q_heads, num_kv_heads, block_size,
      num_blocks;
  float scale_log2;
};

template <int G, int NW, int NS>
struct DecodeSmem {
  static constexpr int kQBytes = G * kRowBytes;
  static constexpr int kStageBytes = kKVBytes + kQBytes;        // K, V, then the q rows
  static constexpr int kStagesBytes = NW * NS * kStageBytes;
  static constexpr int kProbOffset = kStagesBytes;              // float [NW][G][32]
  static constexpr int kProbBytes = NW * kChunk * G * 4;
  static constexpr int kBarOffset = kProbOffset + kProbBytes;   // u64 [NW][NS]
  static constexpr int kBarBytes = NW * NS * 8;
  static constexpr int kPrefixOffset = kBarOffset + kBarBytes;  // int [S + 1] chunk prefix
  static constexpr int total(int num_seqs) { return kPrefixOffset + 4 * (num_seqs + 1) + 128; }
};

// Position in the chunk list: sequence, KV head, chunk within the pair.
struct Cursor {
  int s, g, k;
};

__device__ __forceinline__ int chunks_of(const int *prefix, int s) {
  return prefix[s + 1] - prefix[s];
}

// Cursor of global chunk c (c < C): sequence s owns H_kv * chunks_of(s)
// consecutive chunks starting at H_kv * prefix[s].
__device__ __forceinline__ Cursor locate(const int *prefix, int num_seqs, int H_kv, int64_t c) {
  int lo = 0, hi = num_seqs - 1;  // largest s with H_kv * prefix[s] <= c (never empty)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(H_kv) * prefix[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const int n = chunks_of(prefix, lo);
  const int64_t r = c - static_cast<int64_t>(H_kv) * prefix[lo];
  return Cursor{lo, static_cast<int>(r / n), static_cast<int>(r % n)};
}

// Next chunk in list order; past the last chunk, s becomes num_seqs.
__device__ __forceinline__ void advance(Cursor &cur, const int *prefix, int num_seqs, int H_kv) {
  if (++cur.k < chunks_of(prefix, cur.s)) return;
  cur.k = 0;
  if (++cur.g < H_kv) return;
  cur.g = 0;
  do {
    ++cur.s;
  } while (cur.s < num_seqs && chunks_of(prefix, cur.s) == 0);
}

// First chunk of warp w's range among W warps over C chunks (W <= C, so every
// range is non-empty), and the warp whose range holds chunk c.
__device__ __forceinline__ int64_t range_start(int64_t w, int64_t W, int64_t C) {
  return w * C / W;
}
__device__ __forceinline__ int64_t owner_of(int64_t c, int64_t W, int64_t C) {
  return ((c + 1) * W + C - 1) / C - 1;
}

// Issue chunk `cur` into a stage: K and V boxes, plus the q rows when it opens
// a segment. The stage's barrier completes when every issued byte has landed.
template <int G>
__device__ __forceinline__ void issue_chunk(const CUtensorMap *k_map, const CUtensorMap *v_map,
                                            const CUtensorMap *q_map, const DecodeParams &p,
                                            const Cursor &cur, bool with_q, uint32_t stage,
                                            uint32_t bar, uint64_t policy) {
  const int ctx = p.context_lens[cur.s];
  const int key0 = cur.k * kChunk;
  int32_t rows[2];
  uint32_t bytes = with_q ? G * kRowBytes : 0;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    rows[b] = -1;
    const int kb = key0 + b * kBoxRows;
    if (kb < ctx) {
      const int32_t blk =
          p.block_tables[static_cast<int64_t>(cur.s) * p.max_blocks + kb / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(&g_decode_errors, kErrBlock);
      } else {
        rows[b] = blk * p.block_size + kb % p.block_size;
        bytes += 2 * kBoxBytes;
      }
    }
  }
  mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    if (rows[b] >= 0) {
      tma_load_3d_hint(stage + b * kBoxBytes, k_map, bar, 0, cur.g, rows[b], policy);
      tma_load_3d_hint(stage + kChunk * kRowBytes + b * kBoxBytes, v_map, bar, 0, cur.g, rows[b],
                       policy);
    }
  }
  if (with_q) tma_load_3d(stage + kKVBytes, q_map, bar, 0, cur.g * G, cur.s);
}

// One step of the transposing butterfly: lanes whose sub-index bit is set keep
// the upper half of their partial sums and send the lower half; partners do
// the opposite; both add what they receive.
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
__global__ void __launch_bounds__(NW * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map,
                  const __grid_constant__ CUtensorMap q_map, const DecodeParams p) {
  using L = DecodeSmem<G, NW, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                              ~static_cast<uintptr_t>(127));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int H_kv = p.num_kv_heads;

  // a CTA gave up waiting (in this or an earlier launch): skip the work until
  // the error word is read and cleared; decided once per CTA
  if (__syncthreads_or(threadIdx.x == 0 &&
                       (*reinterpret_cast<volatile uint32_t *>(&g_decode_errors) & kErrTimeout)))
    return;

  // ---- chunk prefix over sequences (invalid lengths count as empty)
  int *prefix = reinterpret_cast<int *>(smem + L::kPrefixOffset);
  if (warp == 0) {
    int carry = 0;
    const int64_t ctx_cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
    for (int base = 0; base < p.num_seqs; base += 32) {
      const int s = base + lane;
      int n = 0;
      if (s < p.num_seqs) {
        const int ctx = p.context_lens[s];
        if (ctx <= 0 || ctx > p.max_context_len || ctx > ctx_cap) {
          if (blockIdx.x == 0) atomicOr(&g_decode_errors, kErrContext);
        } else {
          n = (ctx + kChunk - 1) / kChunk;
        }
      }
      int incl = n;  // inclusive warp scan
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      if (s < p.num_seqs) prefix[s] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[p.num_seqs] = carry;
  }
  __syncthreads();

  const int64_t C = static_cast<int64_t>(H_kv) * prefix[p.num_seqs];
  const int64_t W_all = static_cast<int64_t>(gridDim.x) * NW;
  const int64_t W = W_all < C ? W_all : C;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * NW + warp;
  if (w >= W) return;  // no chunks for this warp (no CTA-wide sync follows)
  const int64_t c_lo = range_start(w, W, C), c_hi = range_start(w + 1, W, C);
  const int n_mine = static_cast<int>(c_hi - c_lo);

  const uint32_t stage0 = smem_u32(smem) + static_cast<uint32_t>(warp * NS) * L::kStageBytes;
  const uint32_t bar0 = smem_u32(smem + L::kBarOffset) + warp * NS * 8;
  float *prob = reinterpret_cast<float *>(smem + L::kProbOffset) + warp * kChunk * G;
  const uint64_t policy = l2_policy_evict_first();

  // the issue cursor runs up to NS chunks ahead of the compute cursor
  Cursor icur = locate(prefix, p.num_seqs, H_kv, c_lo);
  Cursor ccur = icur;
  if (lane == 0) {
    if (warp == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      prefetch_tensormap(&q_map);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_barrier_init();
  }
  __syncwarp();
  for (int i = 0; i < NS && i < n_mine; ++i) {
    if (lane == 0)
      issue_chunk<G>(&k_map, &v_map, &q_map, p, icur, i == 0 || icur.k == 0,
                     stage0 + i * L::kStageBytes, bar0 + 8 * i, policy);
    advance(icur, prefix, p.num_seqs, H_kv);
  }

  const int sub = lane & 7, grp = lane >> 3;
  const int my_key = 4 * sub + grp;        // key owned after the butterfly
  const int half = lane >> 4, vcol = lane & 15;
  float qf[G][16];
  float m[G], lsum[G], o[G][8];
  int seg_first_k = 0;                     // chunk index (in the pair) opening the segment
  bool seg_is_first = true;                // segment opened at this warp's range start
  int ctx = 0;

#pragma unroll 1
  for (int it = 0; it < n_mine; ++it) {
    const int st = it % NS;
    const uint32_t stage = stage0 + st * L::kStageBytes;
    const uint8_t *kst = smem + static_cast<size_t>(warp * NS + st) * L::kStageBytes;
    const uint8_t *vst = kst + kChunk * kRowBytes;
    const bool opens = (it == 0) || (ccur.k == 0);
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * st, (it / NS) & 1, &g_decode_errors))) {
      if (lane == 0) atomicOr(&g_decode_errors, kErrTimeout);
      return;  // a lost copy: rows of this warp's range stay unwritten
    }
    if (opens) {
      // a new segment: its q rows came with this chunk
      ctx = p.context_lens[ccur.s];
      seg_first_k = ccur.k;
      seg_is_first = (it == 0);
      const uint8_t *qs = kst + kKVBytes;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint4 a = *reinterpret_cast<const uint4 *>(qs + h * kRowBytes + sub * 16);
        const uint4 b = *reinterpret_cast<const uint4 *>(qs + h * kRowBytes + 128 + sub * 16);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qf[h][2 * i] = bf16lo(wa[i]) * p.scale_log2;
          qf[h][2 * i + 1] = bf16hi(wa[i]) * p.scale_log2;
          qf[h][8 + 2 * i] = bf16lo(wb[i]) * p.scale_log2;
          qf[h][8 + 2 * i + 1] = bf16hi(wb[i]) * p.scale_log2;
        }
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[h][i] = 0.f;
      }
    }
    const int nvalid = min(kChunk, ctx - ccur.k * kChunk);

    // ---- logits: pass pp covers keys 4*pp + grp; lane group grp, sub-dims sub
    float part[G][8];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      const uint8_t *krow = kst + (4 * pp + grp) * kRowBytes;
      const uint4 ka = *reinterpret_cast<const uint4 *>(krow + sub * 16);
      const uint4 kb = *reinterpret_cast<const uint4 *>(krow + 128 + sub * 16);
      const uint32_t wv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = fmaf(qf[h][2 * i], bf16lo(wv[i]), acc);
          acc = fmaf(qf[h][2 * i + 1], bf16hi(wv[i]), acc);
        }
        part[h][pp] = acc;
      }
    }
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
      const float alpha = fast_exp2(m[h] - m_new);  // 0 on a segment's first chunk
      const float pr = fast_exp2(sc[h] - m_new);    // 0 for masked keys
      lsum[h] = lsum[h] * alpha + pr;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] *= alpha;
      m[h] = m_new;
      prob[h * kChunk + my_key] = pr;
    }
    __syncwarp();

    // ---- P.V: half-warp `half` takes keys 2*pp + half, a lane covers 8 dims
#pragma unroll 4
    for (int pp = 0; pp < kChunk / 2; ++pp) {
      const int key = 2 * pp + half;
      if (2 * pp >= nvalid) break;
      if (key < nvalid) {
        const uint4 vv = *reinterpret_cast<const uint4 *>(vst + key * kRowBytes + vcol * 16);
        const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) pr[h] = prob[h * kChunk + key];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v0 = bf16lo(wv[i]), v1 = bf16hi(wv[i]);
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
    if (it + NS < n_mine) {
      if (lane == 0)
        issue_chunk<G>(&k_map, &v_map, &q_map, p, icur, icur.k == 0, stage, bar0 + 8 * st,
                       policy);
      advance(icur, prefix, p.num_seqs, H_kv);
    }

    // ---- segment end: the pair's last chunk, or this warp's last chunk
    const int nch = chunks_of(prefix, ccur.s);
    const bool pair_ends = ccur.k == nch - 1;
    if (pair_ends || it == n_mine - 1) {
      float lt[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[h][i] += __shfl_xor_sync(0xffffffffu, o[h][i], 16);
        lt[h] = lsum[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], off);
      }
      const int64_t row0 = static_cast<int64_t>(ccur.s) * p.num_q_heads + ccur.g * G;
      if (seg_first_k == 0 && pair_ends) {
        // the whole pair is in this segment: write the final row
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float inv = 1.f / lt[h];
            uint4 v;
            v.x = pack_bf16x2(o[h][0] * inv, o[h][1] * inv);
            v.y = pack_bf16x2(o[h][2] * inv, o[h][3] * inv);
            v.z = pack_bf16x2(o[h][4] * inv, o[h][5] * inv);
            v.w = pack_bf16x2(o[h][6] * inv, o[h][7] * inv);
            *reinterpret_cast<uint4 *>(p.out + (row0 + h) * kD + vcol * 8) = v;
          }
        }
        if (lane == 0 && p.lse != nullptr) {
#pragma unroll
          for (int h = 0; h < G; ++h) p.lse[row0 + h] = (m[h] + log2f(lt[h])) * kLn2;
        }
      } else {
        // a piece of a pair cut by range boundaries: publish the partial
        const int64_t slot = 2 * w + (seg_is_first ? 0 : 1);
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (slot * G + h) * kD + vcol * 8);
            __stcg(dst, make_float4(o[h][0], o[h][1], o[h][2], o[h][3]));
            __stcg(dst + 1, make_float4(o[h][4], o[h][5], o[h][6], o[h][7]));
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            __stcg(p.ws_ml + (slot * G + h) * 2, m[h]);
            __stcg(p.ws_ml + (slot * G + h) * 2 + 1, lt[h]);
          }
        }
        __threadfence();
        __syncwarp();
        const int64_t pair = static_cast<int64_t>(ccur.s) * H_kv + ccur.g;
        const int64_t P0 =
            static_cast<int64_t>(H_kv) * prefix[ccur.s] + static_cast<int64_t>(ccur.g) * nch;
        const int64_t wa = owner_of(P0, W, C), wb = owner_of(P0 + nch - 1, W, C);
        uint32_t arrived = 0;
        if (lane == 0) arrived = atomicAdd(p.ws_cnt + pair, 1u) + 1u;
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == static_cast<uint32_t>(wb - wa + 1)) {
          // last piece in: merge the pair's partials. Warp wa holds it in its
          // last slot unless its range starts at the pair's first chunk.
          __threadfence();
          const int64_t wa_slot = 2 * wa + (range_start(wa, W, C) < P0 ? 1 : 0);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            // max and sum over the pieces: lanes split the pieces, then reduce
            float M = -INFINITY;
            for (int64_t x = wa + lane; x <= wb; x += 32) {
              const int64_t sl = x == wa ? wa_slot : 2 * x;
              M = fmaxf(M, __ldcg(p.ws_ml + (sl * G + h) * 2));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            float Lsum = 0.f;
            for (int64_t x = wa + lane; x <= wb; x += 32) {
              const int64_t sl = x == wa ? wa_slot : 2 * x;
              Lsum += __ldcg(p.ws_ml + (sl * G + h) * 2 + 1) *
                      fast_exp2(__ldcg(p.ws_ml + (sl * G + h) * 2) - M);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
            // output: each lane owns 4 dims
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int64_t x = wa; x <= wb; ++x) {
              const int64_t sl = x == wa ? wa_slot : 2 * x;
              const float f = fast_exp2(__ldcg(p.ws_ml + (sl * G + h) * 2) - M);
              const float4 ov =
                  __ldcg(reinterpret_cast<const float4 *>(p.ws_o + (sl * G + h) * kD) + lane);
              acc[0] = fmaf(ov.x, f, acc[0]);
              acc[1] = fmaf(ov.y, f, acc[1]);
              acc[2] = fmaf(ov.z, f, acc[2]);
              acc[3] = fmaf(ov.w, f, acc[3]);
            }
            const float inv = 1.f / Lsum;
            uint2 v;
            v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2 *>(p.out + (row0 + h) * kD + lane * 4) = v;
            if (lane == 0 && p.lse != nullptr) p.lse[row0 + h] = (M + log2f(Lsum)) * kLn2;
          }
        }
      }
    }
    advance(ccur, prefix, p.num_seqs, H_kv);
  }
}

template <int G, int NW, int NS>
cudaError_t launch_variant(const DecodeArgs &a, const CUtensorMap &k_map,
                           const CUtensorMap &v_map, const CUtensorMap &q_map,
                           const DecodeParams &p, cudaStream_t stream) {
  using L = DecodeSmem<G, NW, NS>;
  static_assert(L::total(kDecodeMaxSeqs) <= 227 * 1024, "decode shared memory");
  auto kern = decode_kernel<G, NW, NS>;
  const int smem = L::total(a.num_seqs);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.ws_cnt, 0,
                      sizeof(uint32_t) * static_cast<size_t>(a.num_seqs) * a.num_kv_heads, stream);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, NW * 32, smem, stream>>>(k_map, v_map, q_map, p);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_group(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                         const CUtensorMap &q_map, const DecodeParams &p, cudaStream_t stream) {
  static_assert(kDecodeNumVariants == 4, "variant table");
  switch (a.variant) {
    case 1: return launch_variant<G, kDecodeVariants[1].warps, kDecodeVariants[1].stages>(
        a, k_map, v_map, q_map, p, stream);
    case 2: return launch_variant<G, kDecodeVariants[2].warps, kDecodeVariants[2].stages>(
        a, k_map, v_map, q_map, p, stream);
    case 3: return launch_variant<G, kDecodeVariants[3].warps, kDecodeVariants[3].stages>(
        a, k_map, v_map, q_map, p, stream);
    default: return launch_variant<G, kDecodeVariants[0].warps, kDecodeVariants[0].stages>(
        a, k_map, v_map, q_map, p, stream);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, const CUtensorMap &q_map,
                          cudaStream_t stream) {
  DecodeParams p;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.ws_cnt = a.ws_cnt;
  p.max_blocks = a.max_blocks;
  p.max_context_len = a.max_context_len;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_group<1>(a, k_map, v_map, q_map, p, stream);
    case 2: return launch_group<2>(a, k_map, v_map, q_map, p, stream);
    case 4: return launch_group<4>(a, k_map, v_map, q_map, p, stream);
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
