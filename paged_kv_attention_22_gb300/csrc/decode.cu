// Paged decode attention, one query token per sequence: the engine's q=1
// decode step ("nano-vllm-sansho" README, "Sansho Serving Roofline Anchors",
// where a q=1 decode kernel runs under CUDA-graph replay and KV traffic is one
// of the costs the crude weight roof ignores).
//
// One persistent kernel on CUDA cores, bound by HBM bandwidth:
//
//   Work list. A unit is 16 consecutive keys of one sequence for a group of
//   HG KV heads (all 8 heads of a Qwen3-0.6B layer): in the cache layout
//   [block, slot, head, dim] those keys are 16 contiguous token rows, so one
//   TMA box moves the whole unit's K (32 KiB for 8 heads) and one its V. Units
//   are listed in (sequence, head group, chunk) order and the list is cut into
//   min(grid, units) equal contiguous ranges, one per CTA (one CTA per SM):
//   every SM moves the same number of bytes whatever the mix of context
//   lengths, in large contiguous copies.
//
//   Warps. One producer warp streams the CTA's units through an NS-deep ring of
//   shared-memory stages (K box, V box and, when a unit opens a segment, the q
//   rows of the group; with the fused store, the new token's rows), each stage
//   freed when all consumer warps are done with it. Consumer warp g owns KV head g of the group and its G query heads:
//   logits with one 8-lane group per key and a transposing butterfly (each
//   lane ends with one key's logit), online softmax in base 2, then P.V with
//   half-warps on alternate keys.
//
//   Merge. A (sequence, KV head) whose keys all fall in one CTA's range is
//   finished by that CTA's warp. One cut by range boundaries leaves one
//   (max, sum, output) partial per CTA in the workspace (a CTA's first segment
//   in slot 2c, its last segment in slot 2c+1), stored with plain stores, and
//   a small second kernel, launched right behind this one, merges those pairs.
//   No fence, atomic or wait on another CTA holds up the stream.
//
//   Fused store. When given the new tokens' K/V rows and slots, the kernel
//   also writes them into the cache (a store warp per CTA, one sequence per
//   CTA in turn) and, for the unit that holds a sequence's new token, copies that
//   token's rows from the inputs over the staged cache row, so the result is
//   exactly that of storing first and attending after.
//
// The 2-wide GQA group makes the logits and P.V skinny matrix-vector products,
// so the kernel is bound by HBM bandwidth, not by any tensor-core contraction.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

static __device__ uint32_t g_decode_errors;

namespace {

constexpr int kD = 128;                 // head dim (the only one supported)
constexpr int kChunk = kDecodeChunk;    // 16 keys per unit
constexpr int kRowBytes = kD * 2;       // 256 bytes of one head's K (or V) row
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLazyMax = 8.0f;         // log2 units the running max may lag
constexpr int kMergeFast = 8;            // pieces merged with all loads issued at once
// Warps per merge CTA (one pair each). With many pairs, eight: the merge of a
// call then occupies fewer SMs, which the next call's decode CTAs find free
// (4 and 16 warps measured slower on 512 pairs). With fewer than
// kMergeWideMin pairs, four: there each pair is typically a long context cut
// into many pieces, and spreading the pairs over more SMs measured faster (64
// pairs of 19 pieces: 41.8 us a call against 46.0 with eight). 2-warp CTAs
// small enough to sit beside a decode CTA, one per SM, measured slower.
constexpr int kMergeWarps = 8;
constexpr int kMergeWarpsFew = 4;
constexpr int64_t kMergeWideMin = 256;

struct DecodeParams {
  const uint8_t *q;                // queries [S, H_q, D] (the CTA's first segment reads them directly)
  const uint4 *k_new, *v_new;      // fused store: the new tokens' rows [S, H_kv, D] (or null)
  uint4 *k_cache_w, *v_cache_w;    // fused store: the caches, written through these
  const int32_t *slot_mapping;     // fused store: slot of each sequence's new token
  const int32_t *block_tables;
  const int32_t *context_lens;
  __nv_bfloat16 *out;
  float *lse;
  float *ws_o;
  float *ws_ml;
  int32_t max_blocks, max_context_len, num_seqs, num_q_heads, num_kv_heads, block_size,
      num_blocks;
  int32_t hg;        // KV heads per group (= consumer warps)
  int32_t n_groups;  // num_kv_heads / hg
  int32_t window;    // sliding window (keys per query, its own included), 0: none
  int32_t stable_inputs;  // caches, tables and lengths may be read before the wait
  float scale_log2;
};

// With a sliding window the query of a sequence with ctx keys (at position
// ctx - 1) sees keys ctx - window .. ctx - 1. Its unit list starts at the
// chunk that holds the first of them; keys before that chunk are never read.
__device__ __forceinline__ int first_chunk(int ctx, int window) {
  return (window > 0 && ctx > window) ? (ctx - window) / kChunk : 0;
}
__device__ __forceinline__ int first_key(int ctx, int window) {
  return (window > 0 && ctx > window) ? ctx - window : 0;
}

// Shared memory layout for G query heads per KV head, head groups of up to
// kMaxHG KV heads and NS stages.
template <int G, int kMaxHG, int NS>
struct DecodeSmem {
  static constexpr int kKBytes = kChunk * kMaxHG * kRowBytes;     // 32 KiB for 8 heads
  static constexpr int kQBytes = kMaxHG * G * kRowBytes;
  static constexpr int kNewBytes = kMaxHG * kRowBytes;            // new token's K (or V) rows
  static constexpr int kStageBytes = 2 * kKBytes + kQBytes + 2 * kNewBytes;  // K, V, q, new K, new V
  static constexpr int kProbOffset = NS * kStageBytes;            // float [HG][G][16]
  static constexpr int kProbBytes = kMaxHG * G * kChunk * 4;
  static constexpr int kBarOffset = kProbOffset + kProbBytes;     // u64 full[NS], empty[NS]
  static constexpr int kPrefixOffset = kBarOffset + 2 * NS * 8;   // int [S + 1] chunk prefix,
                                                                  // then int [S] context lengths
  static constexpr int total(int num_seqs) { return kPrefixOffset + 4 * (2 * num_seqs + 1) + 128; }
};

// Position in the unit list: sequence, head group, chunk within the pair.
struct Cursor {
  int s, hg, k;
};

__device__ __forceinline__ int chunks_of(const int *prefix, int s) {
  return prefix[s + 1] - prefix[s];
}

// Cursor of unit u (u < U): sequence s owns n_groups * chunks_of(s)
// consecutive units starting at n_groups * prefix[s].
__device__ __forceinline__ Cursor locate(const int *prefix, int num_seqs, int n_groups,
                                         int64_t u) {
  int lo = 0, hi = num_seqs - 1;  // largest s with n_groups * prefix[s] <= u (never empty)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(n_groups) * prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int n = chunks_of(prefix, lo);
  const int64_t r = u - static_cast<int64_t>(n_groups) * prefix[lo];
  return Cursor{lo, static_cast<int>(r / n), static_cast<int>(r % n)};
}

// Next unit in list order; past the last unit, s becomes num_seqs.
__device__ __forceinline__ void advance(Cursor &cur, const int *prefix, int num_seqs,
                                        int n_groups) {
  if (++cur.k < chunks_of(prefix, cur.s)) return;
  cur.k = 0;
  if (++cur.hg < n_groups) return;
  cur.hg = 0;
  do {
    ++cur.s;
  } while (cur.s < num_seqs && chunks_of(prefix, cur.s) == 0);
}

// First unit of CTA c's range among W CTAs over U units (W <= U, so every range
// is non-empty), and the CTA whose range holds unit u.
__device__ __forceinline__ int64_t range_start(int64_t c, int64_t W, int64_t U) {
  return c * U / W;
}
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t W, int64_t U) {
  return ((u + 1) * W + U - 1) / U - 1;
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

template <int G, int kMaxHG, int NS>
__global__ void __launch_bounds__((kMaxHG + 2) * 32, 8 / kMaxHG)
    decode_kernel(const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map,
                  const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap kn_map,
                  const __grid_constant__ CUtensorMap vn_map, const DecodeParams p) {
  using L = DecodeSmem<G, kMaxHG, NS>;
  // the consumers load the q rows of the CTA's first segment themselves (G <=
  // 2: with four query heads a KV head the registers that takes would spill)
  constexpr bool kDirectQ = G <= 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                              ~static_cast<uintptr_t>(127));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int HG = p.hg;
  const int n_groups = p.n_groups;

  int *prefix = reinterpret_cast<int *>(smem + L::kPrefixOffset);
  int *ctx_of = prefix + p.num_seqs + 1;
  const uint32_t full0 = smem_u32(smem + L::kBarOffset);
  const uint32_t empty0 = full0 + NS * 8;
  const bool fused = p.k_new != nullptr;
  // independent of the inputs, so done while the previous kernel finishes:
  // barrier initialisation and the tensor-map prefetch
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, HG);
    }
    fence_barrier_init();
  }
  if (warp == HG && lane == 0) {
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    prefetch_tensormap(&q_map);
    if (fused) {
      prefetch_tensormap(&kn_map);
      prefetch_tensormap(&vn_map);
    }
  }

  // Inputs written by the previous kernel are visible after griddep_wait. With
  // stable inputs the context lengths, block tables and caches are not among
  // them: the scan and the first K/V copies go ahead, and every warp waits
  // before it reads q or the new rows or writes anything.
  if (!p.stable_inputs) griddep_wait();
  // a CTA gave up waiting (in this or an earlier launch): skip the work until
  // the error word is read and cleared; decided once per CTA
  if (__syncthreads_or(threadIdx.x == 0 &&
                       (*reinterpret_cast<volatile uint32_t *>(&g_decode_errors) & kErrTimeout)))
    return;

  // ---- chunk prefix over sequences (invalid lengths count as empty) and the
  // context lengths themselves, kept in shared memory
  if (warp == 0) {
    // every length load in flight at once, then the scan
    for (int base = 0; base < p.num_seqs; base += 128) {
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = base + 32 * u + lane;
        v[u] = s < p.num_seqs ? p.context_lens[s] : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = base + 32 * u + lane;
        if (s < p.num_seqs) ctx_of[s] = v[u];
      }
    }
    __syncwarp();
    int carry = 0;
    const int64_t ctx_cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
    for (int base = 0; base < p.num_seqs; base += 32) {
      const int s = base + lane;
      int n = 0;
      if (s < p.num_seqs) {
        const int ctx = ctx_of[s];
        if (ctx <= 0 || ctx > p.max_context_len || ctx > ctx_cap) {
          if (blockIdx.x == 0) atomicOr(&g_decode_errors, kErrContext);
        } else {
          n = (ctx + kChunk - 1) / kChunk - first_chunk(ctx, p.window);
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

  const int64_t U = static_cast<int64_t>(n_groups) * prefix[p.num_seqs];
  const int64_t W = static_cast<int64_t>(gridDim.x) < U ? static_cast<int64_t>(gridDim.x) : U;
  const int64_t cta = blockIdx.x;
  if (cta >= W) return;  // no units for this CTA
  const int64_t u_lo = range_start(cta, W, U), u_hi = range_start(cta + 1, W, U);
  const int n_mine = static_cast<int>(u_hi - u_lo);
  const uint32_t stage0 = smem_u32(smem);

  if (warp == HG) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop: lane l holds the block-table entry of unit
    // i0 + l of the current batch of 32 units, and the next batch is loaded
    // while this one is used, so no copy waits on a table read after the
    // first; lane 0 issues the copies.
    const uint32_t box = static_cast<uint32_t>(kChunk * HG * kRowBytes);
    const uint32_t qbox = static_cast<uint32_t>(HG * G * kRowBytes);
    const uint32_t nbox = static_cast<uint32_t>(HG * kRowBytes);
    const uint64_t policy = l2_policy_evict_first();
    // first key of the unit at `c` (the window, if any, starts its list)
    auto unit_key = [&](const Cursor &c) {
      return (first_chunk(ctx_of[c.s], p.window) + c.k) * kChunk;
    };
    auto entry_of = [&](int i) -> int32_t {  // table entry of this CTA's unit i, 0 past the end
      if (i >= n_mine) return 0;
      const Cursor c = locate(prefix, p.num_seqs, n_groups, u_lo + i);
      return p.block_tables[static_cast<int64_t>(c.s) * p.max_blocks + unit_key(c) / p.block_size];
    };
    int32_t batch = entry_of(lane);
    int32_t next_batch = entry_of(32 + lane);
    Cursor cur = locate(prefix, p.num_seqs, n_groups, u_lo);
    // Copies of unit i into its stage: `arm` sets the stage barrier's byte
    // count (once), `kv` issues the K and V boxes, `inputs` the q and new rows.
    auto issue = [&](int i, const Cursor &c, int32_t blk, bool arm, bool kv, bool inputs) {
      if (lane != 0) return;
      const int st = i % NS;
      const uint32_t stage = stage0 + st * L::kStageBytes;
      const uint32_t bar = full0 + 8 * st;
      // the q rows of every segment the CTA opens (with kDirectQ, after its
      // first: those of the first the consumers load themselves)
      const bool with_q = kDirectQ ? (i > 0 && c.k == 0) : (i == 0 || c.k == 0);
      const bool with_new = fused && c.k == chunks_of(prefix, c.s) - 1;
      const bool ok = blk >= 0 && blk < p.num_blocks;
      if (arm) {
        if (!ok) atomicOr(&g_decode_errors, kErrBlock);
        mbar_arrive_expect_tx(bar, (ok ? 2 * box : 0) + (with_q ? qbox : 0) +
                                       (with_new ? 2 * nbox : 0));
      }
      if (kv && ok) {
        const int32_t row = blk * p.block_size + unit_key(c) % p.block_size;
        tma_load_3d_hint(stage, &k_map, bar, 0, c.hg * HG, row, policy);
        tma_load_3d_hint(stage + L::kKBytes, &v_map, bar, 0, c.hg * HG, row, policy);
      }
      if (inputs) {
        if (with_q) tma_load_3d(stage + 2 * L::kKBytes, &q_map, bar, 0, c.hg * HG * G, c.s);
        if (with_new) {
          const uint32_t na = stage + 2 * L::kKBytes + L::kQBytes;
          tma_load_3d(na, &kn_map, bar, 0, c.hg * HG, c.s);
          tma_load_3d(na + L::kNewBytes, &vn_map, bar, 0, c.hg * HG, c.s);
        }
      }
    };
    // with stable inputs the K/V copies of the first stage go out before the
    // wait for the previous kernel, its q and new rows after it (one stage:
    // when every CTA sends out several stages at once, each CTA's first lands
    // later, behind the others' second and third; measured faster than two or
    // three)
    const int pre = p.stable_inputs ? min(1, n_mine) : 0;
    if (p.stable_inputs) {
      Cursor c = cur;
      for (int i = 0; i < pre; ++i) {
        issue(i, c, __shfl_sync(0xffffffffu, batch, i), true, true, false);
        __syncwarp();
        advance(c, prefix, p.num_seqs, n_groups);
      }
      griddep_wait();
    }
    for (int i = 0; i < n_mine; ++i) {
      if (i > 0 && (i & 31) == 0) {
        batch = next_batch;
        next_batch = entry_of(i + 32 + lane);
      }
      const int32_t blk = __shfl_sync(0xffffffffu, batch, i & 31);
      const int st = i % NS;
      if (i >= NS &&
          !__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, ((i / NS) - 1) & 1, &g_decode_errors))) {
        if (lane == 0) atomicOr(&g_decode_errors, kErrTimeout);
        break;
      }
      issue(i, cur, blk, i >= pre, i >= pre, true);
      __syncwarp();
      advance(cur, prefix, p.num_seqs, n_groups);
    }
    // every copy of this CTA is issued: the next kernel may start launching
    if (lane == 0) griddep_launch_dependents();
    return;
  }
  if (warp == HG + 1) {
    // ------------------------------------------------------------ store warp
    // the new tokens' K/V rows go to their cache slots: sequence s is stored by
    // CTA s mod W (nothing in this launch reads those rows from the cache)
    if (p.stable_inputs) griddep_wait();
    if (fused) {
      const int row_vec = p.num_kv_heads * (kRowBytes / 16);
      const int64_t num_slots = static_cast<int64_t>(p.num_blocks) * p.block_size;
      for (int64_t sq = cta; sq < p.num_seqs; sq += W) {
        const int64_t slot = p.slot_mapping[sq];
        if (slot == -1) continue;
        if (slot < -1 || slot >= num_slots) {
          if (lane == 0) atomicOr(&g_decode_errors, kErrSlot);
          continue;
        }
        for (int idx = lane; idx < row_vec; idx += 32) {
          p.k_cache_w[slot * row_vec + idx] = p.k_new[sq * row_vec + idx];
          p.v_cache_w[slot * row_vec + idx] = p.v_new[sq * row_vec + idx];
        }
      }
    }
    return;
  }
  if (warp > HG + 1) return;

  // -------------------------------------------------------------- consumers
  if (p.stable_inputs) griddep_wait();     // before any output or workspace write
  const int g = warp;                      // KV head within the group
  const int tok_bytes = HG * kRowBytes;    // one token row of the group in a stage
  const int sub = lane & 7, grp = lane >> 3;
  const int my_key = 4 * (sub >> 1) + grp; // key whose logit this lane holds
  const bool counts = (sub & 1) == 0;      // lanes sub, sub^1 hold the same key
  const int half = lane >> 4, vcol = lane & 15;
  float *prob = reinterpret_cast<float *>(smem + L::kProbOffset) + g * G * kChunk;
  Cursor cur = locate(prefix, p.num_seqs, n_groups, u_lo);
  // With kDirectQ the q rows of the CTA's first segment come straight from
  // global memory, loaded here while the first stage lands: a TMA copy issued
  // after the dependency wait would queue behind the K/V copies issued before
  // it.
  uint4 q_first[kDirectQ ? G : 1][2];
  if constexpr (kDirectQ) {
    const uint8_t *qg =
        p.q + (static_cast<int64_t>(cur.s) * p.num_q_heads + (cur.hg * HG + g) * G) * kRowBytes;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      q_first[h][0] = __ldg(reinterpret_cast<const uint4 *>(qg + h * kRowBytes + sub * 16));
      q_first[h][1] = __ldg(reinterpret_cast<const uint4 *>(qg + h * kRowBytes + 128 + sub * 16));
    }
  }
  uint64_t qf[G][8];  // the lane's 16 query dims per head, as scaled fp32 pairs
  float m[G], lsum[G];
  uint64_t o[G][4];   // the lane's 8 output dims per head, as fp32 pairs
  int seg_first_k = 0;
  bool seg_is_first = true;
  int ctx = 0, chunk0 = 0, key_lo = 0;  // the segment's length, first chunk and first key

#pragma unroll 1
  for (int it = 0; it < n_mine; ++it) {
    const int st = it % NS;
    const uint8_t *kst = smem + static_cast<size_t>(st) * L::kStageBytes;
    const uint8_t *vst = kst + L::kKBytes;
    const bool opens = (it == 0) || (cur.k == 0);
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, (it / NS) & 1, &g_decode_errors))) {
      if (lane == 0) atomicOr(&g_decode_errors, kErrTimeout);
      return;  // a lost copy: rows of this CTA's range stay unwritten
    }
    if (opens) {
      ctx = ctx_of[cur.s];
      chunk0 = first_chunk(ctx, p.window);
      key_lo = first_key(ctx, p.window);
      seg_first_k = cur.k;
      seg_is_first = (it == 0);
      const uint8_t *qs = kst + 2 * L::kKBytes + g * G * kRowBytes;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint4 a, b;
        if (kDirectQ && it == 0) {
          a = q_first[kDirectQ ? h : 0][0];
          b = q_first[kDirectQ ? h : 0][1];
        } else {
          a = *reinterpret_cast<const uint4 *>(qs + h * kRowBytes + sub * 16);
          b = *reinterpret_cast<const uint4 *>(qs + h * kRowBytes + 128 + sub * 16);
        }
        const uint32_t wq[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          qf[h][i] = f32x2(bf16lo(wq[i]) * p.scale_log2, bf16hi(wq[i]) * p.scale_log2);
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) o[h][i] = 0ull;
      }
    }
    const int key0 = (chunk0 + cur.k) * kChunk;   // the unit's first key
    const int nvalid = min(kChunk, ctx - key0);   // keys >= nvalid are past the context
    const int nskip = key_lo - key0;              // keys < nskip are before the window
    const bool with_new = fused && cur.k == chunks_of(prefix, cur.s) - 1;
    if (with_new) {
      // the unit holds the sequence's new token (key ctx-1): take its K and V
      // rows from the staged inputs, whatever the cache row held when copied
      const int r_new = ctx - 1 - key0;
      uint8_t *stg = smem + static_cast<size_t>(st) * L::kStageBytes;
      const uint8_t *na = stg + 2 * L::kKBytes + L::kQBytes;
      const int part = lane & 15;
      const int kv = lane >> 4;  // 0: K, 1: V
      const uint4 row = *reinterpret_cast<const uint4 *>(na + kv * L::kNewBytes + g * kRowBytes +
                                                         part * 16);
      *reinterpret_cast<uint4 *>(stg + kv * L::kKBytes + r_new * tok_bytes + g * kRowBytes +
                                 part * 16) = row;
      __syncwarp();
    }

    // ---- logits: pass pp covers keys 4*pp + grp; lane group grp, sub-dims sub
    float part[G][4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const uint8_t *krow = kst + (4 * pp + grp) * tok_bytes + g * kRowBytes;
      const uint4 ka = *reinterpret_cast<const uint4 *>(krow + sub * 16);
      const uint4 kb = *reinterpret_cast<const uint4 *>(krow + 128 + sub * 16);
      const uint32_t wv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lo[i] = wv[i] << 16;
        hi[i] = wv[i] & 0xFFFF0000u;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint64_t acc = 0ull;
#pragma unroll
        for (int i = 0; i < 8; ++i) ffma2(acc, qf[h][i], lo[i], hi[i]);
        part[h][pp] = f32x2_lo(acc) + f32x2_hi(acc);
      }
    }
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      butterfly_half<4>(part[h], (sub & 4) != 0, 4);
      float q2[2] = {part[h][0], part[h][1]};
      butterfly_half<2>(q2, (sub & 2) != 0, 2);
      const float full = q2[0] + __shfl_xor_sync(0xffffffffu, q2[0], 1);
      sc[h] = (my_key < nvalid && my_key >= nskip) ? full : -INFINITY;
    }

    // ---- online softmax over the unit (base 2), with a lazy maximum: the
    // running maximum m only moves (a warp max-reduction and a rescale of the
    // row's sum and output) when some logit exceeds it by more than 2^8;
    // otherwise probabilities up to 256 are kept as they are, exact in fp32
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (__any_sync(0xffffffffu, sc[h] > m[h] + kLazyMax)) {  // always on a first unit
        float mx = sc[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[h], mx);
        const float alpha = fast_exp2(m[h] - m_new);  // 0 on a segment's first unit
        lsum[h] *= alpha;
        const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint64_t r = 0ull;
          ffma2(r, a2, static_cast<uint32_t>(o[h][i]), static_cast<uint32_t>(o[h][i] >> 32));
          o[h][i] = r;
        }
        m[h] = m_new;
      }
      const float pr = fast_exp2(sc[h] - m[h]);  // 0 for masked keys
      lsum[h] += counts ? pr : 0.f;
      if (counts) prob[h * kChunk + my_key] = pr;
    }
    __syncwarp();

    // ---- P.V: half-warp `half` takes keys 2*pp + half, a lane covers 8 dims
    auto pv_key = [&](int key) {
      const uint4 vv =
          *reinterpret_cast<const uint4 *>(vst + key * tok_bytes + g * kRowBytes + vcol * 16);
      const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
      uint64_t pr2[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = prob[h * kChunk + key];
        pr2[h] = f32x2(pr, pr);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v0 = wv[i] << 16, v1 = wv[i] & 0xFFFF0000u;
#pragma unroll
        for (int h = 0; h < G; ++h) ffma2(o[h][i], pr2[h], v0, v1);
      }
    };
    if (nvalid == kChunk) {
      // a full unit (almost every one): fully unrolled, so that all its loads
      // can be issued ahead of the arithmetic
#pragma unroll
      for (int pp = 0; pp < kChunk / 2; ++pp) pv_key(2 * pp + half);
    } else {
#pragma unroll 4
      for (int pp = 0; pp < kChunk / 2; ++pp) {
        const int key = 2 * pp + half;
        if (2 * pp >= nvalid) break;
        if (key < nvalid) pv_key(key);
      }
    }
    // this warp is done with the stage (and with prob): release it (after its
    // own shared-memory writes, if any, are ordered before the next TMA fill)
    if (with_new) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);

    // ---- segment end: the pair's last unit, or this CTA's last unit
    const int nch = chunks_of(prefix, cur.s);
    const bool pair_ends = cur.k == nch - 1;
    if (pair_ends || it == n_mine - 1) {
      float lt[G];
      float of[G][8];
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          of[h][2 * i] = f32x2_lo(o[h][i]);
          of[h][2 * i + 1] = f32x2_hi(o[h][i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) of[h][i] += __shfl_xor_sync(0xffffffffu, of[h][i], 16);
        lt[h] = lsum[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], off);
      }
      const int kvh = cur.hg * HG + g;  // KV head
      const int64_t row0 = static_cast<int64_t>(cur.s) * p.num_q_heads + kvh * G;
      if (seg_first_k == 0 && pair_ends) {
        // the whole pair is in this segment: write the final rows
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float inv = 1.f / lt[h];
            uint4 v;
            v.x = pack_bf16x2(of[h][0] * inv, of[h][1] * inv);
            v.y = pack_bf16x2(of[h][2] * inv, of[h][3] * inv);
            v.z = pack_bf16x2(of[h][4] * inv, of[h][5] * inv);
            v.w = pack_bf16x2(of[h][6] * inv, of[h][7] * inv);
            *reinterpret_cast<uint4 *>(p.out + (row0 + h) * kD + vcol * 8) = v;
          }
        }
        if (lane == 0 && p.lse != nullptr) {
#pragma unroll
          for (int h = 0; h < G; ++h) p.lse[row0 + h] = (m[h] + log2f(lt[h])) * kLn2;
        }
      } else {
        // a piece of a pair cut by range boundaries: store the partial
        const int64_t slot = 2 * cta + (seg_is_first ? 0 : 1);
        const int64_t base = (slot * HG + g) * G;  // partial index of head h: base + h
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (base + h) * kD + vcol * 8);
            __stcg(dst, make_float4(of[h][0], of[h][1], of[h][2], of[h][3]));
            __stcg(dst + 1, make_float4(of[h][4], of[h][5], of[h][6], of[h][7]));
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            __stcg(p.ws_ml + (base + h) * 2, m[h]);
            __stcg(p.ws_ml + (base + h) * 2 + 1, lt[h]);
          }
        }
        // merged by the merge kernel that follows this one
      }
    }
    advance(cur, prefix, p.num_seqs, n_groups);
  }
}

// Chunk prefix over sequences in shared memory, as the decode kernel builds it
// (invalid lengths count as empty); one warp.
__device__ __forceinline__ void build_prefix(const DecodeParams &p, int *prefix, int lane) {
  int carry = 0;
  const int64_t ctx_cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
  for (int base = 0; base < p.num_seqs; base += 32) {
    const int s = base + lane;
    int n = 0;
    if (s < p.num_seqs) {
      const int ctx = p.context_lens[s];
      if (ctx > 0 && ctx <= p.max_context_len && ctx <= ctx_cap)
        n = (ctx + kChunk - 1) / kChunk - first_chunk(ctx, p.window);
    }
    int incl = n;
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

// Merge of the (sequence, KV head) pairs that the decode kernel's CTA ranges
// cut: one warp per pair, combining the pieces' (max, sum, output) partials.
// CTA c of the decode kernel stored its first piece in slot 2c, its last in
// slot 2c+1; the pair's first CTA holds its piece in its last slot unless its
// range starts at the pair's first unit.
template <int G>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeParams p, int32_t decode_grid) {
  extern __shared__ int merge_prefix[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // The partition depends on context lengths only, which the decode kernel
  // before this one does not write, and every kernel before that one has
  // completed (the decode kernel waited for it before it let this one
  // launch): they may be read before the wait below.
  if (warp == 0) build_prefix(p, merge_prefix, lane);
  __syncthreads();
  griddep_launch_dependents();
  const int HG = p.hg, n_groups = p.n_groups;
  const int64_t U = static_cast<int64_t>(n_groups) * merge_prefix[p.num_seqs];
  if (U == 0) return;
  const int64_t W = decode_grid < U ? decode_grid : U;
  griddep_wait();  // the decode kernel's partials are visible from here on
  // after a timeout (in the decode kernel just before this one, or in an
  // earlier launch, which made that kernel skip its work) the partials are
  // stale: write nothing, as the decode kernel did not
  if (*reinterpret_cast<volatile uint32_t *>(&g_decode_errors) & kErrTimeout) return;
  const int64_t n_pairs = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
  const int n_warps = static_cast<int>(blockDim.x >> 5);
  for (int64_t pi = static_cast<int64_t>(blockIdx.x) * n_warps + warp; pi < n_pairs;
       pi += static_cast<int64_t>(gridDim.x) * n_warps) {
    const int s = static_cast<int>(pi / p.num_kv_heads), kvh = static_cast<int>(pi % p.num_kv_heads);
    const int hg = kvh / HG, g = kvh % HG;
    const int nch = chunks_of(merge_prefix, s);
    if (nch == 0) continue;
    const int64_t P0 = static_cast<int64_t>(n_groups) * merge_prefix[s] + static_cast<int64_t>(hg) * nch;
    const int64_t wa = owner_of(P0, W, U), wb = owner_of(P0 + nch - 1, W, U);
    if (wa == wb) continue;  // written whole by the decode kernel
    const int64_t wa_slot = 2 * wa + (range_start(wa, W, U) < P0 ? 1 : 0);
    auto part = [&](int64_t x, int h) { return ((x == wa ? wa_slot : 2 * x) * HG + g) * G + h; };
    const int64_t row0 = static_cast<int64_t>(s) * p.num_q_heads + kvh * G;
    const int64_t n = wb - wa + 1;
    if (n <= kMergeFast) {
      // every load at once: lane x < n fetches piece x's (max, sum), every
      // lane its 4 output dims of each piece
      float mh[G], lh[G];
      float4 ov[kMergeFast][G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mh[h] = -INFINITY;
        lh[h] = 0.f;
        if (lane < n) {
          const int64_t i = part(wa + lane, h);
          mh[h] = p.ws_ml[i * 2];
          lh[h] = p.ws_ml[i * 2 + 1];
        }
      }
#pragma unroll
      for (int x = 0; x < kMergeFast; ++x)
#pragma unroll
        for (int h = 0; h < G; ++h)
          ov[x][h] = x < n ? reinterpret_cast<const float4 *>(p.ws_o + part(wa + x, h) * kD)[lane]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float M = mh[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float f = lane < n ? fast_exp2(mh[h] - M) : 0.f;
        float Lsum = lh[h] * f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int x = 0; x < kMergeFast; ++x) {
          const float fx = __shfl_sync(0xffffffffu, f, x);
          acc[0] = fmaf(ov[x][h].x, fx, acc[0]);
          acc[1] = fmaf(ov[x][h].y, fx, acc[1]);
          acc[2] = fmaf(ov[x][h].z, fx, acc[2]);
          acc[3] = fmaf(ov[x][h].w, fx, acc[3]);
        }
        const float inv = 1.f / Lsum;
        uint2 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(p.out + (row0 + h) * kD + lane * 4) = v;
        if (lane == 0 && p.lse != nullptr) p.lse[row0 + h] = (M + log2f(Lsum)) * kLn2;
      }
      continue;
    }
    // more pieces (long contexts cut across many CTAs): the maxima of up to
    // 32 pieces a round, one piece per lane and every head at once; then each
    // lane's weight and sum, and the outputs in batches of kMergeFast pieces
    // whose loads (all heads) are issued before any is used
    float M[G], Lsum[G], acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      M[h] = -INFINITY;
      Lsum[h] = 0.f;
      acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
    }
    for (int64_t x = wa + lane; x <= wb; x += 32)
#pragma unroll
      for (int h = 0; h < G; ++h) M[h] = fmaxf(M[h], p.ws_ml[part(x, h) * 2]);
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], off));
#pragma unroll 1
    for (int64_t base = wa; base <= wb; base += 32) {
      const int64_t x = base + lane;
      float f[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        f[h] = 0.f;
        if (x <= wb) {
          const int64_t i = part(x, h);
          f[h] = fast_exp2(p.ws_ml[i * 2] - M[h]);
          Lsum[h] += p.ws_ml[i * 2 + 1] * f[h];
        }
      }
      const int n = static_cast<int>(wb - base + 1 < 32 ? wb - base + 1 : 32);
#pragma unroll 1
      for (int j0 = 0; j0 < n; j0 += kMergeFast) {
        float4 ov[kMergeFast][G];
#pragma unroll
        for (int j = 0; j < kMergeFast; ++j)
#pragma unroll
          for (int h = 0; h < G; ++h)
            ov[j][h] = j0 + j < n ? reinterpret_cast<const float4 *>(
                                        p.ws_o + part(base + j0 + j, h) * kD)[lane]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kMergeFast; ++j)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float fj = __shfl_sync(0xffffffffu, f[h], (j0 + j) & 31);
            acc[h][0] = fmaf(ov[j][h].x, fj, acc[h][0]);
            acc[h][1] = fmaf(ov[j][h].y, fj, acc[h][1]);
            acc[h][2] = fmaf(ov[j][h].z, fj, acc[h][2]);
            acc[h][3] = fmaf(ov[j][h].w, fj, acc[h][3]);
          }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Lsum[h] += __shfl_xor_sync(0xffffffffu, Lsum[h], off);
      const float inv = 1.f / Lsum[h];
      uint2 v;
      v.x = pack_bf16x2(acc[h][0] * inv, acc[h][1] * inv);
      v.y = pack_bf16x2(acc[h][2] * inv, acc[h][3] * inv);
      *reinterpret_cast<uint2 *>(p.out + (row0 + h) * kD + lane * 4) = v;
      if (lane == 0 && p.lse != nullptr) p.lse[row0 + h] = (M[h] + log2f(Lsum[h])) * kLn2;
    }
  }
}

template <int G, int HGM, int NS>
cudaError_t launch_variant(const DecodeArgs &a, const CUtensorMap &k_map,
                           const CUtensorMap &v_map, const CUtensorMap &q_map,
                           const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                           const DecodeParams &p, cudaStream_t stream) {
  using L = DecodeSmem<G, HGM, NS>;
  static_assert(L::total(kDecodeMaxSeqs) <= 227 * 1024, "decode shared memory");
  auto kern = decode_kernel<G, HGM, NS>;
  const int smem = L::total(a.num_seqs);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(a.grid), dim3((p.hg + 2) * 32), smem, stream, k_map, v_map, q_map,
                 kn_map, vn_map, p);
  if (e != cudaSuccess) return e;
  const int64_t n_pairs = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  const int merge_warps = n_pairs >= kMergeWideMin ? kMergeWarps : kMergeWarpsFew;
  const int merge_grid = static_cast<int>((n_pairs + merge_warps - 1) / merge_warps);
  return launch_pdl(decode_merge_kernel<G>, dim3(merge_grid), dim3(merge_warps * 32),
                    sizeof(int) * static_cast<size_t>(a.num_seqs + 1), stream, p, a.grid);
}

template <int G>
cudaError_t launch_group(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                         const CUtensorMap &q_map, const CUtensorMap &kn_map,
                         const CUtensorMap &vn_map, const DecodeParams &p, cudaStream_t stream) {
  // three stages when they fit in shared memory, else two
  constexpr int kDefaultStages = DecodeSmem<G, 8, 3>::total(kDecodeMaxSeqs) <= 227 * 1024 ? 3 : 2;
  switch (a.variant) {
    case 1: return launch_variant<G, 8, 2>(a, k_map, v_map, q_map, kn_map, vn_map, p, stream);
    case 2: return launch_variant<G, 4, 2>(a, k_map, v_map, q_map, kn_map, vn_map, p, stream);
    default:
      return launch_variant<G, 8, kDefaultStages>(a, k_map, v_map, q_map, kn_map, vn_map, p,
                                                  stream);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, const CUtensorMap &q_map,
                          const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                          cudaStream_t stream) {
  DecodeParams p;
  p.q = static_cast<const uint8_t *>(a.q);
  p.k_new = static_cast<const uint4 *>(a.k_new);
  p.v_new = static_cast<const uint4 *>(a.v_new);
  p.k_cache_w = static_cast<uint4 *>(a.k_cache_w);
  p.v_cache_w = static_cast<uint4 *>(a.v_cache_w);
  p.slot_mapping = a.slot_mapping;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.max_blocks = a.max_blocks;
  p.max_context_len = a.max_context_len;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.hg = decode_group_heads(a.num_kv_heads, decode_variant_group_max(a.variant));
  p.n_groups = a.num_kv_heads / p.hg;
  p.window = a.window;
  p.stable_inputs = a.stable_inputs ? 1 : 0;
  p.scale_log2 = a.scale_log2;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_group<1>(a, k_map, v_map, q_map, kn_map, vn_map, p, stream);
    case 2: return launch_group<2>(a, k_map, v_map, q_map, kn_map, vn_map, p, stream);
    case 4: return launch_group<4>(a, k_map, v_map, q_map, kn_map, vn_map, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t decode_error_word(uint32_t **word) {
  return cudaGetSymbolAddress(reinterpret_cast<void **>(word), g_decode_errors);
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
