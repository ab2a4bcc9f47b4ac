// Varlen causal prefill attention over the paged KV cache, on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Serves both plain prompts (Lq == Lk) and prompts whose leading blocks are
// already cached (prefix caching: "nano-vllm-sansho" README, "Key Features";
// "How lunaryes/nano-vllm works", where the block manager hands out cached
// blocks). Query i of a segment sees keys p <= Lk - Lq + i.
//
// One CTA owns two 128-row query tiles that share every K/V tile: with grouped
// queries (H_q / H_kv >= 2) the two query heads of a head pair over the same
// 128 rows; without grouping, two consecutive row tiles of one head. 12 warps:
//   warp 0     TMA producer: both Q tiles once, then K and V tiles of 128 keys,
//              two stages deep, 128-byte swizzled; V of step j and K of step
//              j+1 go out together once the MMA warp's release of step j-1
//              has freed both their stages. A tile is copied as boxes of
//              the largest of 128, 64, 32, 16 rows that divides the block size
//              (a box never crosses a cache block): fewer, larger copies
//              (one 128-row box per column half streams from L2 about twice
//              as fast per SM as eight 16-row boxes).
//   warp 1     MMAs (the whole warp runs the loop, one elected lane issues).
//              TMEM holds S_t (128 fp32 columns) and O_t (128) for
//              each tile t. Per KV tile j and query tile t: S_t = Q_t K_j^T
//              (A and B from shared memory), then, once the softmax has
//              written P_t (bf16) over the first 64 columns of S_t,
//              O_t += P_t V_j with A read straight from TMEM. S_t(j+1) is
//              issued after P.V(j), and MMAs run in issue order, so a
//              completed S_t(j+1) also means O_t holds every tile up to j.
//              The V rows past the segment's last key are zeroed before their
//              first P.V, so stale or poisoned rows never meet a zero
//              probability.
//   warps 4-7  softmax of tile 0, warps 8-11 softmax of tile 1: one query row
//              per thread (TMEM lane = row). Read the S row, mask, online
//              softmax in base 2 (the O row in TMEM is rescaled only in tiles
//              where some row's maximum grows), write P back into TMEM; at the
//              end normalise O and store the bf16 output (through a staging
//              area per warp, so that each store writes whole row halves) and
//              the natural-log lse.
// While one tile's softmax runs, the tensor pipe works on the other tile.
//
// Two kernels share this design. Without a sliding window, prefill_kernel
// runs one CTA per work item (two query tiles); with one, where an item is
// only two or three KV steps, prefill_persistent_kernel runs one CTA per SM
// that walks its share of the items, so that the set-up, the TMEM allocation
// and the pipeline's fill and drain are paid once per SM rather than once per
// item. (The persistent walk measured slower on long items, so the first
// kernel stays for them.)
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

static __device__ uint32_t g_prefill_errors;

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                       // query rows per tile
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kTiles = 2;                      // query tiles per CTA
constexpr int kHalfBytes = 128 * 128;          // 128 rows x 64 bf16 (one swizzle column group)
constexpr int kTileBytes = 2 * kHalfBytes;     // 128 rows x 128 bf16
constexpr int kStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTiles * kTileBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
constexpr int kBarOff = kVOff + kStages * kTileBytes;
// barrier slots (8 bytes each)
// kBarK0: K of the first KV step (of the CTA, or of each item of the
// persistent kernel); kBarKV + (g & 1): V of step g and K of step g + 1, when
// that step belongs to the same item; kBarRel + (r & 1): release r, the MMA
// warp's commit after the S MMAs of step r, which frees K(r) and V(r - 1);
// kBarVTail + st: the item's last V tile in stage st, its rows past the
// segment's end zeroed; kBarQEmpty: the item's S MMAs are done with Q;
// kBarDone: every MMA of the CTA has completed
constexpr int kBarQ = 0, kBarK0 = 1, kBarKV = 2, kBarRel = 4, kBarS = 6, kBarP = 8, kBarO = 10,
              kBarVTail = 12, kBarQEmpty = 14, kBarDone = 15, kNumBars = 16;
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kAbortOff = kTmemSlotOff + 8;
// the persistent kernel's current item as the MMA issuer needs it, published
// by the producer before it arms the item's Q barrier: int [4] = steps of
// tiles 0 and 1, KV steps (0: no more items), 1 if the last KV tile extends
// past the segment's last key
constexpr int kItemOff = kAbortOff + 8;
// the output staging areas of the eight softmax warps: 32 rows of 128 bytes
constexpr int kEpiWarpBytes = 32 * 128;
constexpr int kEpiOff = (kItemOff + 32 + 127) / 128 * 128;
constexpr int kSmemBytes = kEpiOff + 8 * kEpiWarpBytes + 1024;  // + slack for 1024-byte alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// warp 0 TMA producer, warp 1 MMAs, warps 2-3 idle, warps 4-11 softmax
// (warpgroup 1 + t for query tile t): three warpgroups, so that setmaxnreg can
// move registers from the first to the two softmax warpgroups. The producer
// and MMA warps come first because the warp scheduler, choosing among ready
// warps of one SM sub-partition, favours the lower-numbered ones: the MMA
// warp shares its sub-partition with two busy softmax warps, and every cycle
// it waits for an issue slot delays the tensor pipe.
constexpr int kThreads = 384;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kSoftmaxWarp0 = 4;
// registers per thread after the split, 2 * softmax + other = 3 * 168 (the
// launch's share per thread of the 64K register file for 384 threads); the
// same in both kernels (the persistent one's producer and MMA warp, which
// reads each item from shared memory, fit in 72 without spills)
struct RegSplit {
  static constexpr int kSoftmax = 216;
  static constexpr int kOther = 72;
  static_assert(2 * kSoftmax + kOther == 3 * 168, "register split");
};
constexpr uint32_t kTmemCols = 512;            // S0, S1, O0, O1: 128 columns each
constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);  // A=Q K-major, B=K K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, 0, 1);   // A=P (TMEM), B=V MN-major
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLazyMax = 8.0f;  // log2 units the running maximum may lag
constexpr float kLazyBound = 256.0f;  // 2^kLazyMax: the largest tile sum taken as is
static_assert(kLazyBound == 256.0f && kLazyMax == 8.0f, "kLazyBound is 2^kLazyMax");

struct PrefillParams {
  const int32_t *cu_q, *cu_k, *block_tables;
  __nv_bfloat16 *out;
  float *lse;
  int32_t max_blocks, num_seqs, total_q, max_seqlen_q, max_seqlen_k;
  int32_t num_q_heads, num_kv_heads, block_size, num_blocks;
  int32_t n_rowtiles, n_pairs, n_items;  // the item list: row tiles x head pairs x sequences
  int32_t window;    // sliding window in keys (0: none)
  int32_t box_rows;  // rows per K/V box: 16, 32, 64 or 128, dividing block_size
  float scale_log2;
};

__device__ __forceinline__ bool wait_(uint32_t bar, uint32_t parity, const volatile int *abort) {
  return mbar_wait(bar, parity, &g_prefill_errors, abort);
}

__device__ __forceinline__ void fail(volatile int *abort) {
  *abort = 1;
  atomicOr(&g_prefill_errors, kErrTimeout);
}

// The warp's 32 normalised O rows (its TMEM lane quadrant, 128 fp32 columns)
// as bf16 rows in global memory: row i of the warp goes to out_w + i *
// row_stride, for i < n_valid. Each thread holds one row and rows lie
// row_stride elements apart, so a store straight from registers writes 32
// lines per instruction. The rows go through the warp's staging area (scr,
// 32 rows of 128 bytes, one column half at a time) instead: written one row
// per thread, read back so that each store writes four whole 128-byte row
// halves. A 16-byte chunk c of row i sits at position c ^ (i & 7), which
// keeps both sides free of shared-memory bank conflicts.
__device__ __forceinline__ void store_o_rows(uint32_t tO, float inv_l, uint32_t scr,
                                             __nv_bfloat16 *out_w, int64_t row_stride,
                                             int n_valid, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t o[32];
      tmem_ld32(tO + h * 64 + q * 32, o);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w0 = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l,
                                        __uint_as_float(o[8 * k + 1]) * inv_l);
        const uint32_t w1 = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l,
                                        __uint_as_float(o[8 * k + 3]) * inv_l);
        const uint32_t w2 = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l,
                                        __uint_as_float(o[8 * k + 5]) * inv_l);
        const uint32_t w3 = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l,
                                        __uint_as_float(o[8 * k + 7]) * inv_l);
        const uint32_t addr = scr + lane * 128 + (((q * 4 + k) ^ (lane & 7)) * 16);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1),
                     "r"(w2), "r"(w3)
                     : "memory");
      }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = 4 * i + (lane >> 3), c = lane & 7;
      uint4 v;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(scr + row * 128 + ((c ^ (row & 7)) * 16))
                   : "memory");
      if (row < n_valid)
        *reinterpret_cast<uint4 *>(out_w + row * row_stride + h * 64 + c * 8) = v;
    }
    __syncwarp();
  }
}

// One work item: two 128-row query tiles that share every K/V tile. With
// grouped queries (H_q / H_kv >= 2) the two query heads of a head pair over
// the same 128 rows; without grouping, two consecutive row tiles of one head.
struct Item {
  int s, q0, Lq, Lk, diag, g;
  int head[kTiles], row0[kTiles];
  int n_tiles[kTiles];  // KV tiles 0 .. n_tiles[t] - 1 hold the keys of tile t (0: no rows)
  int j_start;          // first KV tile any of the rows sees (sliding window)
  int n_steps;          // KV tiles j_start .. j_start + n_steps - 1
};

// Item `lin` of the list, heaviest first: row tiles from the last (which see
// the most keys) to the first, each over all head pairs and sequences. False
// for an item without work (rows past the segment, or lengths that fail the
// checks, which `raise` reports once per sequence).
template <bool kWindowed>
__device__ __forceinline__ bool make_item(const PrefillParams &p, int lin, bool raise, Item &it) {
  const int per_rt = p.n_pairs * p.num_seqs;
  const int rt = p.n_rowtiles - 1 - lin / per_rt;
  const int pair = (lin % per_rt) % p.n_pairs;
  it.s = (lin % per_rt) / p.n_pairs;
  const int G = p.num_q_heads / p.num_kv_heads;
  it.q0 = p.cu_q[it.s];
  const int q1 = p.cu_q[it.s + 1];
  it.Lq = q1 - it.q0;
  it.Lk = p.cu_k[it.s + 1] - p.cu_k[it.s];
  if (it.q0 < 0 || it.Lq < 0 || it.Lk < it.Lq || it.Lq > p.max_seqlen_q ||
      it.Lk > p.max_seqlen_k || q1 > p.total_q ||
      static_cast<int64_t>(it.Lk) > static_cast<int64_t>(p.max_blocks) * p.block_size) {
    if (raise && rt == p.n_rowtiles - 1 && pair == 0) atomicOr(&g_prefill_errors, kErrSeqlens);
    return false;
  }
  if (G >= 2) {
    it.head[0] = 2 * pair;
    it.head[1] = 2 * pair + 1;
    it.row0[0] = it.row0[1] = rt * kBM;
  } else {
    it.head[0] = it.head[1] = pair;
    it.row0[0] = 2 * rt * kBM + kBM;  // the later (heavier) row tile first
    it.row0[1] = 2 * rt * kBM;
  }
  it.g = it.head[0] / G;
  it.diag = it.Lk - it.Lq;  // query i sees keys <= diag + i
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    if (it.row0[t] >= it.Lq) {
      it.n_tiles[t] = 0;
    } else {
      const int kv_end = it.diag + min(it.Lq, it.row0[t] + kBM);  // keys the tile needs (<= Lk)
      it.n_tiles[t] = (kv_end + kBN - 1) / kBN;
    }
  }
  const int n_max = max(it.n_tiles[0], it.n_tiles[1]);
  // With a sliding window query i sees keys >= diag + i - window + 1: the KV
  // tiles before the one that holds the earliest such key of the item's rows
  // are skipped.
  it.j_start = 0;
  if constexpr (kWindowed) {
    int lo = it.Lk;
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if (it.n_tiles[t] > 0) lo = min(lo, max(0, it.diag + it.row0[t] - p.window + 1));
    it.j_start = lo / kBN;
  }
  it.n_steps = n_max - it.j_start;
  return n_max > 0;
}

// This CTA's items in order: CTA c of C takes items c, 2C - 1 - c, 2C + c, ...
// of the heaviest-first list (rounds alternate direction, so that every CTA
// gets a similar mix of heavy and light items).
template <bool kWindowed>
struct ItemWalk {
  int k = 0;         // next round to look at
  int item_no = -1;  // index of the current item among this CTA's items with work
  // The next item with work into `it`; false when there is none.
  __device__ __forceinline__ bool next(const PrefillParams &p, bool raise, Item &it) {
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    for (;;) {
      const int lin = k * C + ((k & 1) ? C - 1 - c : c);
      ++k;
      if (lin >= p.n_items) return false;
      if (make_item<kWindowed>(p, lin, raise, it)) {
        ++item_no;
        return true;
      }
    }
  }
};

// Without a sliding window: one CTA per item, CTA c taking item c of the
// heaviest-first list (the hardware hands CTAs to SMs as they free up, which
// balances these long items). Calls with a window run
// prefill_persistent_kernel.
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA -> (sequence, head pair, row tile): the heaviest row tiles (the last
  // ones, which see the most keys) of every head pair and sequence first, the
  // lightest last, so that the grid's tail holds the shortest CTAs.
  // (a 3-D grid (row tiles, head pairs, sequences) where its dimensions fit,
  // else a 1-D one: the same linear index either way; the 3-D grid's CTA
  // order measured about 1 % faster)
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int per_rt = p.n_pairs * p.num_seqs;  // items per row tile index
  const int rt = p.n_rowtiles - 1 - lin / per_rt;
  const int pair = (lin % per_rt) % p.n_pairs;
  const int s = (lin % per_rt) / p.n_pairs;
  const int G = p.num_q_heads / p.num_kv_heads;

  griddep_wait();  // inputs written by the previous kernel are visible from here on
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
    if (rt == p.n_rowtiles - 1 && pair == 0 && tid == 0) atomicOr(&g_prefill_errors, kErrSeqlens);
    return;
  }
  // the two query tiles: (head, first row) each; heaviest row tiles first
  int head[kTiles], row0[kTiles];
  if (G >= 2) {
    head[0] = 2 * pair;
    head[1] = 2 * pair + 1;
    row0[0] = row0[1] = rt * kBM;
  } else {
    head[0] = head[1] = pair;
    row0[0] = 2 * rt * kBM + kBM;  // the later (heavier) row tile first
    row0[1] = 2 * rt * kBM;
  }
  const int g = head[0] / G;
  const int diag = Lk - Lq;  // query i sees keys <= diag + i
  int n_tiles[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    if (row0[t] >= Lq) {
      n_tiles[t] = 0;
    } else {
      const int kv_end = diag + min(Lq, row0[t] + kBM);  // keys this tile needs (<= Lk)
      n_tiles[t] = (kv_end + kBN - 1) / kBN;
    }
  }
  const int n_max = max(n_tiles[0], n_tiles[1]);
  if (n_max == 0) return;
  // steps jj = 0 .. n_steps - 1 cover KV tiles j_start + jj (the form the
  // persistent kernel shares, where a window may skip leading tiles)
  const int j_start = 0;
  const int n_steps = n_max - j_start;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kQOff, sK = sbase + kKOff, sV = sbase + kVOff;
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile int *abort = reinterpret_cast<volatile int *>(smem + kAbortOff);

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarVTail), 1);
    mbar_init(bar(kBarK0), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKV + i), 1);
      mbar_init(bar(kBarRel + i), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(bar(kBarS + t), 1);
      mbar_init(bar(kBarP + t), kBM);
      mbar_init(bar(kBarO + t), 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(sbase + kTmemSlotOff, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kTmemSlotOff);

  if (warp < kSoftmaxWarp0) {
    setmaxnreg_dec<RegSplit::kOther>();
    if (warp == kProducerWarp) {
      // ------------------------------------------------------------ TMA producer
      // Lane b < kBN / box_rows owns the b-th box of every KV tile: it reads
      // that box's block-table entry a tile ahead of its copy (the read
      // overlaps the wait for a free stage) and issues the box's copies; lane 0
      // arms the barriers. One release per step (the MMA warp's commit that
      // closes step r) frees both K(r), after its last S = Q K(r)^T, and
      // V(r - 1), after its last P.V. K(0) goes first, on its own barrier;
      // then step j's copies, V(j) and K(j + 1), wait for release j - 1 (which
      // frees both their stages) and share one barrier, so that the MMA warp
      // waits once per step for its K and V.
      const int box_rows = p.box_rows;
      const int n_boxes = kBN / box_rows;
      if (lane == 0) {
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < kTiles; ++t) qbytes += n_tiles[t] > 0 ? kTileBytes : 0;
        mbar_arrive_expect_tx(bar(kBarQ), qbytes);
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          if (n_tiles[t] == 0) continue;
          tma_load_3d(sQ + t * kTileBytes, &q_map, bar(kBarQ), 0, head[t], q0 + row0[t]);
          tma_load_3d(sQ + t * kTileBytes + kHalfBytes, &q_map, bar(kBarQ), 64, head[t],
                      q0 + row0[t]);
        }
      }
      const int32_t *table = p.block_tables + static_cast<int64_t>(s) * p.max_blocks;
      auto box_key = [&](int j) { return j * kBN + lane * box_rows; };
      auto has_box = [&](int j) { return lane < n_boxes && j < n_max && box_key(j) < Lk; };
      auto blk_of = [&](int j) {
        return has_box(j) ? __ldg(table + box_key(j) / p.block_size) : -1;
      };
      // cache row of this lane's box in KV tile j (-1: none; a block outside
      // the pool is reported and its box left out)
      auto row_of = [&](int j, int32_t blk) -> int32_t {
        if (!has_box(j)) return -1;
        if (blk < 0 || blk >= p.num_blocks) {
          atomicOr(&g_prefill_errors, kErrBlock);
          return -1;
        }
        return blk * p.block_size + box_key(j) % p.block_size;
      };
      auto tile_bytes = [&](int32_t row) {
        return __popc(__ballot_sync(0xffffffffu, row >= 0)) * 2u * box_rows * 128u;
      };
      int32_t row_cur = row_of(j_start, blk_of(j_start));  // KV tile of step jj
      int32_t blk_nxt = blk_of(j_start + 1);               // and its successor's entry
      {
        const uint32_t bytes = tile_bytes(row_cur);
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarK0), bytes);
        __syncwarp();
        if (row_cur >= 0) {
          const uint32_t kdst = sK + lane * box_rows * 128;
          tma_load_3d(kdst, &k_map, bar(kBarK0), 0, g, row_cur);
          tma_load_3d(kdst + kHalfBytes, &k_map, bar(kBarK0), 64, g, row_cur);
        }
      }
      bool good = true;
      for (int jj = 0; jj < n_steps; ++jj) {
        const int j = j_start + jj;
        const int32_t row_nxt = row_of(j + 1, blk_nxt);  // -1 past the last tile
        blk_nxt = blk_of(j + 2);
        const uint32_t bytes = tile_bytes(row_cur) + tile_bytes(row_nxt);
        if (jj >= 1 &&
            !__all_sync(0xffffffffu,
                        wait_(bar(kBarRel + ((jj - 1) & 1)), ((jj - 1) >> 1) & 1, abort))) {
          good = false;
          break;
        }
        const uint32_t b = bar(kBarKV + (jj & 1));
        if (lane == 0) mbar_arrive_expect_tx(b, bytes);
        __syncwarp();
        if (row_cur >= 0) {
          const uint32_t vdst = sV + (jj & 1) * kTileBytes + lane * box_rows * 128;
          tma_load_3d(vdst, &v_map, b, 0, g, row_cur);
          tma_load_3d(vdst + kHalfBytes, &v_map, b, 64, g, row_cur);
        }
        if (row_nxt >= 0) {
          const uint32_t kdst = sK + ((jj + 1) & 1) * kTileBytes + lane * box_rows * 128;
          tma_load_3d(kdst, &k_map, b, 0, g, row_nxt);
          tma_load_3d(kdst + kHalfBytes, &k_map, b, 64, g, row_nxt);
        }
        row_cur = row_nxt;
      }
      // every copy of this CTA is issued: the next kernel may start launching
      if (lane == 0) griddep_launch_dependents();
      // V rows of the last tile past the segment's last key (poison in a
      // partly used box, stale data in boxes not loaded) are zeroed once the
      // tile has landed, so that they never meet a zero probability
      const int tail_r0 = Lk - (n_max - 1) * kBN;
      if (good && tail_r0 < kBN) {
        const int st = (n_steps - 1) & 1;
        good = __all_sync(0xffffffffu, wait_(bar(kBarKV + st), ((n_steps - 1) >> 1) & 1, abort));
        if (good) {
          const uint32_t vbase = sV + st * kTileBytes;
          const int n16 = (kBN - tail_r0) * 16;  // 16-byte pieces over both column halves
          for (int idx = lane; idx < n16; idx += 32) {
            const int row = tail_r0 + idx / 16, piece = idx % 16;
            const uint32_t addr = vbase + (piece / 8) * kHalfBytes + row * 128 + (piece % 8) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(0u), "r"(0u),
                         "r"(0u), "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarVTail));
        }
      }
      // wait for the last release of each slot, so that no arrival from the
      // tensor core reaches this CTA's shared memory after it has exited
      for (int r = max(n_steps - 1, 0); good && r <= n_steps; ++r)
        good = __all_sync(0xffffffffu, wait_(bar(kBarRel + (r & 1)), (r >> 1) & 1, abort));
      if (!good && lane == 0) fail(abort);
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop and its waits, so that its control flow
      // stays warp-uniform; one elected lane (lane 0, always the same one, as
      // a commit covers the MMAs its own thread issued) issues every MMA and
      // commit. A lone thread in its own branch measured about 200 cycles
      // slower per group of eight MMAs, and slower still beside busy softmax
      // warps, which share this warp's SM sub-partition.
      // K, V and Q arrive by TMA (the barrier's completion orders them before
      // the MMAs); P is written by other threads' tcgen05.st, so its wait is
      // followed by the tcgen05 fence that pairs with theirs.
      // Steps are counted from the CTA's first KV tile (j_start); query tile t
      // has steps 0 .. n_tiles[t] - j_start - 1 (none if that is not positive).
      auto wait_all = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_(b, parity, abort));
      };
      // Q and K(0) first; then at the head of step jj one wait covers V(jj - 1)
      // and K(jj), which the producer copies on one barrier
      bool good = wait_all(bar(kBarQ), 0) && wait_all(bar(kBarK0), 0);
      // The operand descriptors are 32-bit low halves over one common high half
      // (all have a 1024-byte stride between 8-row groups and 128-byte
      // swizzle). Every one differs from Q's first by a constant (its offset
      // / 16 in the start-address field, the low 14 bits, which no
      // shared-memory address carries out of; for V also the larger leading
      // byte offset, bits 16-29), so the warp keeps one base and each MMA adds
      // an immediate.
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(sQ, 16, 1024) >> 32);
      const uint32_t q_lo0 = static_cast<uint32_t>(smem_desc_sw128(sQ, 16, 1024));
      constexpr uint32_t kVLbo = static_cast<uint32_t>((kHalfBytes - 16) >> 4) << 16;
      auto desc = [&](int off) { return q_lo0 + static_cast<uint32_t>(off >> 4); };
      auto issue_s = [&](int t, int jj) {
        const int st = jj & 1;
        const uint32_t tS = tmem + t * kBN;
        const uint32_t qd = desc(kQOff + t * kTileBytes);
        const uint32_t kd = desc(kKOff + st * kTileBytes);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off16 = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tS, qd + off16, kd + off16, desc_hi, kIdescQK, kk > 0);
          }
          mma_commit(bar(kBarS + t));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int jj) -> bool {
        const int st = jj & 1;
        // P_t of this step is in TMEM once the softmax of tile t has arrived
        if (!wait_all(bar(kBarP + t), jj & 1)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + t * kBN;             // P over the first 64 columns of S_t
        const uint32_t tO = tmem + 2 * kBN + t * kD;
        const uint32_t vd = desc(kVOff + st * kTileBytes) + kVLbo;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_bf16_ts(tO, tP + kk * 8, vd + ((kk * 16 * 128) >> 4), desc_hi, kIdescPV,
                        (jj > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(kBarO + t));
        }
        __syncwarp();
        return true;
      };
      for (int t = 0; good && t < kTiles; ++t)
        if (n_tiles[t] - j_start > 0) issue_s(t, 0);
      // Release r (slot r & 1 of the kBarRel pair) closes step r: K of
      // step r has had its last S and V of step r - 1 its last P.V. Release 0
      // follows the S MMAs of step 0.
      if (good) {
        if (elect_one()) mma_commit(bar(kBarRel));
        __syncwarp();
      }
      for (int jj = 1; good && jj <= n_steps; ++jj) {
        // V(jj - 1) and K(jj) are resident; the producer zeroes the tail of
        // the segment's last KV tile, which comes with no K
        const int b = jj - 1;
        const bool tail = Lk - (j_start + b) * kBN < kBN;
        good = tail ? wait_all(bar(kBarVTail), 0)
                    : wait_all(bar(kBarKV + (b & 1)), (b >> 1) & 1);
        // finish step jj-1 for every query tile, starting step jj where needed
        for (int t = 0; good && t < kTiles; ++t) {
          if (b >= n_tiles[t] - j_start) continue;
          good = issue_pv(t, b);
          if (good && jj < n_tiles[t] - j_start) issue_s(t, jj);
        }
        if (good) {
          if (elect_one()) mma_commit(bar(kBarRel + (jj & 1)));
          __syncwarp();
        }
      }
      if (!good && lane == 0) fail(abort);
    }
  } else {
    setmaxnreg_inc<RegSplit::kSoftmax>();
    // ------------------------------------------------------------ softmax / epilogue
    const int t = (warp - kSoftmaxWarp0) >> 2;  // query tile of this warpgroup
    const int quad = warp & 3;              // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;         // row within the tile == TMEM lane
    const int n_t = n_tiles[t] > 0 ? n_tiles[t] - j_start : 0;  // steps of this tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + t * kBN + lane_off;
    const uint32_t tO = tmem + 2 * kBN + t * kD + lane_off;
    const int qi = row0[t] + r;             // query index within the segment
    const int lim = diag + qi;              // last key this row may see

    // Running maximum m (log2 units) and two running sums: l of the fp32
    // probabilities, for the lse, and lr of the same probabilities rounded to
    // bf16 as the P.V product sees them, which normalises the output. The
    // maximum is lazy: a row keeps its m while a tile's probabilities sum to
    // at most 2^kLazyMax, so no probability exceeds that bound and O is
    // rescaled only when some row of the warp passes it. Dividing by
    // the sum of the rounded probabilities keeps the output a convex
    // combination of the V rows with the weights the tensor core used, so a
    // large probability rounded to bf16 costs no more than it does under an
    // exact maximum.
    float m = 0.f, l = 0.f, lr = 0.f;
    bool good = true;
    const uint64_t scl = f32x2(p.scale_log2, p.scale_log2);
    for (int jj = 0; jj < n_t; ++jj) {
      if (!__all_sync(0xffffffffu, wait_(bar(kBarS + t), jj & 1, abort))) {
        good = false;
        break;
      }
      tc_fence_after();
      const int kbase = (j_start + jj) * kBN;
      uint32_t x[kBN];
#pragma unroll
      for (int c = 0; c < kBN; c += 32)
        tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&x[c]));
      tmem_wait_ld();
      // keys past the row's causal limit or the segment end are masked (their
      // logit becomes -inf, their probability 0); only the diagonal and the
      // tail tiles have any
      if ((kbase + kBN - 1 > diag + row0[t]) || (kbase + kBN > Lk)) {
        const int keep = min(lim, Lk - 1) - kbase + 1;  // columns < keep are at or before the limit
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= keep) x[c] = 0xFF800000u;
      }
      // P = 2^(x * scale - mm), packed two per column over the first 64
      // columns of S_t (all of S is already in registers); ts and tr get the
      // tile's sums of the fp32 and of the bf16-rounded probabilities
      auto exps = [&](float mm, float &ts, float &tr) {
        const uint64_t nm = f32x2(-mm, -mm);
        uint64_t s0 = 0, s1 = 0;
        float r0l = 0.f, r0h = 0.f, r1l = 0.f, r1h = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int k = hf * 64 + 2 * c;
            const uint64_t e =
                fma2(f32x2(__uint_as_float(x[k]), __uint_as_float(x[k + 1])), scl, nm);
            const float p0 = fast_exp2(f32x2_lo(e)), p1 = fast_exp2(f32x2_hi(e));
            pk[c] = pack_bf16x2(p0, p1);
            if (c & 1) {
              add2(s1, f32x2(p0, p1));
              add_bf16x2_to_f32(r1l, r1h, pk[c]);
            } else {
              add2(s0, f32x2(p0, p1));
              add_bf16x2_to_f32(r0l, r0h, pk[c]);
            }
          }
          tmem_st32(tS + hf * 32, pk);
        }
        add2(s0, s1);
        ts = f32x2_lo(s0) + f32x2_hi(s0);
        tr = (r0l + r1l) + (r0h + r1h);
      };
      // First with the row's current maximum, without looking for a larger
      // one: if no row of the warp then has a tile sum above 2^kLazyMax, no
      // probability exceeds that bound either and the tile is done. Otherwise
      // (some logit lies more than a little above m; an infinite sum included)
      // the warp takes the exact maximum, rescales O and recomputes P over
      // what it wrote. The first tile of a row always takes the maximum.
      float ts, tr;
      bool exact = jj == 0;
#pragma unroll 1
      for (;;) {
        if (exact) {
          // row max of the raw logits (the scale is positive): eight chains
          // of three-input maxima
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(x[i]);
#pragma unroll
          for (int c = 8; c < kBN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              a[i] = fmax3(a[i], __uint_as_float(x[c + i]), __uint_as_float(x[c + 8 + i]));
          const float mx =
              fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
          const float mxs = mx * p.scale_log2;  // -inf stays -inf
          if (jj == 0) {
            // nothing is in O yet; every row sees key 0
            m = mxs;
          } else {
            // P.V of the previous step is complete (this S was issued after
            // it): rescale the O rows in TMEM. The accesses are warp-wide, so
            // the whole warp takes its new maxima.
            const float m_new = fmaxf(m, mxs);
            const float alpha = fast_exp2(m - m_new);
            // 32 columns at a time: all of S is held in registers meanwhile
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
              uint32_t o[32];
              tmem_ld32(tO + c, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + c, o);
            }
            tmem_wait_st();
            l *= alpha;
            lr *= alpha;
            m = m_new;
          }
        }
        exps(m, ts, tr);
        if (exact || !__any_sync(0xffffffffu, !(ts <= kLazyBound))) break;
        exact = true;
      }
      l += ts;
      lr += tr;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarP + t));
    }
    if (n_t > 0 &&
        __all_sync(0xffffffffu, good && wait_(bar(kBarO + t), (n_t - 1) & 1, abort))) {
      tc_fence_after();
      const float inv_l = 1.f / lr;
      const bool store = qi < Lq;
      const int qw = row0[t] + quad * 32;  // query of the warp's first row
      store_o_rows(tO, inv_l, sbase + kEpiOff + (warp - kSoftmaxWarp0) * kEpiWarpBytes,
                   p.out + (static_cast<int64_t>(q0 + qw) * p.num_q_heads + head[t]) * kD,
                   static_cast<int64_t>(p.num_q_heads) * kD, min(32, Lq - qw), lane);
      if (store && p.lse != nullptr)
        p.lse[static_cast<int64_t>(q0 + qi) * p.num_q_heads + head[t]] = (m + log2f(l)) * kLn2;
    } else if (n_t > 0 && r == 0) {
      fail(abort);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// Persistent: one CTA per SM walks its items. Used with a sliding window,
// where an item is two or three KV steps and a CTA's fixed cost (a few
// microseconds of set-up, pipeline fill and drain) would otherwise rival its
// work. Barrier phases run on across items: the K/V, release and V-tail
// barriers count the CTA's KV steps, the S, P and O barriers of tile t count
// that tile's steps, the Q and first-K barriers count items. The next item's Q is loaded once every S MMA of the current item has
// completed (kBarQEmpty), its first S MMAs follow the current item's last
// P.V in issue order, and its first P.V (which overwrites O) waits for the
// softmax warps' P, which they write only after reading the current O.
template <bool kWindowed>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_persistent_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kQOff, sK = sbase + kKOff, sV = sbase + kVOff;
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile int *abort = reinterpret_cast<volatile int *>(smem + kAbortOff);

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarQEmpty), 1);
    mbar_init(bar(kBarK0), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKV + i), 1);
      mbar_init(bar(kBarRel + i), 1);
      mbar_init(bar(kBarVTail + i), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(bar(kBarS + t), 1);
      mbar_init(bar(kBarP + t), kBM);
      mbar_init(bar(kBarO + t), 1);
    }
    mbar_init(bar(kBarDone), 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(sbase + kTmemSlotOff, kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();  // inputs written by the previous kernel are visible from here on
  tc_fence_before();
  // a CTA gave up waiting (in this or an earlier launch): skip the work until
  // the error word is read and cleared; decided once per CTA
  const bool skipped = __syncthreads_or(
      tid == 0 && (*reinterpret_cast<volatile uint32_t *>(&g_prefill_errors) & kErrTimeout));
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kTmemSlotOff);
  auto wait_ = [&](uint32_t b, uint32_t parity) {
    return mbar_wait(b, parity, &g_prefill_errors, abort);
  };
  auto fail = [&]() {
    *abort = 1;
    atomicOr(&g_prefill_errors, kErrTimeout);
  };

  if (warp < kSoftmaxWarp0) {
    setmaxnreg_dec<RegSplit::kOther>();
    if (warp == kProducerWarp && !skipped) {
      // ------------------------------------------------------------ TMA producer
      // Per item: both Q tiles (once the previous item's S MMAs are done with
      // the Q buffer), then K and V tiles of 128 keys. Lane b < kBN / box_rows
      // owns the b-th box of every KV tile: it reads that box's block-table
      // entry one tile ahead (the read overlaps the wait for a free stage) and
      // issues the box's copies; lane 0 arms the barriers.
      const int box_rows = p.box_rows;
      const int n_boxes = kBN / box_rows;
      if (lane == 0) {
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
      }
      ItemWalk<kWindowed> w;
      int G0 = 0;  // KV steps of earlier items
      bool good = true;
      Item it;
      while (w.next(p, lane == 0, it)) {
        if (w.item_no >= 1 &&
            !__all_sync(0xffffffffu, wait_(bar(kBarQEmpty), (w.item_no - 1) & 1))) {
          good = false;
          break;
        }
        if (lane == 0) {
          volatile int *dv = reinterpret_cast<volatile int *>(smem + kItemOff);
          dv[0] = it.n_tiles[0] > 0 ? it.n_tiles[0] - it.j_start : 0;
          dv[1] = it.n_tiles[1] > 0 ? it.n_tiles[1] - it.j_start : 0;
          dv[2] = it.n_steps;
          dv[3] = it.Lk - (it.j_start + it.n_steps - 1) * kBN < kBN ? 1 : 0;
          uint32_t qbytes = 0;
#pragma unroll
          for (int t = 0; t < kTiles; ++t) qbytes += it.n_tiles[t] > 0 ? kTileBytes : 0;
          // the arrival releases the descriptor written above to the MMA issuer
          mbar_arrive_expect_tx(bar(kBarQ), qbytes);
#pragma unroll
          for (int t = 0; t < kTiles; ++t) {
            if (it.n_tiles[t] == 0) continue;
            tma_load_3d(sQ + t * kTileBytes, &q_map, bar(kBarQ), 0, it.head[t],
                        it.q0 + it.row0[t]);
            tma_load_3d(sQ + t * kTileBytes + kHalfBytes, &q_map, bar(kBarQ), 64, it.head[t],
                        it.q0 + it.row0[t]);
          }
        }
        // Release r (the MMA warp's commit after the S MMAs of global step r)
        // frees K(r) and V(r - 1). The item's first K goes on its own barrier
        // once release G0 - 2 has freed its stage; then step gk's copies,
        // V(gk) and (within the item) K(gk + 1), wait for release gk - 1,
        // which frees both their stages, and share one barrier.
        const int n_max = it.j_start + it.n_steps;
        const int32_t *table = p.block_tables + static_cast<int64_t>(it.s) * p.max_blocks;
        auto box_key = [&](int j) { return j * kBN + lane * box_rows; };
        auto has_box = [&](int j) { return lane < n_boxes && j < n_max && box_key(j) < it.Lk; };
        auto blk_of = [&](int j) {
          return has_box(j) ? __ldg(table + box_key(j) / p.block_size) : -1;
        };
        // cache row of this lane's box in KV tile j (-1: none; a block outside
        // the pool is reported and its box left out)
        auto row_of = [&](int j, int32_t blk) -> int32_t {
          if (!has_box(j)) return -1;
          if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(&g_prefill_errors, kErrBlock);
            return -1;
          }
          return blk * p.block_size + box_key(j) % p.block_size;
        };
        auto tile_bytes = [&](int32_t row) {
          return __popc(__ballot_sync(0xffffffffu, row >= 0)) * 2u * box_rows * 128u;
        };
        int32_t row_cur = row_of(it.j_start, blk_of(it.j_start));
        int32_t blk_nxt = blk_of(it.j_start + 1);
        if (G0 >= 2 &&
            !__all_sync(0xffffffffu, wait_(bar(kBarRel + (G0 & 1)), ((G0 - 2) >> 1) & 1))) {
          good = false;
          break;
        }
        {
          const uint32_t bytes = tile_bytes(row_cur);
          if (lane == 0) mbar_arrive_expect_tx(bar(kBarK0), bytes);
          __syncwarp();
          if (row_cur >= 0) {
            const uint32_t kdst = sK + (G0 & 1) * kTileBytes + lane * box_rows * 128;
            tma_load_3d(kdst, &k_map, bar(kBarK0), 0, it.g, row_cur);
            tma_load_3d(kdst + kHalfBytes, &k_map, bar(kBarK0), 64, it.g, row_cur);
          }
        }
        for (int jj = 0; jj < it.n_steps; ++jj) {
          const int j = it.j_start + jj, gk = G0 + jj;
          const int32_t row_nxt = row_of(j + 1, blk_nxt);  // -1 past the item's last tile
          blk_nxt = blk_of(j + 2);
          const uint32_t bytes = tile_bytes(row_cur) + tile_bytes(row_nxt);
          if (gk >= 1 &&
              !__all_sync(0xffffffffu,
                          wait_(bar(kBarRel + ((gk - 1) & 1)), ((gk - 1) >> 1) & 1))) {
            good = false;
            break;
          }
          const uint32_t b = bar(kBarKV + (gk & 1));
          if (lane == 0) mbar_arrive_expect_tx(b, bytes);
          __syncwarp();
          if (row_cur >= 0) {
            const uint32_t vdst = sV + (gk & 1) * kTileBytes + lane * box_rows * 128;
            tma_load_3d(vdst, &v_map, b, 0, it.g, row_cur);
            tma_load_3d(vdst + kHalfBytes, &v_map, b, 64, it.g, row_cur);
          }
          if (row_nxt >= 0) {
            const uint32_t kdst = sK + ((gk + 1) & 1) * kTileBytes + lane * box_rows * 128;
            tma_load_3d(kdst, &k_map, b, 0, it.g, row_nxt);
            tma_load_3d(kdst + kHalfBytes, &k_map, b, 64, it.g, row_nxt);
          }
          row_cur = row_nxt;
        }
        if (!good) break;
        // V rows of the item's last tile past the segment's last key (poison
        // in a partly used box, stale data in boxes not loaded) are zeroed once
        // the tile has landed, so that they never meet a zero probability
        const int tail_r0 = it.Lk - (n_max - 1) * kBN;
        if (tail_r0 < kBN) {
          const int gk = G0 + it.n_steps - 1, st = gk & 1;
          if (!__all_sync(0xffffffffu, wait_(bar(kBarKV + st), (gk >> 1) & 1))) {
            good = false;
            break;
          }
          const uint32_t vbase = sV + st * kTileBytes;
          const int n16 = (kBN - tail_r0) * 16;  // 16-byte pieces over both column halves
          for (int idx = lane; idx < n16; idx += 32) {
            const int r = tail_r0 + idx / 16, piece = idx % 16;
            const uint32_t addr = vbase + (piece / 8) * kHalfBytes + r * 128 + (piece % 8) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(0u), "r"(0u),
                         "r"(0u), "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarVTail + st));
        }
        G0 += it.n_steps;
      }
      // every copy of this CTA is issued: the next kernel may start launching
      if (lane == 0) griddep_launch_dependents();
      // an empty descriptor ends the MMA issuer's walk (once it is done with
      // the last item's descriptor: its S MMAs have completed)
      if (good && w.item_no >= 0 &&
          !__all_sync(0xffffffffu, wait_(bar(kBarQEmpty), w.item_no & 1)))
        good = false;
      if (good && lane == 0) {
        reinterpret_cast<volatile int *>(smem + kItemOff)[2] = 0;  // n_steps
        mbar_arrive(bar(kBarQ));
      }
      // wait for the last release of each slot (the MMA warp's final commit is
      // release G0), so that no arrival from the tensor core reaches this
      // CTA's shared memory after it has exited
      for (int r = max(G0 - 1, 0); good && G0 > 0 && r <= G0; ++r)
        good = __all_sync(0xffffffffu, wait_(bar(kBarRel + (r & 1)), (r >> 1) & 1));
      if (!good && lane == 0) fail();
    } else if (warp == kMmaWarp && !skipped) {
      // ------------------------------------------------------------ MMA issuer
      // As in prefill_kernel: the whole warp runs the loop and its waits
      // (warp-uniform control flow) and one elected lane, always lane 0,
      // issues every MMA and commit. K, V and Q arrive by TMA (the barrier's
      // completion orders them before the MMAs); P is written by other
      // threads' tcgen05.st, so its wait is followed by the tcgen05 fence
      // that pairs with theirs.
      // The operand descriptors are built once, as 32-bit low halves over one
      // common high half (all have a 1024-byte stride between 8-row groups
      // and 128-byte swizzle), and each MMA adds a constant to the
      // start-address field (address / 16 in the low 14 bits; no
      // shared-memory address carries out of it).
      auto wait_all = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_(b, parity));
      };
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(sQ, 16, 1024) >> 32);
      auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
      const uint32_t q_lo0 = lo(smem_desc_sw128(sQ, 16, 1024));
      const uint32_t q_lo1 = lo(smem_desc_sw128(sQ + kTileBytes, 16, 1024));
      const uint32_t k_lo0 = lo(smem_desc_sw128(sK, 16, 1024));
      const uint32_t k_lo1 = lo(smem_desc_sw128(sK + kTileBytes, 16, 1024));
      const uint32_t v_lo0 = lo(smem_desc_sw128(sV, kHalfBytes, 1024));
      const uint32_t v_lo1 = lo(smem_desc_sw128(sV + kTileBytes, kHalfBytes, 1024));
      uint32_t tail_parity = 0;  // bit st: parity of the next tail of V stage st
      // The MMAs of one item: tiles 0 and 1 take n_t0 and n_t1 of its n_steps
      // KV steps; G0, T00 and T01 count the CTA's steps (of the KV stream and
      // of each tile) before it. Without persistence they are all 0.
      auto run_item = [&](int n_t0, int n_t1, int n_steps, bool has_tail, int G0, int T00,
                          int T01, int item_no) -> bool {
        int s_left = n_t0 + n_t1;  // S MMA groups of this item still to issue
        auto issue_s = [&](int t, int jj) {
          const int gk = G0 + jj, st = gk & 1;
          const uint32_t tS = tmem + t * kBN;
          const uint32_t qd = t ? q_lo1 : q_lo0;
          const uint32_t kd = st ? k_lo1 : k_lo0;
          --s_left;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off16 = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
              mma_bf16_ss(tS, qd + off16, kd + off16, desc_hi, kIdescQK, kk > 0);
            }
            mma_commit(bar(kBarS + t));
            // the item's last S: the Q buffer is free for the next item once it completes
            if (s_left == 0) mma_commit(bar(kBarQEmpty));
          }
          __syncwarp();
        };
        auto issue_pv = [&](int t, int jj) -> bool {
          const int gk = G0 + jj, st = gk & 1;
          // P_t of this step is in TMEM once the softmax of tile t has arrived
          if (!wait_all(bar(kBarP + t), ((t ? T01 : T00) + jj) & 1)) return false;
          tc_fence_after();
          const uint32_t tP = tmem + t * kBN;             // P over the first 64 columns of S_t
          const uint32_t tO = tmem + 2 * kBN + t * kD;
          const uint32_t vd = st ? v_lo1 : v_lo0;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_bf16_ts(tO, tP + kk * 8, vd + ((kk * 16 * 128) >> 4), desc_hi, kIdescPV,
                          (jj > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(kBarO + t));
          }
          __syncwarp();
          return true;
        };
        // the item's first K (its own barrier, one phase per item), its first
        // S MMAs, then release G0 (K(G0), and V(G0 - 1) of the item before)
        bool ok = wait_all(bar(kBarK0), item_no & 1);
        if (ok && n_t0 > 0) issue_s(0, 0);
        if (ok && n_t1 > 0) issue_s(1, 0);
        if (ok) {
          if (elect_one()) mma_commit(bar(kBarRel + (G0 & 1)));
          __syncwarp();
        }
        for (int jj = 1; ok && jj <= n_steps; ++jj) {
          // V(jj - 1) and K(jj) are resident: one barrier (the producer zeroes
          // the tail of the item's last KV tile, which comes with no K)
          const int gb = G0 + jj - 1, sb = gb & 1;
          if (has_tail && jj == n_steps) {
            const uint32_t par = (tail_parity >> sb) & 1u;
            tail_parity ^= 1u << sb;
            ok = wait_all(bar(kBarVTail + sb), par);
          } else {
            ok = wait_all(bar(kBarKV + sb), (gb >> 1) & 1);
          }
          // finish step jj-1 for every query tile, starting step jj where needed
          if (ok && jj - 1 < n_t0) {
            ok = issue_pv(0, jj - 1);
            if (ok && jj < n_t0) issue_s(0, jj);
          }
          if (ok && jj - 1 < n_t1) {
            ok = issue_pv(1, jj - 1);
            if (ok && jj < n_t1) issue_s(1, jj);
          }
          // release G0 + jj: K(G0 + jj) has had its last S, V(G0 + jj - 1)
          // its last P.V (the item's last V is released by the next item's
          // first release, or by the final one)
          if (ok && jj < n_steps) {
            if (elect_one()) mma_commit(bar(kBarRel + ((G0 + jj) & 1)));
            __syncwarp();
          }
        }
        return ok;
      };
      bool good = true;
      // item by item, as the producer publishes them with their Q
      int G0 = 0, T00 = 0, T01 = 0;
      for (int item_no = 0; good; ++item_no) {
        if (!wait_all(bar(kBarQ), item_no & 1)) {
          good = false;
          break;
        }
        const volatile int *dv = reinterpret_cast<volatile int *>(smem + kItemOff);
        const int n_t0 = dv[0], n_t1 = dv[1], n_steps = dv[2], tail = dv[3];
        if (n_steps == 0) break;  // no more items
        good = run_item(n_t0, n_t1, n_steps, tail != 0, G0, T00, T01, item_no);
        G0 += n_steps;
        T00 += n_t0;
        T01 += n_t1;
      }
      // the final release G0 frees the last V; every MMA issued here has
      // completed before the CTA frees its TMEM
      if (good && G0 > 0) {
        if (elect_one()) mma_commit(bar(kBarRel + (G0 & 1)));
        __syncwarp();
      }
      if (elect_one()) mma_commit(bar(kBarDone));
      __syncwarp();
      if (!wait_all(bar(kBarDone), 0)) good = false;
      if (!good && lane == 0) fail();
    }
  } else {
    setmaxnreg_inc<RegSplit::kSoftmax>();
    if (!skipped) {
      // ------------------------------------------------------------ softmax / epilogue
      const int t = (warp - kSoftmaxWarp0) >> 2;  // query tile of this warpgroup
      const int quad = warp & 3;              // TMEM lane quadrant this warp may access
      const int r = quad * 32 + lane;         // row within the tile == TMEM lane
      const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t tS = tmem + t * kBN + lane_off;
      const uint32_t tO = tmem + 2 * kBN + t * kD + lane_off;
      const uint64_t scl = f32x2(p.scale_log2, p.scale_log2);
      // One item's softmax and epilogue for this tile; T0 counts the tile's
      // steps before it (0 without persistence). False if a wait gave up.
      // The walk to the next item (a few global loads and divisions) runs in
      // the middle of this one: after the tile's last P, while its last P.V
      // completes, instead of between the epilogue and the next item's start.
      ItemWalk<kWindowed> w;
      Item nxt;
      bool have_nxt = false;
      auto run_item = [&](const Item &it, int T0) -> bool {
        bool good = true;
        // this tile's part of the item, in scalars (selects, not indexed arrays)
        const int j_start = it.j_start, Lk = it.Lk, Lq = it.Lq, diag = it.diag, q0 = it.q0;
        const int tiles_t = t ? it.n_tiles[1] : it.n_tiles[0];
        const int n_t = tiles_t > 0 ? tiles_t - j_start : 0;  // steps of this tile
        const int row0 = t ? it.row0[1] : it.row0[0];
        const int head_t = t ? it.head[1] : it.head[0];
        const int qi = row0 + r;                // query index within the segment
        const int lim = diag + qi;              // last key this row may see
        const int first = kWindowed ? lim - p.window + 1 : 0;  // first key (may be < 0)
        // the largest first key of the tile's rows: KV tiles below it need masking
        const int first_hi = kWindowed ? diag + row0 + kBM - p.window : 0;
        // Running maximum m (log2 units) and two running sums: l of the fp32
        // probabilities, for the lse, and lr of the same probabilities rounded to
        // bf16 as the P.V product sees them, which normalises the output. The
        // maximum is lazy: a row keeps its m while a tile's probabilities sum to
        // at most 2^kLazyMax, so no probability exceeds that bound and O is
        // rescaled only when some row of the warp passes it. Dividing by
        // the sum of the rounded probabilities keeps the output a convex
        // combination of the V rows with the weights the tensor core used, so a
        // large probability rounded to bf16 costs no more than it does under an
        // exact maximum. A row whose first tiles lie wholly before its window
        // starts from a finite floor, so that its masked logits give probability
        // 0 and its first visible tile rescales an O of zeros.
        constexpr float kFloor = -1e30f;
        float m = kFloor, l = 0.f, lr = 0.f;
        for (int jj = 0; jj < n_t; ++jj) {
          if (!__all_sync(0xffffffffu, wait_(bar(kBarS + t), (T0 + jj) & 1))) {
            good = false;
            break;
          }
          tc_fence_after();
          const int kbase = (j_start + jj) * kBN;
          uint32_t x[kBN];
#pragma unroll
          for (int c = 0; c < kBN; c += 32)
            tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&x[c]));
          tmem_wait_ld();
          // keys past the row's causal limit or the segment end, or before its
          // window, are masked (their logit becomes -inf, their probability 0);
          // only the diagonal, the tail and the window's first tiles have any
          if ((kbase + kBN - 1 > diag + row0) || (kbase + kBN > Lk) ||
              (kWindowed && kbase < first_hi)) {
            const int keep = min(lim, Lk - 1) - kbase + 1;  // columns < keep: at or before the limit
            if constexpr (kWindowed) {
              const int skip = first - kbase;                  // columns < skip: before the window
#pragma unroll
              for (int c = 0; c < kBN; ++c)
                if (c >= keep || c < skip) x[c] = 0xFF800000u;
            } else {
#pragma unroll
              for (int c = 0; c < kBN; ++c)
                if (c >= keep) x[c] = 0xFF800000u;
            }
          }
          // P = 2^(x * scale - mm), packed two per column over the first 64
          // columns of S_t (all of S is already in registers); ts and tr get the
          // tile's sums of the fp32 and of the bf16-rounded probabilities
          auto exps = [&](float mm, float &ts, float &tr) {
            const uint64_t nm = f32x2(-mm, -mm);
            uint64_t s0 = 0, s1 = 0;
            float r0l = 0.f, r0h = 0.f, r1l = 0.f, r1h = 0.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t pk[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int k = hf * 64 + 2 * c;
                const uint64_t e =
                    fma2(f32x2(__uint_as_float(x[k]), __uint_as_float(x[k + 1])), scl, nm);
                const float p0 = fast_exp2(f32x2_lo(e)), p1 = fast_exp2(f32x2_hi(e));
                pk[c] = pack_bf16x2(p0, p1);
                if (c & 1) {
                  add2(s1, f32x2(p0, p1));
                  add_bf16x2_to_f32(r1l, r1h, pk[c]);
                } else {
                  add2(s0, f32x2(p0, p1));
                  add_bf16x2_to_f32(r0l, r0h, pk[c]);
                }
              }
              tmem_st32(tS + hf * 32, pk);
            }
            add2(s0, s1);
            ts = f32x2_lo(s0) + f32x2_hi(s0);
            tr = (r0l + r1l) + (r0h + r1h);
          };
          // First with the row's current maximum, without looking for a larger
          // one: if no row of the warp then has a tile sum above 2^kLazyMax, no
          // probability exceeds that bound either and the tile is done. Otherwise
          // (some logit lies more than a little above m; an infinite sum included)
          // the warp takes the exact maximum, rescales O and recomputes P over
          // what it wrote. The first tile of a row always takes the maximum.
          float ts, tr;
          bool exact = jj == 0;
#pragma unroll 1
          for (;;) {
            if (exact) {
              // row max of the raw logits (the scale is positive): eight chains
              // of three-input maxima
              float a[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(x[i]);
#pragma unroll
              for (int c = 8; c < kBN; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  a[i] = fmax3(a[i], __uint_as_float(x[c + i]), __uint_as_float(x[c + 8 + i]));
              const float mx =
                  fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
              const float mxs = mx * p.scale_log2;  // -inf stays -inf
              if (jj == 0) {
                // nothing is in O yet; without a window every row sees key 0
                m = kWindowed ? fmaxf(mxs, kFloor) : mxs;
              } else {
                // P.V of the previous step is complete (this S was issued after
                // it): rescale the O rows in TMEM. The accesses are warp-wide, so
                // the whole warp takes its new maxima.
                const float m_new = fmaxf(m, mxs);
                const float alpha = fast_exp2(m - m_new);
                // 32 columns at a time: all of S is held in registers meanwhile
#pragma unroll 1
                for (int c = 0; c < kD; c += 32) {
                  uint32_t o[32];
                  tmem_ld32(tO + c, o);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st32(tO + c, o);
                }
                tmem_wait_st();
                l *= alpha;
                lr *= alpha;
                m = m_new;
              }
            }
            exps(m, ts, tr);
            if (exact || !__any_sync(0xffffffffu, !(ts <= kLazyBound))) break;
            exact = true;
          }
          l += ts;
          lr += tr;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kBarP + t));
        }
        if (!good) return false;
        have_nxt = w.next(p, false, nxt);
        if (n_t > 0) {
          // epilogue: the last P.V of the item has completed once its O barrier
          // phase has; the next item's first P.V (which overwrites O) waits for
          // this warp's next P, written only after these reads
          if (!__all_sync(0xffffffffu, wait_(bar(kBarO + t), (T0 + n_t - 1) & 1))) return false;
          tc_fence_after();
          const float inv_l = 1.f / lr;
          const bool store = qi < Lq;
          const int qw = row0 + quad * 32;  // query of the warp's first row
          store_o_rows(tO, inv_l, sbase + kEpiOff + (warp - kSoftmaxWarp0) * kEpiWarpBytes,
                       p.out + (static_cast<int64_t>(q0 + qw) * p.num_q_heads + head_t) * kD,
                       static_cast<int64_t>(p.num_q_heads) * kD, min(32, Lq - qw), lane);
          if (store && p.lse != nullptr)
            p.lse[static_cast<int64_t>(q0 + qi) * p.num_q_heads + head_t] =
                (m + log2f(l)) * kLn2;
        }
        return true;
      };
      bool good = true;
      int T0 = 0;  // steps of this tile in earlier items
      Item it;
      bool have = w.next(p, false, it);
      while (good && have) {
        good = run_item(it, T0);
        const int tiles_t = t ? it.n_tiles[1] : it.n_tiles[0];
        T0 += tiles_t > 0 ? tiles_t - it.j_start : 0;
        it = nxt;
        have = have_nxt;
      }
      if (!good && r == 0) fail();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// The kernel to launch: prefill_persistent_kernel or prefill_kernel.
template <bool kWindowed, bool kPersistent>
constexpr auto prefill_entry() {
  if constexpr (kPersistent)
    return prefill_persistent_kernel<kWindowed>;
  else
    return prefill_kernel;
}

template <bool kWindowed, bool kPersistent>
cudaError_t launch_instance(dim3 grid, const CUtensorMap &q_map, const CUtensorMap &k_map,
                            const CUtensorMap &v_map, const PrefillParams &p,
                            cudaStream_t stream) {
  auto kern = prefill_entry<kWindowed, kPersistent>();
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until registers released by the other warpgroup are
  // free: launch only a build whose per-thread allocation covers the split
  static const int launch_regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, prefill_entry<kWindowed, kPersistent>()) == cudaSuccess
               ? fa.numRegs
               : 0;
  }();
  using R = RegSplit;
  if (launch_regs * kThreads < (2 * R::kSoftmax + R::kOther) * 128)
    return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, stream, q_map, k_map, v_map, p);
}

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t stream) {
  if (a.total_q == 0 || a.max_seqlen_q == 0 || a.num_seqs == 0) return cudaSuccess;
  const int G = a.num_q_heads / a.num_kv_heads;
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
  const int rows_per_item = G >= 2 ? kBM : 2 * kBM;
  p.n_rowtiles = (a.max_seqlen_q + rows_per_item - 1) / rows_per_item;
  p.n_pairs = G >= 2 ? a.num_q_heads / 2 : a.num_q_heads;
  const int64_t n_items = static_cast<int64_t>(p.n_rowtiles) * p.n_pairs * a.num_seqs;
  if (n_items > kMaxPrefillItems) return cudaErrorInvalidValue;
  p.n_items = static_cast<int32_t>(n_items);
  p.window = a.window;
  p.box_rows = a.box_rows;
  p.scale_log2 = a.scale_log2;
  if (p.window > 0) {
    // persistent: one CTA per SM (the shared memory admits no second one)
    const dim3 grid(static_cast<unsigned>(n_items < a.num_sms ? n_items : a.num_sms));
    return launch_instance<true, true>(grid, q_map, k_map, v_map, p, stream);
  }
  const dim3 grid = p.n_pairs <= 65535 && p.num_seqs <= 65535
                       ? dim3(p.n_rowtiles, p.n_pairs, p.num_seqs)
                       : dim3(static_cast<unsigned>(n_items));
  return launch_instance<false, false>(grid, q_map, k_map, v_map, p, stream);
}

cudaError_t prefill_error_word(uint32_t **word) {
  return cudaGetSymbolAddress(reinterpret_cast<void **>(word), g_prefill_errors);
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
