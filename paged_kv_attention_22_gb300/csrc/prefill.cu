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
//   warp 8     TMA producer: both Q tiles once, then K and V tiles of 128 keys,
//              two stages deep, 128-byte swizzled. A tile is copied as boxes of
//              the largest of 128, 64, 32, 16 rows that divides the block size
//              (a box never crosses a cache block): fewer, larger copies
//              (one 128-row box per column half streams from L2 about twice
//              as fast per SM as eight 16-row boxes).
//   warp 9     MMA issuer. TMEM holds S_t (128 fp32 columns) and O_t (128) for
//              each tile t. Per KV tile j and query tile t: S_t = Q_t K_j^T
//              (A and B from shared memory), then, once the softmax has
//              written P_t (bf16) over the first 64 columns of S_t,
//              O_t += P_t V_j with A read straight from TMEM. S_t(j+1) is
//              issued after P.V(j), and MMAs run in issue order, so a
//              completed S_t(j+1) also means O_t holds every tile up to j.
//              The V rows past the segment's last key are zeroed before their
//              first P.V, so stale or poisoned rows never meet a zero
//              probability.
//   warps 0-3  softmax of tile 0, warps 4-7 softmax of tile 1: one query row
//              per thread (TMEM lane = row). Read the S row, mask, online
//              softmax in base 2 (the O row in TMEM is rescaled only in tiles
//              where some row's maximum grows), write P back into TMEM; at the
//              end normalise O and store the bf16 output and the natural-log
//              lse.
// While one tile's softmax runs, the tensor pipe works on the other tile.
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
// kBarVTail: the last V tile, its rows past the segment's end zeroed
constexpr int kBarQ = 0, kBarKFull = 1, kBarVFull = 3, kBarKEmpty = 5, kBarVEmpty = 7, kBarS = 9,
              kBarP = 11, kBarO = 13, kBarVTail = 15, kNumBars = 16;
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kAbortOff = kTmemSlotOff + 8;
constexpr int kSmemBytes = kAbortOff + 8 + 1024;  // + slack for 1024-byte alignment
// warps 0-7 softmax (warpgroup t for query tile t), warp 8 TMA producer,
// warp 9 MMA issuer, warps 10-11 idle: three warpgroups, so that setmaxnreg
// can move registers from the third to the two softmax warpgroups
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
// registers per thread after the split; 2 * 216 + 72 = 3 * 168, the launch's
// share per thread of the 64K register file for 384 threads
constexpr int kSoftmaxRegs = 216, kOtherRegs = 72;
constexpr uint32_t kTmemCols = 512;            // S0, S1, O0, O1: 128 columns each
constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);  // A=Q K-major, B=K K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, 0, 1);   // A=P (TMEM), B=V MN-major
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLazyMax = 8.0f;  // log2 units the running maximum may lag
constexpr float kLazyBound = 256.0f;  // 2^kLazyMax: the largest tile sum taken as is

struct PrefillParams {
  const int32_t *cu_q, *cu_k, *block_tables;
  __nv_bfloat16 *out;
  float *lse;
  int32_t max_blocks, num_seqs, total_q, max_seqlen_q, max_seqlen_k;
  int32_t num_q_heads, num_kv_heads, block_size, num_blocks, n_rowtiles;
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

// kWindowed: a sliding window is set (p.window > 0). The kernel without one
// is a separate instantiation, so that it keeps no window bookkeeping at all.
template <bool kWindowed>
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
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int per_rt = gridDim.y * gridDim.z;  // CTAs per row tile index
  const int rt = p.n_rowtiles - 1 - lin / per_rt;
  const int pair = (lin % per_rt) % gridDim.y;
  const int s = (lin % per_rt) / gridDim.y;
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
  // With a sliding window query i sees keys >= diag + i - window + 1: the KV
  // tiles before the one that holds the earliest such key of this CTA's rows
  // are skipped. Steps jj = 0 .. n_steps - 1 cover KV tiles j_start + jj;
  // stages and barrier phases count steps.
  int j_start = 0;
  if constexpr (kWindowed) {
    int lo = Lk;
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if (n_tiles[t] > 0) lo = min(lo, max(0, diag + row0[t] - p.window + 1));
    j_start = lo / kBN;
  }
  const int n_steps = n_max - j_start;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kQOff, sK = sbase + kKOff, sV = sbase + kVOff;
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile int *abort = reinterpret_cast<volatile int *>(smem + kAbortOff);

  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarVTail), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarKEmpty + i), 1);
      mbar_init(bar(kBarVEmpty + i), 1);
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

  if (warp >= kProducerWarp) {
    setmaxnreg_dec<kOtherRegs>();
    if (warp == kProducerWarp) {
      // ------------------------------------------------------------ TMA producer
      // Lane b < kBN / box_rows owns the b-th box of every KV tile: it reads
      // that box's block-table entry one tile ahead (the read overlaps the
      // wait for a free stage) and issues the box's copies; lane 0 arms the
      // barriers. K and V stages are released separately: K(j) once every
      // S = Q K(j)^T is done, V(j) once every P.V(j) is.
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
      int32_t next_blk = has_box(j_start) ? __ldg(table + box_key(j_start) / p.block_size) : -1;
      bool good = true;
      for (int jj = 0; jj < n_steps; ++jj) {
        const int j = j_start + jj;
        const int st = jj & 1;
        const int32_t blk = next_blk;
        if (has_box(j + 1)) next_blk = __ldg(table + box_key(j + 1) / p.block_size);
        int32_t row = -1;
        if (has_box(j)) {
          if (blk < 0 || blk >= p.num_blocks)
            atomicOr(&g_prefill_errors, kErrBlock);
          else
            row = blk * p.block_size + box_key(j) % p.block_size;
        }
        const uint32_t bytes =
            __popc(__ballot_sync(0xffffffffu, row >= 0)) * 2u * box_rows * 128u;
        if (jj >= kStages &&
            !__all_sync(0xffffffffu, wait_(bar(kBarKEmpty + st), ((jj >> 1) - 1) & 1, abort))) {
          good = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarKFull + st), bytes);
        __syncwarp();
        const uint32_t kdst = sK + st * kTileBytes + lane * box_rows * 128;
        if (row >= 0) {
          tma_load_3d(kdst, &k_map, bar(kBarKFull + st), 0, g, row);
          tma_load_3d(kdst + kHalfBytes, &k_map, bar(kBarKFull + st), 64, g, row);
        }
        if (jj >= kStages &&
            !__all_sync(0xffffffffu, wait_(bar(kBarVEmpty + st), ((jj >> 1) - 1) & 1, abort))) {
          good = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarVFull + st), bytes);
        __syncwarp();
        const uint32_t vdst = sV + st * kTileBytes + lane * box_rows * 128;
        if (row >= 0) {
          tma_load_3d(vdst, &v_map, bar(kBarVFull + st), 0, g, row);
          tma_load_3d(vdst + kHalfBytes, &v_map, bar(kBarVFull + st), 64, g, row);
        }
      }
      // every copy of this CTA is issued: the next kernel may start launching
      if (lane == 0) griddep_launch_dependents();
      // V rows of the last tile past the segment's last key (poison in a
      // partly used box, stale data in boxes not loaded) are zeroed once the
      // tile has landed, so that they never meet a zero probability
      const int tail_r0 = Lk - (n_max - 1) * kBN;
      if (good && tail_r0 < kBN) {
        const int st = (n_steps - 1) & 1;
        good = __all_sync(0xffffffffu, wait_(bar(kBarVFull + st), ((n_steps - 1) >> 1) & 1, abort));
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
      // wait for the last release of each stage, so that no arrival from the
      // tensor core reaches this CTA's shared memory after it has exited
      for (int jj = max(n_steps - kStages, 0); good && jj < n_steps; ++jj) {
        const uint32_t par = (jj >> 1) & 1;
        good = __all_sync(0xffffffffu, wait_(bar(kBarKEmpty + (jj & 1)), par, abort) &&
                                           wait_(bar(kBarVEmpty + (jj & 1)), par, abort));
      }
      if (!good && lane == 0) fail(abort);
    } else if (warp == kMmaWarp && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // One thread issues every MMA and commit. K, V and Q arrive by TMA (the
      // barrier's completion orders them before the MMAs); P is written by
      // other threads' tcgen05.st, so its wait is followed by the tcgen05
      // fence that pairs with theirs.
      // Steps are counted from the CTA's first KV tile (j_start); query tile t
      // has steps 0 .. n_tiles[t] - j_start - 1 (none if that is not positive).
      bool good = wait_(bar(kBarQ), 0, abort);
      int v_ready = -1;  // last step whose V is resident (and tail-zeroed)
      // This thread shares its SM sub-partition with two softmax warps, which
      // take most issue slots while they run: every instruction here delays
      // the next MMA. So the operand descriptors are built once, as 32-bit
      // low halves over one common high half (all have a 1024-byte stride
      // between 8-row groups and 128-byte swizzle), and each MMA adds a
      // constant to the start-address field (address / 16 in the low 14 bits;
      // no shared-memory address carries out of it).
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(sQ, 16, 1024) >> 32);
      auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
      const uint32_t q_lo0 = lo(smem_desc_sw128(sQ, 16, 1024));
      const uint32_t q_lo1 = lo(smem_desc_sw128(sQ + kTileBytes, 16, 1024));
      const uint32_t k_lo0 = lo(smem_desc_sw128(sK, 16, 1024));
      const uint32_t k_lo1 = lo(smem_desc_sw128(sK + kTileBytes, 16, 1024));
      const uint32_t v_lo0 = lo(smem_desc_sw128(sV, kHalfBytes, 1024));
      const uint32_t v_lo1 = lo(smem_desc_sw128(sV + kTileBytes, kHalfBytes, 1024));
      auto issue_s = [&](int t, int jj) -> bool {
        const int st = jj & 1;
        if (!wait_(bar(kBarKFull + st), (jj >> 1) & 1, abort)) return false;
        const uint32_t tS = tmem + t * kBN;
        const uint32_t qd = t ? q_lo1 : q_lo0;
        const uint32_t kd = st ? k_lo1 : k_lo0;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off16 = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tS, qd + off16, kd + off16, desc_hi, kIdescQK, kk > 0);
        }
        mma_commit(bar(kBarS + t));
        return true;
      };
      auto issue_pv = [&](int t, int jj) -> bool {
        const int st = jj & 1;
        if (v_ready != jj) {
          // the producer zeroes the tail of the segment's last KV tile
          const bool tail = Lk - (j_start + jj) * kBN < kBN;
          if (!(tail ? wait_(bar(kBarVTail), 0, abort)
                     : wait_(bar(kBarVFull + st), (jj >> 1) & 1, abort)))
            return false;
          v_ready = jj;
        }
        // P_t of this step is in TMEM once the softmax of tile t has arrived
        if (!wait_(bar(kBarP + t), jj & 1, abort)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + t * kBN;             // P over the first 64 columns of S_t
        const uint32_t tO = tmem + 2 * kBN + t * kD;
        const uint32_t vd = st ? v_lo1 : v_lo0;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tO, tP + kk * 8, vd + ((kk * 16 * 128) >> 4), desc_hi, kIdescPV,
                      (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kBarO + t));
        return true;
      };
      for (int t = 0; good && t < kTiles; ++t)
        if (n_tiles[t] - j_start > 0) good = issue_s(t, 0);
      if (good) mma_commit(bar(kBarKEmpty));  // K of step 0 is free once those are done
      for (int jj = 1; good && jj <= n_steps; ++jj) {
        // finish step jj-1 for every query tile, starting step jj where needed
        for (int t = 0; good && t < kTiles; ++t) {
          if (jj - 1 >= n_tiles[t] - j_start) continue;
          good = issue_pv(t, jj - 1);
          if (good && jj < n_tiles[t] - j_start) good = issue_s(t, jj);
        }
        // V of step jj-1 has had its last P.V; K of step jj its last S
        if (good) {
          mma_commit(bar(kBarVEmpty + ((jj - 1) & 1)));
          if (jj < n_steps) mma_commit(bar(kBarKEmpty + (jj & 1)));
        }
      }
      if (!good) fail(abort);
    }
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;                // query tile of this warpgroup
    const int quad = warp & 3;              // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;         // row within the tile == TMEM lane
    const int n_t = n_tiles[t] > 0 ? n_tiles[t] - j_start : 0;  // steps of this tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + t * kBN + lane_off;
    const uint32_t tO = tmem + 2 * kBN + t * kD + lane_off;
    const int qi = row0[t] + r;             // query index within the segment
    const int lim = diag + qi;              // last key this row may see
    const int first = kWindowed ? lim - p.window + 1 : 0;  // first key (may be < 0)
    // the largest first key of the tile's rows: KV tiles below it need masking
    const int first_hi = kWindowed ? diag + row0[t] + kBM - p.window : 0;
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
      // keys past the row's causal limit or the segment end, or before its
      // window, are masked (their logit becomes -inf, their probability 0);
      // only the diagonal, the tail and the window's first tiles have any
      if ((kbase + kBN - 1 > diag + row0[t]) || (kbase + kBN > Lk) ||
          (kWindowed && kbase < first_hi)) {
        const int keep = min(lim, Lk - 1) - kbase + 1;  // columns < keep are at or before the limit
        if constexpr (kWindowed) {
          const int skip = first - kbase;               // columns < skip are before the window
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
    if (n_t > 0 &&
        __all_sync(0xffffffffu, good && wait_(bar(kBarO + t), (n_t - 1) & 1, abort))) {
      tc_fence_after();
      const float inv_l = 1.f / lr;
      const bool store = qi < Lq;
      __nv_bfloat16 *orow =
          p.out + (static_cast<int64_t>(q0 + qi) * p.num_q_heads + head[t]) * kD;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
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

}  // namespace

template <bool kWindowed>
cudaError_t launch_instance(dim3 grid, const CUtensorMap &q_map, const CUtensorMap &k_map,
                            const CUtensorMap &v_map, const PrefillParams &p,
                            cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kWindowed>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until registers released by the other warpgroup are
  // free: launch only a build whose per-thread allocation covers the split
  static const int launch_regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, prefill_kernel<kWindowed>) == cudaSuccess ? fa.numRegs : 0;
  }();
  if (launch_regs * kThreads < (2 * kSoftmaxRegs + kOtherRegs) * 128)
    return cudaErrorInvalidConfiguration;
  return launch_pdl(prefill_kernel<kWindowed>, grid, dim3(kThreads), kSmemBytes, stream, q_map,
                    k_map, v_map, p);
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
  const int rows_per_cta = G >= 2 ? kBM : 2 * kBM;
  p.n_rowtiles = (a.max_seqlen_q + rows_per_cta - 1) / rows_per_cta;
  p.window = a.window;
  p.box_rows = a.box_rows;
  p.scale_log2 = a.scale_log2;
  dim3 grid(p.n_rowtiles, G >= 2 ? a.num_q_heads / 2 : a.num_q_heads, a.num_seqs);
  return p.window > 0 ? launch_instance<true>(grid, q_map, k_map, v_map, p, stream)
                      : launch_instance<false>(grid, q_map, k_map, v_map, p, stream);
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
