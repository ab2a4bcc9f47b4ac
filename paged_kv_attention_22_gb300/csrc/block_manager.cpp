// Host-side KV block manager (pkv_blocks.h): reference-counted fixed-size
// blocks, a free list, and prefix sharing of full blocks found by a chained
// hash of their token ids ("How lunaryes/nano-vllm works", Components: KV Block
// Manager; nano-vllm-sansho README, "Key Features": prefix caching).
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_blocks.h"

namespace {

// 64-bit FNV-1a (Fowler-Noll-Vo) over the previous block's hash and the block's
// token ids, little-endian bytes.
constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t chain_hash(uint64_t prev, const int32_t *tokens, int32_t n) {
  uint64_t h = kFnvOffset;
  auto mix32 = [&h](uint32_t w) {
    for (int b = 0; b < 4; ++b) {
      h ^= (w >> (8 * b)) & 0xFFu;
      h *= kFnvPrime;
    }
  };
  mix32(static_cast<uint32_t>(prev));
  mix32(static_cast<uint32_t>(prev >> 32));
  for (int32_t i = 0; i < n; ++i) mix32(static_cast<uint32_t>(tokens[i]));
  return h;
}

struct Block {
  int32_t ref = 0;
  bool in_free = false;
  int32_t prev_free = -1, next_free = -1;  // free-list links while in_free
  bool findable = false;                   // registered under `hash`
  uint64_t hash = 0, parent = 0;           // own chain hash and the previous block's
};

struct Sequence {
  std::vector<int32_t> blocks;
  std::vector<int32_t> tokens;
  std::vector<uint64_t> chain;  // chain hash of each full block
};

}  // namespace

struct pkv_block_manager {
  int32_t num_blocks = 0, block_size = 0;
  std::vector<Block> blocks;
  std::vector<int32_t> content;  // token ids of each findable block [num_blocks][block_size]
  int32_t free_head = -1, free_tail = -1, num_free = 0;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Sequence> seqs;

  void push_free(int32_t b) {
    Block &x = blocks[b];
    x.in_free = true;
    x.prev_free = free_tail;
    x.next_free = -1;
    if (free_tail >= 0) blocks[free_tail].next_free = b; else free_head = b;
    free_tail = b;
    ++num_free;
  }

  void unlink_free(int32_t b) {
    Block &x = blocks[b];
    if (x.prev_free >= 0) blocks[x.prev_free].next_free = x.next_free; else free_head = x.next_free;
    if (x.next_free >= 0) blocks[x.next_free].prev_free = x.prev_free; else free_tail = x.prev_free;
    x.in_free = false;
    x.prev_free = x.next_free = -1;
    --num_free;
  }

  // The oldest free block, no longer findable under its old content.
  int32_t take_fresh() {
    const int32_t b = free_head;
    unlink_free(b);
    Block &x = blocks[b];
    if (x.findable) {
      auto it = by_hash.find(x.hash);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
      x.findable = false;
    }
    x.ref = 1;
    return b;
  }

  // The findable block holding these tokens after `parent`, or -1.
  int32_t lookup(uint64_t hash, uint64_t parent, const int32_t *tokens) const {
    auto it = by_hash.find(hash);
    if (it == by_hash.end()) return -1;
    const int32_t b = it->second;
    const Block &x = blocks[b];
    if (x.parent != parent) return -1;
    const int32_t *have = content.data() + static_cast<size_t>(b) * block_size;
    return std::memcmp(have, tokens, sizeof(int32_t) * block_size) == 0 ? b : -1;
  }

  // Make full block b findable under hash (unless another block already is).
  void publish(int32_t b, uint64_t hash, uint64_t parent, const int32_t *tokens) {
    if (by_hash.count(hash)) return;
    by_hash.emplace(hash, b);
    Block &x = blocks[b];
    x.findable = true;
    x.hash = hash;
    x.parent = parent;
    std::memcpy(content.data() + static_cast<size_t>(b) * block_size, tokens,
                sizeof(int32_t) * block_size);
  }
};

extern "C" {

pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size) {
  // slots are int32: block * block_size + offset must fit
  if (num_blocks <= 0 || block_size <= 0 ||
      static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return nullptr;
  pkv_block_manager *bm = new (std::nothrow) pkv_block_manager;
  if (bm == nullptr) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->blocks.resize(num_blocks);
    bm->content.resize(static_cast<size_t>(num_blocks) * block_size);
    for (int32_t b = 0; b < num_blocks; ++b) bm->push_free(b);
  } catch (const std::bad_alloc &) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int32_t pkv_bm_num_free_blocks(const pkv_block_manager *bm) {
  return bm == nullptr ? 0 : bm->num_free;
}

int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t b) {
  if (bm == nullptr || b < 0 || b >= bm->num_blocks) return -1;
  return bm->blocks[b].ref;
}

pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, const int32_t *token_ids,
                               int32_t num_tokens, int32_t *num_cached_tokens) {
  if (bm == nullptr || token_ids == nullptr || num_tokens <= 0 || num_cached_tokens == nullptr ||
      bm->seqs.count(seq_id))
    return PKV_ERR_INVALID_ARG;
  const int32_t bs = bm->block_size;
  const int32_t n_blocks = (num_tokens + bs - 1) / bs;
  const int32_t n_full = num_tokens / bs;
  const int32_t max_shared = (num_tokens - 1) / bs;  // keep at least one token to compute

  // which leading full blocks are already in the cache (no change yet)
  std::vector<int32_t> shared;
  std::vector<uint64_t> chain;
  uint64_t parent = 0;
  int32_t shared_free = 0;
  for (int32_t i = 0; i < max_shared; ++i) {
    const int32_t *tok = token_ids + static_cast<size_t>(i) * bs;
    const uint64_t h = chain_hash(parent, tok, bs);
    const int32_t b = bm->lookup(h, parent, tok);
    if (b < 0) break;
    shared.push_back(b);
    chain.push_back(h);
    if (bm->blocks[b].ref == 0) ++shared_free;
    parent = h;
  }
  const int32_t fresh = n_blocks - static_cast<int32_t>(shared.size());
  if (fresh > bm->num_free - shared_free) return PKV_ERR_OUT_OF_BLOCKS;

  Sequence seq;
  try {
    seq.tokens.assign(token_ids, token_ids + num_tokens);
    seq.blocks.reserve(n_blocks);
    seq.chain = chain;
    bm->seqs.reserve(bm->seqs.size() + 1);
  } catch (const std::bad_alloc &) {
    return PKV_ERR_INVALID_ARG;
  }
  for (const int32_t b : shared) {
    if (bm->blocks[b].in_free) bm->unlink_free(b);
    ++bm->blocks[b].ref;
    seq.blocks.push_back(b);
  }
  for (int32_t i = static_cast<int32_t>(shared.size()); i < n_blocks; ++i) {
    const int32_t b = bm->take_fresh();
    seq.blocks.push_back(b);
    if (i < n_full) {  // full: findable from now on (its tokens are stored this step)
      const int32_t *tok = token_ids + static_cast<size_t>(i) * bs;
      const uint64_t h = chain_hash(parent, tok, bs);
      bm->publish(b, h, parent, tok);
      seq.chain.push_back(h);
      parent = h;
    }
  }
  *num_cached_tokens = static_cast<int32_t>(shared.size()) * bs;
  bm->seqs.emplace(seq_id, std::move(seq));
  return PKV_OK;
}

pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int32_t token_id) {
  if (bm == nullptr) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  Sequence &seq = it->second;
  const int32_t bs = bm->block_size;
  const int32_t n = static_cast<int32_t>(seq.tokens.size());
  if (n % bs == 0 && bm->num_free == 0) return PKV_ERR_OUT_OF_BLOCKS;
  try {
    seq.tokens.reserve(n + 1);
    seq.blocks.reserve(n / bs + 1);
    seq.chain.reserve(n / bs + 1);
  } catch (const std::bad_alloc &) {
    return PKV_ERR_INVALID_ARG;
  }
  if (n % bs == 0) seq.blocks.push_back(bm->take_fresh());
  seq.tokens.push_back(token_id);
  if ((n + 1) % bs == 0) {  // the last block is now full
    const int32_t i = n / bs;
    const uint64_t parent = i > 0 ? seq.chain[i - 1] : 0;
    const int32_t *tok = seq.tokens.data() + static_cast<size_t>(i) * bs;
    const uint64_t h = chain_hash(parent, tok, bs);
    bm->publish(seq.blocks[i], h, parent, tok);
    seq.chain.push_back(h);
  }
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
  if (bm == nullptr) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  // the last block first, so that a prompt's tail is handed out before its
  // (more shareable) head
  const std::vector<int32_t> &blocks = it->second.blocks;
  for (size_t k = blocks.size(); k-- > 0;) {
    Block &x = bm->blocks[blocks[k]];
    if (--x.ref == 0) bm->push_free(blocks[k]);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_num_tokens(const pkv_block_manager *bm, int64_t seq_id, int32_t *num_tokens) {
  if (bm == nullptr || num_tokens == nullptr) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  *num_tokens = static_cast<int32_t>(it->second.tokens.size());
  return PKV_OK;
}

pkv_status pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *row,
                              int32_t max_blocks, int32_t *num_blocks) {
  if (bm == nullptr || num_blocks == nullptr || max_blocks < 0 || (row == nullptr && max_blocks > 0))
    return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const std::vector<int32_t> &blocks = it->second.blocks;
  *num_blocks = static_cast<int32_t>(blocks.size());
  if (static_cast<int32_t>(blocks.size()) > max_blocks) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < max_blocks; ++i)
    row[i] = i < static_cast<int32_t>(blocks.size()) ? blocks[i] : -1;
  return PKV_OK;
}

pkv_status pkv_bm_slots(const pkv_block_manager *bm, int64_t seq_id, int32_t first,
                        int32_t count, int32_t *slots) {
  if (bm == nullptr || first < 0 || count < 0 || (slots == nullptr && count > 0))
    return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const Sequence &seq = it->second;
  if (static_cast<int64_t>(first) + count > static_cast<int64_t>(seq.tokens.size()))
    return PKV_ERR_INVALID_ARG;
  const int32_t bs = bm->block_size;
  for (int32_t i = 0; i < count; ++i) {
    const int32_t p = first + i;
    slots[i] = seq.blocks[p / bs] * bs + p % bs;
  }
  return PKV_OK;
}

}  // extern "C"
