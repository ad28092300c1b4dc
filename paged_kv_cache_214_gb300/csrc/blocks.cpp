// blocks.cpp — host-side block manager for the paged KV cache (include/pkv_blocks.h).
//
// "Nano-vLLM System Architecture Analysis", §2 Core Components, "Paged KV
// Cache": fixed-size blocks, a free list, a content hash -> block id table for
// prefix caching, and reference counts for sharing with copy-on-write.  §3
// "Lifecycle of a Request": the block tables and slot mappings it produces are
// the inputs the attention kernels read.

#include <stdint.h>

#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv_blocks.h"

namespace {

// 64-bit mixing step (the splitmix64 finaliser, a public-domain bit mixer).
inline uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ull;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebull;
  x ^= x >> 31;
  return x;
}

// Hash of a full block chained on the hash of the block before it.
uint64_t block_hash(uint64_t prev, const int32_t* tokens, int n) {
  uint64_t h = mix64(prev ^ 0x9e3779b97f4a7c15ull);
  for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tokens[i]));
  return h;
}

struct Block {
  int64_t ref = 0;
  bool hashed = false;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;  // content of a hashed (full) block
  uint64_t free_stamp = 0;      // identifies this block's current free-list entry
};

struct Seq {
  std::vector<int32_t> blocks;
  int64_t n_tokens = 0;
  uint64_t prev_hash = 0;         // hash of the last full block (0 if none)
  std::vector<int32_t> partial;   // tokens of the last, partly filled block
};

}  // namespace

struct pkv_block_manager {
  int64_t num_blocks;
  int bs;
  std::vector<Block> blocks;
  std::deque<std::pair<int32_t, uint64_t>> free_list;  // (block, stamp); stale entries skipped
  int64_t n_free;
  uint64_t stamp = 0;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Seq> seqs;

  void push_free(int32_t b) {
    blocks[b].free_stamp = ++stamp;
    free_list.emplace_back(b, blocks[b].free_stamp);
    ++n_free;
  }

  // Take the oldest free block for new content; its cached identity is dropped.
  int32_t take_fresh() {
    while (!free_list.empty()) {
      const auto e = free_list.front();
      free_list.pop_front();
      Block& blk = blocks[e.first];
      if (blk.ref != 0 || blk.free_stamp != e.second) continue;  // stale entry
      if (blk.hashed) {
        auto it = by_hash.find(blk.hash);
        if (it != by_hash.end() && it->second == e.first) by_hash.erase(it);
        blk.hashed = false;
        blk.tokens.clear();
      }
      blk.ref = 1;
      blk.free_stamp = 0;
      --n_free;
      return e.first;
    }
    return -1;
  }

  // Claim a cached block (a prefix-cache hit); it may be in use or free.
  void claim(int32_t b) {
    Block& blk = blocks[b];
    if (blk.ref == 0) {
      blk.free_stamp = 0;  // its free-list entry becomes stale
      --n_free;
    }
    ++blk.ref;
  }

  void release(int32_t b) {
    if (--blocks[b].ref == 0) push_free(b);
  }

  // A cached block holding exactly these tokens after prefix hash `h`, or -1.
  int32_t lookup(uint64_t h, const int32_t* tokens) const {
    auto it = by_hash.find(h);
    if (it == by_hash.end()) return -1;
    const Block& blk = blocks[it->second];
    if (!blk.hashed || blk.hash != h || static_cast<int>(blk.tokens.size()) != bs) return -1;
    for (int i = 0; i < bs; ++i)
      if (blk.tokens[i] != tokens[i]) return -1;
    return it->second;
  }

  void register_full(int32_t b, uint64_t h, const int32_t* tokens) {
    Block& blk = blocks[b];
    blk.hashed = true;
    blk.hash = h;
    blk.tokens.assign(tokens, tokens + bs);
    by_hash[h] = b;
  }
};

extern "C" {

pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size) {
  if (num_blocks < 0 || num_blocks > INT32_MAX || block_size < 1) return nullptr;
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->bs = block_size;
  bm->n_free = 0;
  bm->blocks.resize(static_cast<size_t>(num_blocks));
  for (int64_t b = 0; b < num_blocks; ++b) bm->push_free(static_cast<int32_t>(b));
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
  return bm ? bm->n_free : PKV_BM_ERR_ARG;
}

int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                        int64_t n_tokens, int64_t* num_cached_tokens) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PKV_BM_ERR_ARG;
  if (bm->seqs.count(seq_id)) return PKV_BM_ERR_EXISTS;
  const int bs = bm->bs;
  const int64_t n_full = n_tokens / bs;
  const bool partial = n_tokens % bs != 0;
  // Plan: leading full blocks that hit the cache, then fresh blocks.
  std::vector<int32_t> hits;
  std::vector<uint64_t> hashes(static_cast<size_t>(n_full));
  uint64_t h = 0;
  int64_t need_free = 0;
  bool missed = false;
  for (int64_t i = 0; i < n_full; ++i) {
    h = block_hash(h, tokens + i * bs, bs);
    hashes[static_cast<size_t>(i)] = h;
    if (missed) continue;
    const int32_t b = bm->lookup(h, tokens + i * bs);
    if (b < 0) {
      missed = true;
      continue;
    }
    hits.push_back(b);
    if (bm->blocks[b].ref == 0) ++need_free;  // taking a cached free block uses one
  }
  need_free += (n_full - static_cast<int64_t>(hits.size())) + (partial ? 1 : 0);
  if (need_free > bm->n_free) return PKV_BM_ERR_NO_BLOCKS;

  Seq s;
  for (int32_t b : hits) {
    bm->claim(b);
    s.blocks.push_back(b);
  }
  for (int64_t i = static_cast<int64_t>(hits.size()); i < n_full; ++i) {
    const int32_t b = bm->take_fresh();
    bm->register_full(b, hashes[static_cast<size_t>(i)], tokens + i * bs);
    s.blocks.push_back(b);
  }
  if (partial) {
    s.blocks.push_back(bm->take_fresh());
    s.partial.assign(tokens + n_full * bs, tokens + n_tokens);
  }
  s.n_tokens = n_tokens;
  s.prev_hash = n_full > 0 ? hashes[static_cast<size_t>(n_full - 1)] : 0;
  bm->seqs.emplace(seq_id, std::move(s));
  if (num_cached_tokens) *num_cached_tokens = static_cast<int64_t>(hits.size()) * bs;
  return PKV_BM_OK;
}

int pkv_bm_append_token(pkv_block_manager* bm, int64_t seq_id, int32_t token, int64_t* slot,
                        int32_t* copy_src, int32_t* copy_dst) {
  if (!bm) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_BM_ERR_NO_SEQ;
  Seq& s = it->second;
  const int bs = bm->bs;
  const int64_t pos = s.n_tokens;
  int32_t src = -1, dst = -1;
  if (pos % bs == 0) {  // the last block is full (or there is none): a new block
    if (bm->n_free < 1) return PKV_BM_ERR_NO_BLOCKS;
    s.blocks.push_back(bm->take_fresh());
  } else if (bm->blocks[s.blocks.back()].ref > 1) {  // shared and partly filled
    if (bm->n_free < 1) return PKV_BM_ERR_NO_BLOCKS;
    src = s.blocks.back();
    dst = bm->take_fresh();
    bm->release(src);
    s.blocks.back() = dst;
  }
  const int32_t b = s.blocks.back();
  if (slot) *slot = static_cast<int64_t>(b) * bs + pos % bs;
  if (copy_src) *copy_src = src;
  if (copy_dst) *copy_dst = dst;
  s.partial.push_back(token);
  s.n_tokens = pos + 1;
  if (s.n_tokens % bs == 0) {  // the block just filled up: cacheable from now on
    const uint64_t h = block_hash(s.prev_hash, s.partial.data(), bs);
    bm->register_full(b, h, s.partial.data());
    s.prev_hash = h;
    s.partial.clear();
  }
  return PKV_BM_OK;
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end()) return PKV_BM_ERR_NO_SEQ;
  if (bm->seqs.count(child_id)) return PKV_BM_ERR_EXISTS;
  Seq child = it->second;
  for (int32_t b : child.blocks) bm->claim(b);
  bm->seqs.emplace(child_id, std::move(child));
  return PKV_BM_OK;
}

int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_BM_ERR_NO_SEQ;
  const std::vector<int32_t>& blocks = it->second.blocks;
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) bm->release(*b);
  bm->seqs.erase(it);
  return PKV_BM_OK;
}

int64_t pkv_bm_num_tokens(const pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? PKV_BM_ERR_NO_SEQ : it->second.n_tokens;
}

int64_t pkv_bm_num_blocks(const pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? PKV_BM_ERR_NO_SEQ
                              : static_cast<int64_t>(it->second.blocks.size());
}

int pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out,
                       int64_t max_blocks) {
  if (!bm || !out || max_blocks < 0) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_BM_ERR_NO_SEQ;
  const std::vector<int32_t>& blocks = it->second.blocks;
  if (static_cast<int64_t>(blocks.size()) > max_blocks) return PKV_BM_ERR_SMALL;
  for (int64_t i = 0; i < max_blocks; ++i)
    out[i] = i < static_cast<int64_t>(blocks.size()) ? blocks[static_cast<size_t>(i)] : -1;
  return PKV_BM_OK;
}

int pkv_bm_slot_mapping(const pkv_block_manager* bm, int64_t seq_id, int64_t begin,
                        int64_t end, int32_t* out) {
  if (!bm || (end > begin && !out) || begin < 0 || end < begin) return PKV_BM_ERR_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_BM_ERR_NO_SEQ;
  const Seq& s = it->second;
  if (end > s.n_tokens) return PKV_BM_ERR_ARG;
  for (int64_t p = begin; p < end; ++p) {
    const int64_t slot =
        static_cast<int64_t>(s.blocks[static_cast<size_t>(p / bm->bs)]) * bm->bs + p % bm->bs;
    if (slot > INT32_MAX) return PKV_BM_ERR_ARG;
    out[p - begin] = static_cast<int32_t>(slot);
  }
  return PKV_BM_OK;
}

int64_t pkv_bm_ref_count(const pkv_block_manager* bm, int64_t block_id) {
  if (!bm || block_id < 0 || block_id >= bm->num_blocks) return PKV_BM_ERR_ARG;
  return bm->blocks[static_cast<size_t>(block_id)].ref;
}

}  // extern "C"
