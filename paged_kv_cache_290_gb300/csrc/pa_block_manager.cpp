// Host allocator of the paged KV pool with prefix caching (include/pa_block_manager.h).
//
// "Local_LLM_03_vLLM_Architecture", prefix-caching slide: each block's token content is hashed
// and requests with the same first N tokens share those N / block_size physical blocks;
// "Scaling inference with vLLM": requests that start alike physically share pages;
// "vLLM: LLM Inference That Doesn't Waste Your GPU", "PagedAttention: virtual memory for KV":
// paging makes eviction cheap and sharing copy-free.
//
// State: per physical block a reference count, whether it is in the prefix cache (then its
// chain key, salt and tokens), and its place in the evictable LRU list; per sequence its tokens,
// block list and the chain keys of its full blocks.  Every entry point first checks that it can
// finish (arguments, pool capacity), then mutates, so a failing call changes nothing.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pa_block_manager.h"

namespace pa {
int set_last_error(int status, const std::string& message);
}

namespace {

// 128-bit chained key of a full block.
struct Key {
  uint64_t a = 0, b = 0;
  bool operator==(const Key& o) const { return a == o.a && b == o.b; }
};
struct KeyHash {
  size_t operator()(const Key& k) const { return static_cast<size_t>(k.a ^ (k.b << 1)); }
};

// The SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014) as the mixing step of a two-lane multiplicative hash.
uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

Key chain_key(const Key& parent, int64_t salt, const int32_t* tokens, int32_t n) {
  uint64_t a = mix64(parent.a ^ 0x243F6A8885A308D3ull), b = mix64(parent.b ^ 0x13198A2E03707344ull);
  auto feed = [&](uint64_t w) {
    a = mix64(a ^ w);
    b = mix64(b + (w ^ 0xA4093822299F31D0ull));
  };
  feed(static_cast<uint64_t>(salt));
  for (int32_t i = 0; i < n; ++i) feed(static_cast<uint32_t>(tokens[i]));
  feed(static_cast<uint64_t>(n));
  return Key{a, b};
}

const Key kRootKey{0x6A09E667F3BCC908ull, 0xBB67AE8584CAA73Bull};

struct Block {
  int32_t ref = 0;
  bool cached = false;
  bool in_lru = false;
  Key key;
  int64_t salt = 0;
  std::vector<int32_t> tokens;  // the block's tokens while it is cached
  std::list<int32_t>::iterator lru_pos;
};

struct Seq {
  std::vector<int32_t> tokens;
  std::vector<int32_t> blocks;
  std::vector<Key> keys;  // chain key of each full block, in order
  int64_t salt = 0;
};

int fail(int status, const std::string& msg) { return pa::set_last_error(status, msg); }
int ok() { return pa::set_last_error(PA_OK, ""); }

}  // namespace

struct pa_block_manager {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  bool caching = true;
  std::vector<Block> blocks;
  std::vector<int32_t> free_list;  // unused, uncached blocks (a stack)
  std::list<int32_t> lru;          // unused cached blocks, least recently released first
  std::unordered_map<Key, int32_t, KeyHash> cache;
  std::unordered_map<int64_t, Seq> seqs;

  int32_t blocks_for(int64_t tokens) const {
    return static_cast<int32_t>((tokens + block_size - 1) / block_size);
  }
  int64_t available() const { return static_cast<int64_t>(free_list.size() + lru.size()); }

  void uncache(int32_t id) {
    Block& b = blocks[id];
    if (!b.cached) return;
    auto it = cache.find(b.key);
    if (it != cache.end() && it->second == id) cache.erase(it);
    b.cached = false;
    b.tokens.clear();
    if (b.in_lru) {
      lru.erase(b.lru_pos);
      b.in_lru = false;
      free_list.push_back(id);
    }
  }

  // Caller has checked available() first.
  int32_t take() {
    int32_t id;
    if (!free_list.empty()) {
      id = free_list.back();
      free_list.pop_back();
    } else {
      id = lru.front();
      Block& b = blocks[id];
      lru.pop_front();
      b.in_lru = false;
      auto it = cache.find(b.key);
      if (it != cache.end() && it->second == id) cache.erase(it);
      b.cached = false;
      b.tokens.clear();
    }
    blocks[id].ref = 1;
    return id;
  }

  void pin(int32_t id) {
    Block& b = blocks[id];
    if (b.ref == 0 && b.in_lru) {
      lru.erase(b.lru_pos);
      b.in_lru = false;
    }
    ++b.ref;
  }

  void release(int32_t id) {
    Block& b = blocks[id];
    if (--b.ref > 0) return;
    if (b.cached) {
      b.lru_pos = lru.insert(lru.end(), id);
      b.in_lru = true;
    } else {
      free_list.push_back(id);
    }
  }

  // Enter full block `id` (content tokens[0..bs), chain key k) into the cache unless an equal
  // block is already there.
  void offer(int32_t id, const Key& k, int64_t salt, const int32_t* tokens) {
    if (!caching || cache.count(k)) return;
    Block& b = blocks[id];
    b.cached = true;
    b.key = k;
    b.salt = salt;
    b.tokens.assign(tokens, tokens + block_size);
    cache.emplace(k, id);
  }

  // Cached block for chain key k whose own content is tokens (exact compare), or -1.
  int32_t lookup(const Key& k, int64_t salt, const int32_t* tokens) const {
    auto it = cache.find(k);
    if (it == cache.end()) return -1;
    const Block& b = blocks[it->second];
    if (b.salt != salt ||
        std::memcmp(b.tokens.data(), tokens, sizeof(int32_t) * static_cast<size_t>(block_size)))
      return -1;
    return it->second;
  }
};

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_caching) {
  if (num_blocks < 1 || block_size < 1) return nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->caching = prefix_caching != 0;
    bm->blocks.resize(static_cast<size_t>(num_blocks));
    bm->free_list.reserve(static_cast<size_t>(num_blocks));
    for (int32_t i = num_blocks - 1; i >= 0; --i) bm->free_list.push_back(i);  // 0 taken first
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                       int64_t cache_salt, int32_t* num_cached_tokens) {
  if (!bm || !tokens || n < 1) return fail(PA_ERR_INVALID_ARG, "add_sequence needs a manager and n >= 1 tokens");
  if (bm->seqs.count(seq_id)) return fail(PA_ERR_INVALID_ARG, "sequence id already present");
  const int32_t bs = bm->block_size, nblocks = bm->blocks_for(n), nfull = n / bs;
  // Chain keys of the full blocks; reuse cached ones up to, not including, the last token's block.
  std::vector<Key> keys(static_cast<size_t>(nfull));
  Key prev = kRootKey;
  for (int32_t i = 0; i < nfull; ++i) prev = keys[i] = chain_key(prev, cache_salt, tokens + i * bs, bs);
  std::vector<int32_t> hits;
  if (bm->caching)
    for (int32_t i = 0; i < (n - 1) / bs; ++i) {
      const int32_t id = bm->lookup(keys[i], cache_salt, tokens + i * bs);
      if (id < 0) break;
      hits.push_back(id);
    }
  int64_t pinned_from_lru = 0;
  for (int32_t id : hits) pinned_from_lru += bm->blocks[id].ref == 0 ? 1 : 0;
  const int64_t need = nblocks - static_cast<int64_t>(hits.size());
  if (need > bm->available() - pinned_from_lru)
    return fail(PA_ERR_NO_BLOCKS, "not enough free or evictable blocks for the prompt");

  Seq s;
  s.salt = cache_salt;
  s.tokens.assign(tokens, tokens + n);
  s.keys = keys;
  for (int32_t id : hits) {
    bm->pin(id);
    s.blocks.push_back(id);
  }
  for (int32_t i = static_cast<int32_t>(hits.size()); i < nblocks; ++i) {
    const int32_t id = bm->take();
    s.blocks.push_back(id);
    if (i < nfull) bm->offer(id, keys[i], cache_salt, tokens + i * bs);
  }
  bm->seqs.emplace(seq_id, std::move(s));
  if (num_cached_tokens) *num_cached_tokens = static_cast<int32_t>(hits.size()) * bs;
  return ok();
}

int pa_bm_append(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                 int32_t* copies, int32_t* num_copies) {
  if (!bm || !tokens || n < 1) return fail(PA_ERR_INVALID_ARG, "append needs a manager and n >= 1 tokens");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  Seq& s = it->second;
  const int32_t bs = bm->block_size;
  const int64_t len = static_cast<int64_t>(s.tokens.size());
  bool cow = false, reclaim = false;
  if (len % bs != 0) {
    const Block& last = bm->blocks[s.blocks.back()];
    cow = last.ref > 1;
    reclaim = !cow && last.cached;
  }
  if (cow && !copies) return fail(PA_ERR_INVALID_ARG, "a copy-on-write is needed but copies is NULL");
  const int64_t need = bm->blocks_for(len + n) - bm->blocks_for(len) + (cow ? 1 : 0);
  if (need > bm->available()) return fail(PA_ERR_NO_BLOCKS, "not enough free or evictable blocks to append");

  if (num_copies) *num_copies = 0;
  if (reclaim) bm->uncache(s.blocks.back());  // sole user of a truncated cached block
  if (cow) {
    const int32_t src = s.blocks.back(), dst = bm->take();
    bm->release(src);
    s.blocks.back() = dst;
    copies[0] = src;
    copies[1] = dst;
    if (num_copies) *num_copies = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    if (s.tokens.size() % bs == 0) s.blocks.push_back(bm->take());
    s.tokens.push_back(tokens[i]);
    if (s.tokens.size() % bs == 0) {  // a block just filled up: key it and offer it to the cache
      const size_t full = s.tokens.size() / bs;
      const Key prev = full > 1 ? s.keys[full - 2] : kRootKey;
      const int32_t* blk_tokens = s.tokens.data() + (full - 1) * bs;
      s.keys.push_back(chain_key(prev, s.salt, blk_tokens, bs));
      bm->offer(s.blocks[full - 1], s.keys.back(), s.salt, blk_tokens);
    }
  }
  return ok();
}

int pa_bm_truncate(pa_block_manager* bm, int64_t seq_id, int32_t new_len) {
  if (!bm) return fail(PA_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  Seq& s = it->second;
  if (new_len < 1 || new_len > static_cast<int64_t>(s.tokens.size()))
    return fail(PA_ERR_INVALID_ARG, "new_len must be in 1 .. length");
  const size_t keep = static_cast<size_t>(bm->blocks_for(new_len));
  for (size_t i = keep; i < s.blocks.size(); ++i) bm->release(s.blocks[i]);
  s.blocks.resize(keep);
  s.tokens.resize(static_cast<size_t>(new_len));
  s.keys.resize(static_cast<size_t>(new_len / bm->block_size));
  return ok();
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return fail(PA_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown parent sequence id");
  if (bm->seqs.count(child)) return fail(PA_ERR_INVALID_ARG, "child sequence id already present");
  Seq c = it->second;
  for (int32_t id : c.blocks) bm->pin(id);
  bm->seqs.emplace(child, std::move(c));
  return ok();
}

int pa_bm_free(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return fail(PA_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  for (int32_t id : it->second.blocks) bm->release(id);
  bm->seqs.erase(it);
  return ok();
}

int pa_bm_stats(const pa_block_manager* bm, int32_t* free_blocks, int32_t* evictable_blocks,
                int32_t* cached_blocks, int32_t* num_seqs) {
  if (!bm) return fail(PA_ERR_INVALID_ARG, "manager is NULL");
  if (free_blocks) *free_blocks = static_cast<int32_t>(bm->free_list.size());
  if (evictable_blocks) *evictable_blocks = static_cast<int32_t>(bm->lru.size());
  if (cached_blocks) *cached_blocks = static_cast<int32_t>(bm->cache.size());
  if (num_seqs) *num_seqs = static_cast<int32_t>(bm->seqs.size());
  return ok();
}

int pa_bm_sequence(const pa_block_manager* bm, int64_t seq_id, int32_t* length, int32_t* out,
                   int32_t max_blocks, int32_t* num_blocks) {
  if (!bm) return fail(PA_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  const Seq& s = it->second;
  const int32_t nb = static_cast<int32_t>(s.blocks.size());
  if (out && nb > max_blocks) return fail(PA_ERR_INVALID_ARG, "block table does not fit max_blocks");
  if (length) *length = static_cast<int32_t>(s.tokens.size());
  if (num_blocks) *num_blocks = nb;
  if (out) std::memcpy(out, s.blocks.data(), sizeof(int32_t) * static_cast<size_t>(nb));
  return ok();
}

int pa_bm_step_descriptor(const pa_block_manager* bm, const int64_t* seq_ids,
                          const int32_t* query_lens, int32_t n, int32_t max_blocks,
                          int32_t pad_block, int32_t* block_tables, int32_t* seq_lens,
                          int32_t* query_start_loc, int64_t* slot_mapping) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !query_lens || !block_tables ||
                                                   !seq_lens)) || !query_start_loc)
    return fail(PA_ERR_INVALID_ARG, "step_descriptor: NULL argument or negative size");
  std::vector<const Seq*> rows(static_cast<size_t>(n));
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "unknown sequence id in the step");
    const Seq& s = it->second;
    if (query_lens[i] < 0 || query_lens[i] > static_cast<int64_t>(s.tokens.size()))
      return fail(PA_ERR_INVALID_ARG, "query_len must be in 0 .. length");
    if (static_cast<int64_t>(s.blocks.size()) > max_blocks)
      return fail(PA_ERR_INVALID_ARG, "a block table does not fit max_blocks");
    rows[i] = &s;
    total += query_lens[i];
  }
  if (total > INT32_MAX) return fail(PA_ERR_INVALID_ARG, "too many query rows");
  if (total > 0 && !slot_mapping) return fail(PA_ERR_INVALID_ARG, "slot_mapping is NULL");
  const int32_t bs = bm->block_size;
  int64_t row = 0;
  query_start_loc[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    const Seq& s = *rows[i];
    int32_t* bt = block_tables + static_cast<int64_t>(i) * max_blocks;
    for (int32_t j = 0; j < max_blocks; ++j)
      bt[j] = j < static_cast<int32_t>(s.blocks.size()) ? s.blocks[j] : pad_block;
    const int64_t len = static_cast<int64_t>(s.tokens.size());
    seq_lens[i] = static_cast<int32_t>(len);
    for (int64_t p = len - query_lens[i]; p < len; ++p)
      slot_mapping[row++] = static_cast<int64_t>(s.blocks[p / bs]) * bs + p % bs;
    query_start_loc[i + 1] = static_cast<int32_t>(row);
  }
  return ok();
}

int pa_step_slot_mapping(int32_t n, const int32_t* seq_lens, const int32_t* query_lens,
                         const int32_t* block_tables, int64_t bt_stride, int32_t max_blocks,
                         int32_t block_size, int32_t* query_start_loc, int64_t* slot_mapping,
                         int64_t slot_capacity) {
  if (n < 0 || block_size < 1 || max_blocks < 0 || bt_stride < max_blocks || !query_start_loc ||
      (n > 0 && (!seq_lens || !query_lens || (max_blocks > 0 && !block_tables))))
    return fail(PA_ERR_INVALID_ARG, "step_slot_mapping: NULL argument or bad size");
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (query_lens[i] < 0 || query_lens[i] > seq_lens[i])
      return fail(PA_ERR_INVALID_ARG, "step_slot_mapping: need 0 <= query_len <= seq_len");
    if ((static_cast<int64_t>(seq_lens[i]) + block_size - 1) / block_size > max_blocks &&
        query_lens[i] > 0)
      return fail(PA_ERR_INVALID_ARG, "step_slot_mapping: a block table is too short");
    total += query_lens[i];
  }
  if (total > INT32_MAX) return fail(PA_ERR_INVALID_ARG, "step_slot_mapping: too many rows");
  if (total > slot_capacity || (total > 0 && !slot_mapping))
    return fail(PA_ERR_INVALID_ARG, "step_slot_mapping: slot_mapping holds " +
                                        std::to_string(slot_capacity) + " entries, " +
                                        std::to_string(total) + " needed");
  int64_t row = 0;
  query_start_loc[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* bt = block_tables + static_cast<int64_t>(i) * bt_stride;
    for (int64_t p = seq_lens[i] - query_lens[i]; p < seq_lens[i]; ++p)
      slot_mapping[row++] = static_cast<int64_t>(bt[p / block_size]) * block_size + p % block_size;
    query_start_loc[i + 1] = static_cast<int32_t>(row);
  }
  return ok();
}

}  // extern "C"
