// pa_block_manager.cpp - host KV block manager (C ABI in include/pa_block_manager.h).
//
// Free queue: a doubly linked list over block ids, so a cached block that is
// hit while it sits in the queue leaves it in O(1) ("PagedAttention是什麼？",
// sections "vLLM v1的Block Pool" and "Eviction與Free Queue").  New blocks come
// from the head, released blocks go to the tail, so the least recently
// released cached block is the first to be reused (and evicted from the cache).
//
// Prefix cache ("PagedAttention 详解：缓存的存储结构", section "使用流程"): each full
// prompt block gets a chained hash h_i = H(h_{i-1}, tokens of block i), with
// h_{-1} = 0 and H = 64-bit FNV-1a over the little-endian bytes of h_{i-1}
// followed by those of the block's int32 tokens.  A hit is confirmed against
// the stored parent hash and tokens, so a hash collision never aliases content.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_block_manager.h"

namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv1a_bytes(uint64_t h, const unsigned char* p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= kFnvPrime;
  }
  return h;
}

uint64_t chain_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  unsigned char buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = (unsigned char)(parent >> (8 * i));
  uint64_t h = fnv1a_bytes(kFnvOffset, buf, 8);
  for (int32_t t = 0; t < n; ++t) {
    const uint32_t u = (uint32_t)tokens[t];
    unsigned char b[4] = {(unsigned char)u, (unsigned char)(u >> 8), (unsigned char)(u >> 16),
                          (unsigned char)(u >> 24)};
    h = fnv1a_bytes(h, b, 4);
  }
  return h;
}

// splitmix64 (Steele, Lea, Flood 2014): the generator behind the optional shuffle.
uint64_t splitmix64(uint64_t& state) {
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct Seq {
  std::vector<int32_t> blocks;
  int32_t len = 0;
};

}  // namespace

struct pa_block_manager {
  int32_t num_blocks = 0, block_size = 0;
  std::vector<int32_t> ref, prev, next;
  std::vector<uint8_t> in_queue;
  int32_t head = -1, tail = -1, free_count = 0;
  // prefix cache
  std::vector<uint8_t> cached;
  std::vector<uint64_t> hash, parent_hash;
  std::vector<std::vector<int32_t>> tokens;
  std::unordered_map<uint64_t, int32_t> cache;
  std::unordered_map<int64_t, Seq> seqs;

  void push_tail(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    in_queue[b] = 1;
    ++free_count;
  }
  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    in_queue[b] = 0;
    --free_count;
  }
  void uncache(int32_t b) {
    if (!cached[b]) return;
    auto it = cache.find(hash[b]);
    if (it != cache.end() && it->second == b) cache.erase(it);
    cached[b] = 0;
    tokens[b].clear();
  }
  // a fresh block from the head of the free queue (its old cache entry is dropped)
  int32_t take() {
    const int32_t b = head;
    unlink(b);
    uncache(b);
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) push_tail(b);
  }
  int32_t blocks_for(int32_t n) const { return (n + block_size - 1) / block_size; }
};

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, uint64_t shuffle_seed) {
  if (num_blocks < 0 || block_size <= 0) return nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (bm == nullptr) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->prev.assign(num_blocks, -1);
  bm->next.assign(num_blocks, -1);
  bm->in_queue.assign(num_blocks, 0);
  bm->cached.assign(num_blocks, 0);
  bm->hash.assign(num_blocks, 0);
  bm->parent_hash.assign(num_blocks, 0);
  bm->tokens.assign(num_blocks, {});
  std::vector<int32_t> order(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) order[i] = i;
  if (shuffle_seed != 0) {
    uint64_t state = shuffle_seed;
    for (int32_t i = num_blocks - 1; i > 0; --i) {
      const int32_t j = (int32_t)(splitmix64(state) % (uint64_t)(i + 1));
      const int32_t t = order[i];
      order[i] = order[j];
      order[j] = t;
    }
  }
  for (int32_t b : order) bm->push_tail(b);
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free(const pa_block_manager* bm) { return bm ? bm->free_count : PA_BM_ERR_INVALID_ARG; }

int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

int pa_bm_allocate(pa_block_manager* bm, int64_t seq, int32_t num_tokens) {
  if (!bm || num_tokens < 0) return PA_BM_ERR_INVALID_ARG;
  if (bm->seqs.count(seq)) return PA_BM_ERR_SEQ_EXISTS;
  const int32_t need = bm->blocks_for(num_tokens);
  if (need > bm->free_count) return PA_BM_ERR_NO_BLOCKS;
  Seq s;
  s.len = num_tokens;
  s.blocks.reserve(need);
  for (int32_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  bm->seqs.emplace(seq, std::move(s));
  return PA_BM_OK;
}

int pa_bm_allocate_with_prefix(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int32_t num_tokens,
                               int32_t* num_hit_blocks) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_BM_ERR_INVALID_ARG;
  if (bm->seqs.count(seq)) return PA_BM_ERR_SEQ_EXISTS;
  const int32_t B = bm->block_size;
  const int32_t full = num_tokens / B;
  const int32_t need = bm->blocks_for(num_tokens);
  // pass 1: chained hashes and the leading run of cache hits
  std::vector<uint64_t> h(full);
  std::vector<int32_t> hit;
  uint64_t parent = 0;
  bool chain = true;
  for (int32_t i = 0; i < full; ++i) {
    h[i] = chain_hash(parent, tokens + (size_t)i * B, B);
    if (chain) {
      auto it = bm->cache.find(h[i]);
      const int32_t b = it == bm->cache.end() ? -1 : it->second;
      if (b >= 0 && bm->parent_hash[b] == parent &&
          std::memcmp(bm->tokens[b].data(), tokens + (size_t)i * B, sizeof(int32_t) * B) == 0)
        hit.push_back(b);
      else
        chain = false;
    }
    parent = h[i];
  }
  // blocks that must come from the free queue: misses, minus hit blocks that sit in it
  int32_t queued_hits = 0;
  for (int32_t b : hit) queued_hits += bm->in_queue[b] ? 1 : 0;
  const int32_t fresh = need - (int32_t)hit.size();
  if (fresh > bm->free_count - queued_hits) return PA_BM_ERR_NO_BLOCKS;
  // pass 2: commit
  Seq s;
  s.len = num_tokens;
  s.blocks.reserve(need);
  for (int32_t b : hit) {
    if (bm->in_queue[b]) bm->unlink(b);
    ++bm->ref[b];
    s.blocks.push_back(b);
  }
  for (int32_t i = (int32_t)hit.size(); i < need; ++i) {
    const int32_t b = bm->take();
    s.blocks.push_back(b);
    if (i < full && !bm->cache.count(h[i])) {  // enter the new full block in the prefix cache
      bm->cached[b] = 1;
      bm->hash[b] = h[i];
      bm->parent_hash[b] = i == 0 ? 0 : h[i - 1];
      bm->tokens[b].assign(tokens + (size_t)i * B, tokens + (size_t)(i + 1) * B);
      bm->cache.emplace(h[i], b);
    }
  }
  bm->seqs.emplace(seq, std::move(s));
  if (num_hit_blocks) *num_hit_blocks = (int32_t)hit.size();
  return PA_BM_OK;
}

int pa_bm_append_slot(pa_block_manager* bm, int64_t seq, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  if (!bm || !slot) return PA_BM_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_BM_ERR_UNKNOWN_SEQ;
  Seq& s = it->second;
  const int32_t B = bm->block_size;
  const int32_t off = s.len % B;
  int32_t src = -1, dst = -1;
  if (off == 0) {  // the last block is full (or there is none): append a fresh block
    if (bm->free_count == 0) return PA_BM_ERR_NO_BLOCKS;
    s.blocks.push_back(bm->take());
  } else if (bm->ref[s.blocks.back()] > 1) {  // partly filled and shared: copy-on-write
    if (bm->free_count == 0) return PA_BM_ERR_NO_BLOCKS;
    src = s.blocks.back();
    dst = bm->take();
    s.blocks.back() = dst;
    bm->release(src);
  }
  *slot = (int64_t)s.blocks.back() * B + off;
  ++s.len;
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  return PA_BM_OK;
}

int pa_bm_append_slots(pa_block_manager* bm, const int64_t* seqs, int32_t n, int64_t* slots, int32_t* pairs,
                       int32_t* num_pairs) {
  if (!bm || n < 0 || (n > 0 && (!seqs || !slots || !pairs)) || !num_pairs) return PA_BM_ERR_INVALID_ARG;
  *num_pairs = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t src, dst;
    const int rc = pa_bm_append_slot(bm, seqs[i], &slots[i], &src, &dst);
    if (rc != PA_BM_OK) return rc;
    if (src >= 0) {
      pairs[2 * *num_pairs] = src;
      pairs[2 * *num_pairs + 1] = dst;
      ++*num_pairs;
    }
  }
  return PA_BM_OK;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return PA_BM_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PA_BM_ERR_UNKNOWN_SEQ;
  if (bm->seqs.count(child)) return PA_BM_ERR_SEQ_EXISTS;
  Seq s = it->second;  // copy of the parent's table
  for (int32_t b : s.blocks) ++bm->ref[b];
  bm->seqs.emplace(child, std::move(s));
  return PA_BM_OK;
}

int pa_bm_free(pa_block_manager* bm, int64_t seq) {
  if (!bm) return PA_BM_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_BM_ERR_UNKNOWN_SEQ;
  for (int32_t b : it->second.blocks) bm->release(b);
  bm->seqs.erase(it);
  return PA_BM_OK;
}

int32_t pa_bm_seq_len(const pa_block_manager* bm, int64_t seq) {
  if (!bm) return PA_BM_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? PA_BM_ERR_UNKNOWN_SEQ : it->second.len;
}

int32_t pa_bm_num_seq_blocks(const pa_block_manager* bm, int64_t seq) {
  if (!bm) return PA_BM_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? PA_BM_ERR_UNKNOWN_SEQ : (int32_t)it->second.blocks.size();
}

int32_t pa_bm_max_seq_blocks(const pa_block_manager* bm, const int64_t* seqs, int32_t n) {
  if (!bm || n < 0 || (n > 0 && !seqs)) return PA_BM_ERR_INVALID_ARG;
  int32_t width = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_BM_ERR_UNKNOWN_SEQ;
    if ((int32_t)it->second.blocks.size() > width) width = (int32_t)it->second.blocks.size();
  }
  return width;
}

int pa_bm_build_tables(const pa_block_manager* bm, const int64_t* seqs, int32_t n, int32_t width,
                       int32_t* tables_out, int32_t* lens_out) {
  if (!bm || n < 0 || width < 0 || (n > 0 && (!seqs || !tables_out || !lens_out))) return PA_BM_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_BM_ERR_UNKNOWN_SEQ;
    if ((int32_t)it->second.blocks.size() > width) return PA_BM_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const Seq& s = bm->seqs.find(seqs[i])->second;
    int32_t* row = tables_out + (size_t)i * width;
    const int32_t nb = (int32_t)s.blocks.size();
    for (int32_t j = 0; j < nb; ++j) row[j] = s.blocks[j];
    for (int32_t j = nb; j < width; ++j) row[j] = 0;
    lens_out[i] = s.len;
  }
  return PA_BM_OK;
}

}  // extern "C"
