// pkv_blocks.cu -- host-side KV block manager (C ABI in include/pkv_blocks.h).
//
// Block pool, per-sequence block tables, reference counts, a chained-hash
// prefix cache and a free queue in release order ("How to design an LLM
// serving system (a vLLM deep dive)", "PagedAttention (vLLM KV manager)" and
// "Latency and scaling knobs"; nanoserve, "Prefix caching").  Host code only.
#include <stdint.h>
#include <string.h>

#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv_blocks.h"
#include "pkv_kernels.h"

namespace {

constexpr int32_t kNone = -1;

// 64-bit FNV-1a over the parent hash and a block's token ids: the content
// address of a full block (the block and every block before it).
uint64_t chain_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](uint64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= (v >> (8 * i)) & 0xFFu;
      h *= 1099511628211ull;
    }
  };
  mix(parent);
  for (int32_t i = 0; i < n; ++i) mix(static_cast<uint32_t>(tokens[i]));
  return h;
}

struct Sequence {
  std::vector<int32_t> blocks;  // block table
  std::vector<int32_t> tokens;  // every token id so far (prompt first)
  int32_t n_tokens = 0;         // tokens whose K/V are (or are being) in the cache
  int32_t n_hashed = 0;         // leading full blocks registered in the prefix cache
  uint64_t last_hash = 0;       // hash of block n_hashed - 1 (0 before the first)
};

}  // namespace

struct pkv_block_manager {
  int32_t num_blocks = 0, bs = 0;
  std::vector<int32_t> ref;          // reference count per block
  std::vector<uint8_t> hashed;       // block has a registered hash
  std::vector<uint64_t> hash;        // its hash
  std::vector<int32_t> content;      // token ids of hashed blocks [num_blocks * bs]
  std::vector<int32_t> prev, next;   // free queue links (kNone at the ends)
  int32_t head = kNone, tail = kNone, n_free = 0, n_hashed = 0;
  std::vector<uint8_t> in_queue;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Sequence> seqs;
  int64_t hit_blocks = 0, evictions = 0;

  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = kNone;
    if (tail != kNone) next[tail] = b; else head = b;
    tail = b;
    in_queue[b] = 1;
    ++n_free;
  }
  void unlink(int32_t b) {
    if (prev[b] != kNone) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] != kNone) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = kNone;
    in_queue[b] = 0;
    --n_free;
  }
  // the least recently released free block; a cached one loses its hash
  int32_t pop_block() {
    const int32_t b = head;
    unlink(b);
    if (hashed[b]) {
      auto it = by_hash.find(hash[b]);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
      hashed[b] = 0;
      --n_hashed;
      ++evictions;
    }
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) push_back(b);
  }
  // blocks that appending n tokens to s needs beyond the ones it holds
  int32_t blocks_needed(const Sequence& s, int32_t n) const {
    const int64_t total = ((int64_t)s.n_tokens + n + bs - 1) / bs;
    return (int32_t)(total - (int64_t)s.blocks.size());
  }
  // registers the full blocks of s that are not yet in the prefix cache
  void publish(Sequence& s) {
    while ((int64_t)(s.n_hashed + 1) * bs <= s.n_tokens) {
      const int32_t i = s.n_hashed;
      const int32_t* toks = s.tokens.data() + (int64_t)i * bs;
      const uint64_t h = chain_hash(s.last_hash, toks, bs);
      const int32_t b = s.blocks[i];
      if (!hashed[b] && by_hash.find(h) == by_hash.end()) {
        hashed[b] = 1;
        hash[b] = h;
        memcpy(content.data() + (int64_t)b * bs, toks, sizeof(int32_t) * bs);
        by_hash.emplace(h, b);
        ++n_hashed;
      }
      s.last_hash = h;
      ++s.n_hashed;
    }
  }
  // appends tokens to s; the caller has checked that the pool suffices
  void append(Sequence& s, const int32_t* toks, int32_t n, int32_t* slots) {
    for (int32_t i = 0; i < n; ++i) {
      const int32_t p = s.n_tokens + i;
      if (p / bs >= (int32_t)s.blocks.size()) s.blocks.push_back(pop_block());
      if (slots) slots[i] = s.blocks[p / bs] * bs + p % bs;
      if (p >= (int32_t)s.tokens.size()) s.tokens.push_back(toks[i]);
      else s.tokens[p] = toks[i];
    }
    s.n_tokens += n;
    publish(s);
  }
};

namespace {

pkv_status fail(pkv_status st, const std::string& msg) { return pkv::record_failure(st, msg); }

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out) {
  if (out == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, "out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || block_size < 1 || (int64_t)num_blocks * block_size > INT32_MAX)
    return fail(PKV_ERR_INVALID_ARGUMENT, "need num_blocks >= 1, block_size >= 1 and "
                                          "num_blocks * block_size within int32");
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, "out of host memory");
  bm->num_blocks = num_blocks;
  bm->bs = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->hashed.assign(num_blocks, 0);
  bm->hash.assign(num_blocks, 0);
  bm->content.assign((size_t)num_blocks * block_size, 0);
  bm->prev.assign(num_blocks, kNone);
  bm->next.assign(num_blocks, kNone);
  bm->in_queue.assign(num_blocks, 0);
  for (int32_t b = 0; b < num_blocks; ++b) bm->push_back(b);
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* prompt, int32_t n,
                               int32_t* cached_tokens) {
  if (bm == nullptr || cached_tokens == nullptr || (n > 0 && prompt == nullptr) || n < 0)
    return fail(PKV_ERR_INVALID_ARGUMENT, "bad arguments to pkv_bm_add_sequence");
  if (bm->seqs.count(seq_id)) return fail(PKV_ERR_INVALID_ARGUMENT, "sequence id already live");
  Sequence s;
  s.tokens.assign(prompt, prompt + n);
  // longest cached prefix of full blocks, leaving the last prompt token to compute
  const int32_t max_blocks = n > 0 ? (n - 1) / bm->bs : 0;
  uint64_t h = 0;
  for (int32_t i = 0; i < max_blocks; ++i) {
    const int32_t* toks = prompt + (int64_t)i * bm->bs;
    const uint64_t hi = chain_hash(h, toks, bm->bs);
    auto it = bm->by_hash.find(hi);
    if (it == bm->by_hash.end()) break;
    const int32_t b = it->second;
    if (memcmp(bm->content.data() + (int64_t)b * bm->bs, toks, sizeof(int32_t) * bm->bs) != 0) break;
    if (bm->ref[b] == 0) bm->unlink(b);  // a cached free block comes back into use
    ++bm->ref[b];
    s.blocks.push_back(b);
    h = hi;
    ++bm->hit_blocks;
  }
  s.n_hashed = (int32_t)s.blocks.size();
  s.n_tokens = s.n_hashed * bm->bs;
  s.last_hash = h;
  *cached_tokens = s.n_tokens;
  bm->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n, int32_t* slots) {
  if (bm == nullptr || n < 0 || (n > 0 && (tokens == nullptr || slots == nullptr)))
    return fail(PKV_ERR_INVALID_ARGUMENT, "bad arguments to pkv_bm_append");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence id");
  Sequence& s = it->second;
  if ((int64_t)s.n_tokens + n > INT32_MAX) return fail(PKV_ERR_INVALID_ARGUMENT, "sequence too long");
  const int32_t need = bm->blocks_needed(s, n);
  if (need > bm->n_free)
    return fail(PKV_ERR_OUT_OF_BLOCKS, "append needs " + std::to_string(need) + " blocks, " +
                                           std::to_string(bm->n_free) + " free");
  bm->append(s, tokens, n, slots);
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, "bm is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence id");
  // the last blocks first, so that a prompt's leading blocks stay cached longest
  const std::vector<int32_t>& bl = it->second.blocks;
  for (size_t i = bl.size(); i-- > 0;) bm->release(bl[i]);
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* table, int32_t capacity,
                              int32_t* n_blocks, int32_t* n_tokens) {
  if (bm == nullptr || n_blocks == nullptr || n_tokens == nullptr || capacity < 0 ||
      (capacity > 0 && table == nullptr))
    return fail(PKV_ERR_INVALID_ARGUMENT, "bad arguments to pkv_bm_block_table");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence id");
  const Sequence& s = it->second;
  const int32_t nb = (int32_t)s.blocks.size();
  for (int32_t i = 0; i < nb && i < capacity; ++i) table[i] = s.blocks[i];
  *n_blocks = nb;
  *n_tokens = s.n_tokens;
  return PKV_OK;
}

pkv_status pkv_bm_build_step(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* n_new,
                             const int32_t* tokens, int32_t B, int32_t max_blocks, int32_t* cu_seqlens_q,
                             int32_t* seq_lens, int32_t* block_tables, int32_t* slot_mapping) {
  if (bm == nullptr || B < 0 || max_blocks < 0 || (B > 0 && (seq_ids == nullptr || n_new == nullptr ||
                                                            cu_seqlens_q == nullptr || seq_lens == nullptr ||
                                                            block_tables == nullptr)))
    return fail(PKV_ERR_INVALID_ARGUMENT, "bad arguments to pkv_bm_build_step");
  if (cu_seqlens_q != nullptr) cu_seqlens_q[0] = 0;
  // check everything before changing anything
  std::vector<Sequence*> ss(B);
  int64_t need = 0, total = 0;
  for (int32_t b = 0; b < B; ++b) {
    auto it = bm->seqs.find(seq_ids[b]);
    if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence id in step");
    if (n_new[b] < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "negative token count");
    for (int32_t c = 0; c < b; ++c)
      if (ss[c] == &it->second) return fail(PKV_ERR_INVALID_ARGUMENT, "sequence twice in one step");
    ss[b] = &it->second;
    const int64_t len = (int64_t)ss[b]->n_tokens + n_new[b];
    if ((len + bm->bs - 1) / bm->bs > max_blocks)
      return fail(PKV_ERR_INVALID_ARGUMENT, "a sequence needs more than max_blocks blocks");
    need += bm->blocks_needed(*ss[b], n_new[b]);
    total += n_new[b];
  }
  if (total > INT32_MAX) return fail(PKV_ERR_INVALID_ARGUMENT, "step too large");
  if (total > 0 && (tokens == nullptr || slot_mapping == nullptr))
    return fail(PKV_ERR_INVALID_ARGUMENT, "tokens and slot_mapping are required");
  if (need > bm->n_free)
    return fail(PKV_ERR_OUT_OF_BLOCKS, "step needs " + std::to_string(need) + " blocks, " +
                                           std::to_string(bm->n_free) + " free");
  int32_t t = 0;
  for (int32_t b = 0; b < B; ++b) {
    Sequence& s = *ss[b];
    bm->append(s, tokens + t, n_new[b], slot_mapping + t);
    t += n_new[b];
    cu_seqlens_q[b + 1] = t;
    seq_lens[b] = s.n_tokens;
    int32_t* row = block_tables + (int64_t)b * max_blocks;
    const int32_t nb = (int32_t)s.blocks.size();
    for (int32_t i = 0; i < max_blocks; ++i) row[i] = i < nb ? s.blocks[i] : -1;
  }
  return PKV_OK;
}

pkv_status pkv_bm_stats(const pkv_block_manager* bm, pkv_bm_stats_t* out) {
  if (bm == nullptr || out == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, "bad arguments to pkv_bm_stats");
  out->num_blocks = bm->num_blocks;
  out->free_blocks = bm->n_free;
  out->cached_blocks = bm->n_hashed;
  out->num_sequences = (int32_t)bm->seqs.size();
  out->prefix_hit_blocks = bm->hit_blocks;
  out->evictions = bm->evictions;
  return PKV_OK;
}

}  // extern "C"
