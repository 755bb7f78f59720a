// Host block manager: free list, per-sequence block tables, reference counts,
// fork / copy-on-write / free.  Plain C++17, no GPU.
//
// Follows "vLLM High-Performance Inference Engine: PagedAttention Principles
// and Deployment Guide" ("PagedAttention Architecture Deep Dive": block table
// with ref_count, pages shared between sequences), "vLLM Guide: High-Throughput
// Multi-GPU LLM Serving with PagedAttention" ("What Is PagedAttention?": blocks
// allocated on demand, shared prefixes -- system prompts, few-shot examples,
// earlier turns of a conversation -- with copy-on-write) and "Configuring
// vLLM and PagedAttention for High Throughput Enterprise LLM Serving"
// ("High-Throughput Batching": pages go back to the free pool on <eos>, and
// the preemptive-swapping answer: a paused request's pages move to host RAM
// and come back when device blocks free up; "Zero-Copy Prefix Caching &
// Shared Sampling": requests with a common prefix point at the same pages).
#include <algorithm>
#include <climits>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;  // device block ids, or host block ids while swapped out
  int len = 0;
  bool swapped = false;
  uint64_t stamp = 0;  // last batch call that listed this sequence
  // Token ids are known for every token so far (admitted with its prompt's
  // ids, every append given its id): then `tail` holds the ids of the partly
  // filled last block (room for a whole block is reserved), and a block that
  // an append fills is registered in the prefix cache.
  bool tracked = false;
  std::vector<int32_t> tail;
};

// No C++ exception leaves an entry point: a failed allocation (the only
// exception these containers throw) becomes PA_ERR_OOM.  Each entry point
// makes its allocations before it changes any state, or undoes its changes,
// so that a failure leaves the manager as it was.
template <class F>
int guarded(F &&f) noexcept {
  try {
    return f();
  } catch (const std::bad_alloc &) {
    return PA_ERR_OOM;
  } catch (...) {
    return PA_ERR_INVALID;
  }
}

}  // namespace

struct pa_bm {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ref;  // per block, 0 = free
  // Free blocks in two tiers.  Blocks holding no cached content are handed
  // out first, most recently freed first (a stack; initially in increasing
  // id order).  Free blocks still in the prefix cache are handed out only
  // when no other is left, least recently freed first (a list, oldest at its
  // head), so the content most likely to be asked for again stays longest.
  // A block is freed no earlier than the blocks that continue it (whoever
  // holds a block holds the ones before it), so leaves leave the cache first.
  std::vector<int32_t> stack;                 // free, not cached
  std::vector<int32_t> lru_prev, lru_next;    // free and cached
  int32_t lru_head = -1, lru_tail = -1;
  std::vector<uint8_t> where;                 // per block: 0 in use, 1 on the stack, 2 in the list
  int nfree = 0;                              // blocks with ref 0
  // Prefix cache: full blocks registered by content.  A block's key is its
  // parent (the block before it in the sequence, -1 for the first) and its B
  // token ids; lookups compare both exactly, the hash only picks the bucket.
  // A cached block keeps its content after its last user frees it, until the
  // block is handed out again; then every cached block that continues it (its
  // children, their children, ...) leaves the cache with it, since their K/V
  // were computed after the old content.  A block in use never loses a cached
  // ancestor: whoever holds a block holds the blocks before it.
  // All of it lives in arrays sized up front (the token copies on first use),
  // so registering, finding and dropping entries never allocates.
  std::vector<int32_t> c_parent;  // per block, -2 = not cached
  std::vector<uint64_t> c_hash;
  std::vector<int32_t> c_next, c_prev;    // hash-bucket chain
  std::vector<int32_t> c_kid;             // first cached child
  std::vector<int32_t> c_snext, c_sprev;  // chain of the parent's cached children
  std::vector<int32_t> bucket;            // head of each hash bucket, -1 = empty
  uint64_t bucket_mask = 0;
  std::vector<int32_t> c_tok;  // [num_blocks][block_size] token ids of cached blocks
  int ncached = 0;
  std::vector<int32_t> host_free;  // free host blocks (LIFO), for swapped-out sequences
  int num_host_blocks = 0;
  std::unordered_map<int, Seq> seqs;
  // Scratch of the batch calls: a call number, per block the call that last
  // counted it and how many of that call's sequences append into it.
  uint64_t batch_no = 0;
  std::vector<uint64_t> blk_stamp;
  std::vector<int32_t> blk_count;
  std::vector<Seq *> batch_seqs;
  std::vector<const Seq *> batch_cseqs;

  static uint64_t key_hash(int32_t parent, const int32_t *tok, int n) {
    uint64_t h = 0x9E3779B97F4A7C15ull ^ (uint64_t)(uint32_t)parent;
    for (int i = 0; i < n; ++i) {
      h ^= (uint64_t)(uint32_t)tok[i] + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
      h = (h ^ (h >> 31)) * 0xBF58476D1CE4E5B9ull;
    }
    return h ^ (h >> 29);
  }
  void unlink(int32_t b) {  // b is cached and has no cached children
    const int32_t pv = c_prev[b], nx = c_next[b];
    if (pv >= 0)
      c_next[pv] = nx;
    else
      bucket[c_hash[b] & bucket_mask] = nx;
    if (nx >= 0) c_prev[nx] = pv;
    const int32_t p = c_parent[b];
    if (p >= 0) {
      const int32_t sp = c_sprev[b], sn = c_snext[b];
      if (sp >= 0)
        c_snext[sp] = sn;
      else
        c_kid[p] = sn;
      if (sn >= 0) c_sprev[sn] = sp;
    }
    c_parent[b] = -2;
    --ncached;
    if (where[b] == 2) {  // free, and now nothing to keep: first in line again
      lru_remove(b);
      stack.push_back(b);
      where[b] = 1;
    }
  }
  void lru_remove(int32_t b) {
    const int32_t pv = lru_prev[b], nx = lru_next[b];
    if (pv >= 0)
      lru_next[pv] = nx;
    else
      lru_head = nx;
    if (nx >= 0)
      lru_prev[nx] = pv;
    else
      lru_tail = pv;
    where[b] = 0;
  }
  void lru_push(int32_t b) {  // as the most recently freed
    lru_prev[b] = lru_tail;
    lru_next[b] = -1;
    if (lru_tail >= 0)
      lru_next[lru_tail] = b;
    else
      lru_head = b;
    lru_tail = b;
    where[b] = 2;
  }
  void uncache(int32_t root) {  // root and all its cached descendants, leaves first
    if (c_parent[root] == -2) return;
    int32_t b = root;
    for (;;) {
      while (c_kid[b] >= 0) b = c_kid[b];
      const int32_t p = c_parent[b];
      unlink(b);
      if (b == root) return;
      b = p;
    }
  }
  int32_t take() {  // caller checked nfree > 0
    int32_t b;
    if (!stack.empty()) {
      b = stack.back();
      stack.pop_back();
      where[b] = 0;
    } else {  // evict the least recently freed cached block
      b = lru_head;
      lru_remove(b);
      uncache(b);  // its old content is about to be overwritten
    }
    ref[b] = 1;
    --nfree;
    return b;
  }
  void revive(int32_t b) {  // a prefix-cache hit on b
    if (ref[b]++ == 0) {
      lru_remove(b);
      --nfree;
    }
  }
  void drop(int32_t b) {  // never allocates: the stack has room for every block
    if (--ref[b] == 0) {
      if (c_parent[b] != -2) {
        lru_push(b);
      } else {
        stack.push_back(b);
        where[b] = 1;
      }
      ++nfree;
    }
  }
  bool needs_block(const Seq &s) const {  // appending to s takes a free block
    return s.len % block_size == 0 || ref[s.blocks[s.len / block_size]] > 1;
  }
  void grow(Seq &s) { s.blocks.reserve(std::max<size_t>(8, 2 * s.blocks.size())); }
  // Appending `token` (nullptr: an id not given) to s fills a block that is
  // then registered, so the cache's key store must exist first.
  bool fills_tracked(const Seq &s, const int32_t *token) const {
    return token && s.tracked && (s.len + 1) % block_size == 0;
  }
  void ensure_keys() {  // allocates once
    if (c_tok.empty()) c_tok.assign((size_t)num_blocks * block_size, 0);
  }
  // One token onto s; the caller checked that a block is free if one is
  // needed, that s.blocks has room for a new one and, when the token fills a
  // tracked block, that the key store exists.  Never allocates.
  void append_one(Seq &s, int64_t *slot_out, int64_t *cow_pair_out, const int32_t *token) {
    const int B = block_size;
    const int j = s.len;
    cow_pair_out[0] = cow_pair_out[1] = -1;
    if (j % B == 0) {  // the token opens a new block
      s.blocks.push_back(take());
    } else {
      int32_t &last = s.blocks[j / B];
      if (ref[last] > 1) {  // shared partial block: copy on write
        const int32_t fresh = take();
        cow_pair_out[0] = last;
        cow_pair_out[1] = fresh;
        drop(last);
        last = fresh;
      }
    }
    *slot_out = (int64_t)s.blocks[j / B] * B + (j % B);
    s.len = j + 1;
    if (!token) {  // an id not given: from here on nothing of s is registered
      s.tracked = false;
      s.tail.clear();
      return;
    }
    if (!s.tracked) return;
    s.tail.push_back(*token);  // within the reserved block's room
    if (s.len % B == 0) {      // the token filled its block: findable by later prompts
      const size_t nb = s.blocks.size();
      const int32_t b = s.blocks[nb - 1], parent = nb >= 2 ? s.blocks[nb - 2] : -1;
      // only reachable when the chain before it is cached; its K/V are valid
      // once this step's cache write of the token has run
      if ((parent < 0 || c_parent[parent] != -2) && c_parent[b] == -2) register_block(b, parent, s.tail.data());
      s.tail.clear();
    }
  }
  int32_t lookup(int32_t parent, const int32_t *tok) const {
    if (c_tok.empty()) return -1;
    const uint64_t h = key_hash(parent, tok, block_size);
    for (int32_t b = bucket[h & bucket_mask]; b >= 0; b = c_next[b])
      if (c_hash[b] == h && c_parent[b] == parent && std::equal(tok, tok + block_size, &c_tok[(size_t)b * block_size]))
        return b;
    return -1;
  }
  void register_block(int32_t b, int32_t parent, const int32_t *tok) {  // b not cached; c_tok allocated
    std::copy(tok, tok + block_size, &c_tok[(size_t)b * block_size]);
    const uint64_t h = key_hash(parent, tok, block_size);
    c_hash[b] = h;
    c_parent[b] = parent;
    c_kid[b] = -1;
    int32_t &head = bucket[h & bucket_mask];
    c_prev[b] = -1;
    c_next[b] = head;
    if (head >= 0) c_prev[head] = b;
    head = b;
    if (parent >= 0) {
      c_sprev[b] = -1;
      c_snext[b] = c_kid[parent];
      if (c_kid[parent] >= 0) c_sprev[c_kid[parent]] = b;
      c_kid[parent] = b;
    }
    ++ncached;
  }
};

namespace {

int append_single(pa_bm *bm, int seq_id, const int32_t *token, int64_t *slot_out, int64_t cow_pair_out[2]) {
  if (!bm || !slot_out || !cow_pair_out) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_STATE;
  Seq &s = it->second;
  if (s.len == INT_MAX) return PA_ERR_INVALID;
  if (bm->needs_block(s) && bm->nfree == 0) return PA_ERR_OOM;
  const int st = guarded([&]() -> int {  // allocations first
    if (s.len % bm->block_size == 0 && s.blocks.size() == s.blocks.capacity()) bm->grow(s);
    if (bm->fills_tracked(s, token)) bm->ensure_keys();
    return PA_OK;
  });
  if (st != PA_OK) return st;
  bm->append_one(s, slot_out, cow_pair_out, token);
  return PA_OK;
}

}  // namespace

extern "C" {

pa_bm *pa_bm_create_with_host(int num_blocks, int num_host_blocks, int block_size) {
  if (num_blocks <= 0 || num_host_blocks < 0 || block_size <= 0) return nullptr;
  pa_bm *bm = new (std::nothrow) pa_bm();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign(num_blocks, 0);
    bm->stack.reserve(num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) bm->stack.push_back(b);
    bm->nfree = num_blocks;
    bm->where.assign(num_blocks, 1);
    bm->lru_prev.assign(num_blocks, -1);
    bm->lru_next.assign(num_blocks, -1);
    bm->c_parent.assign(num_blocks, -2);
    bm->c_hash.assign(num_blocks, 0);
    bm->c_next.assign(num_blocks, -1);
    bm->c_prev.assign(num_blocks, -1);
    bm->c_kid.assign(num_blocks, -1);
    bm->c_snext.assign(num_blocks, -1);
    bm->c_sprev.assign(num_blocks, -1);
    size_t nb = 1;
    while (nb < (size_t)num_blocks) nb <<= 1;
    bm->bucket.assign(nb, -1);
    bm->bucket_mask = nb - 1;
    bm->blk_stamp.assign(num_blocks, 0);
    bm->blk_count.assign(num_blocks, 0);
    bm->num_host_blocks = num_host_blocks;
    bm->host_free.reserve(num_host_blocks);
    for (int b = num_host_blocks - 1; b >= 0; --b) bm->host_free.push_back(b);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

pa_bm *pa_bm_create(int num_blocks, int block_size) { return pa_bm_create_with_host(num_blocks, 0, block_size); }

void pa_bm_destroy(pa_bm *bm) { delete bm; }

int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens) {
  if (!bm || seq_id < 0 || num_tokens < 0) return PA_ERR_INVALID;
  return guarded([&]() -> int {
    if (bm->seqs.count(seq_id)) return PA_ERR_STATE;
    const int64_t need = ((int64_t)num_tokens + bm->block_size - 1) / bm->block_size;
    if (need > (int64_t)bm->nfree) return PA_ERR_OOM;
    Seq s;
    s.len = num_tokens;
    s.blocks.reserve(need);
    // the last allocation; the blocks then go into the reserved room
    Seq &q = bm->seqs.emplace(seq_id, std::move(s)).first->second;
    for (int64_t i = 0; i < need; ++i) q.blocks.push_back(bm->take());
    return PA_OK;
  });
}

int pa_bm_fork(pa_bm *bm, int parent_id, int child_id) {
  if (!bm || child_id < 0) return PA_ERR_INVALID;
  return guarded([&]() -> int {
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end() || bm->seqs.count(child_id) || it->second.swapped) return PA_ERR_STATE;
    auto c = bm->seqs.emplace(child_id, it->second).first;  // copies
    if (c->second.tracked) {
      try {
        c->second.tail.reserve(bm->block_size);  // a copy keeps only the ids' own room
      } catch (...) {
        bm->seqs.erase(c);
        throw;
      }
    }
    for (int32_t b : c->second.blocks) ++bm->ref[b];  // no allocation from here
    return PA_OK;
  });
}

int pa_bm_append(pa_bm *bm, int seq_id, int64_t *slot_out, int64_t cow_pair_out[2]) {
  return append_single(bm, seq_id, nullptr, slot_out, cow_pair_out);
}

int pa_bm_append_token(pa_bm *bm, int seq_id, int32_t token, int64_t *slot_out, int64_t cow_pair_out[2]) {
  return append_single(bm, seq_id, &token, slot_out, cow_pair_out);
}

int pa_bm_append_batch(pa_bm *bm, const int32_t *seq_ids, const int32_t *tokens, int n, int64_t *slots_out,
                       int64_t *cow_pairs_out) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out))) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  return guarded([&]() -> int {
    // every check and allocation first: a failure leaves no trace
    bm->batch_seqs.resize(n);
    Seq **sq = bm->batch_seqs.data();
    const uint64_t call = ++bm->batch_no;
    const int B = bm->block_size;
    for (int i = 0; i < n; ++i) {
      auto it = bm->seqs.find(seq_ids[i]);
      if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_STATE;
      Seq &s = it->second;
      if (s.stamp == call || s.len == INT_MAX) return PA_ERR_INVALID;  // listed twice
      s.stamp = call;
      sq[i] = &s;
    }
    // k of the batch appending into a partial block of ref_count r copy it
    // min(k, r - 1) times: after r - 1 copies the last holder owns it alone
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
      const Seq &s = *sq[i];
      if (s.len % B == 0) {
        ++need;
        continue;
      }
      const int32_t x = s.blocks[s.len / B];
      if (bm->ref[x] < 2) continue;
      if (bm->blk_stamp[x] != call) {
        bm->blk_stamp[x] = call;
        bm->blk_count[x] = 0;
      }
      if (bm->blk_count[x]++ < bm->ref[x] - 1) ++need;
    }
    if (need > (int64_t)bm->nfree) return PA_ERR_OOM;
    for (int i = 0; i < n; ++i) {
      if (sq[i]->len % B == 0 && sq[i]->blocks.size() == sq[i]->blocks.capacity()) bm->grow(*sq[i]);
      if (bm->fills_tracked(*sq[i], tokens ? tokens + i : nullptr)) bm->ensure_keys();
    }
    for (int i = 0; i < n; ++i) bm->append_one(*sq[i], slots_out + i, cow_pairs_out + 2 * i, tokens ? tokens + i : nullptr);
    return PA_OK;
  });
}

int pa_bm_free_seq(pa_bm *bm, int seq_id) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_STATE;
  if (it->second.swapped) {  // its blocks live on the host
    const auto &hb = it->second.blocks;
    for (auto r = hb.rbegin(); r != hb.rend(); ++r) bm->host_free.push_back(*r);
    bm->seqs.erase(it);
    return PA_OK;
  }
  for (int32_t b : it->second.blocks) {
    if (bm->ref[b] <= 0) return PA_ERR_STATE;  // cannot happen unless corrupted
  }
  // Last to first: an uncached first block is handed out again first, and a
  // cached block stays longer than the blocks that continue it.
  const auto &bl = it->second.blocks;
  for (auto r = bl.rbegin(); r != bl.rend(); ++r) bm->drop(*r);
  bm->seqs.erase(it);
  return PA_OK;
}

int pa_bm_block_table(const pa_bm *bm, int seq_id, int32_t *out, int cap, int *n) {
  if (!bm || !n) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_STATE;
  const auto &bl = it->second.blocks;
  *n = (int)bl.size();
  if (cap < *n || (!out && *n > 0)) return PA_ERR_INVALID;
  std::copy(bl.begin(), bl.end(), out);
  return PA_OK;
}

int pa_bm_block_tables(const pa_bm *bm, const int32_t *seq_ids, int n, int32_t *out, int max_blocks, int32_t pad,
                       int32_t *context_lens_out) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || (!out && max_blocks > 0)))) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  pa_bm *m = const_cast<pa_bm *>(bm);  // only the scratch list of sequences changes
  return guarded([&]() -> int {
    m->batch_cseqs.resize(n);
    const Seq **sq = m->batch_cseqs.data();
    for (int i = 0; i < n; ++i) {  // check every id first: nothing is written on error
      auto it = bm->seqs.find(seq_ids[i]);
      if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_STATE;
      if ((int64_t)it->second.blocks.size() > max_blocks) return PA_ERR_INVALID;
      sq[i] = &it->second;
    }
    for (int i = 0; i < n; ++i) {
      int32_t *row = out + (size_t)i * max_blocks;
      std::copy(sq[i]->blocks.begin(), sq[i]->blocks.end(), row);
      std::fill(row + sq[i]->blocks.size(), row + max_blocks, pad);
      if (context_lens_out) context_lens_out[i] = sq[i]->len;
    }
    return PA_OK;
  });
}

int pa_bm_seq_len(const pa_bm *bm, int seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

int pa_bm_ref_count(const pa_bm *bm, int block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

int pa_bm_num_free(const pa_bm *bm) { return bm ? bm->nfree : -1; }

int pa_bm_add_seq_tokens(pa_bm *bm, int seq_id, const int32_t *tokens, int num_tokens, int *cached_tokens) {
  if (!bm || seq_id < 0 || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_ERR_INVALID;
  return guarded([&]() -> int {
    if (bm->seqs.count(seq_id)) return PA_ERR_STATE;
    const int B = bm->block_size;
    const int64_t nfull = num_tokens / B;
    const int64_t need = ((int64_t)num_tokens + B - 1) / B;
    // longest chain of cached full blocks from the start
    std::vector<int32_t> hit;
    int32_t parent = -1;
    for (int64_t i = 0; i < nfull; ++i) {
      const int32_t b = bm->lookup(parent, tokens + (size_t)i * B);
      if (b < 0) break;
      hit.push_back(b);
      parent = b;
    }
    int64_t revive = 0;  // hits that sit in the free pool
    for (int32_t b : hit) revive += bm->ref[b] == 0;
    if (need - (int64_t)hit.size() > (int64_t)bm->nfree - revive) return PA_ERR_OOM;
    Seq s;
    s.len = num_tokens;
    s.blocks.reserve(need);
    s.tracked = true;
    s.tail.reserve(B);
    s.tail.assign(tokens + (size_t)nfull * B, tokens + num_tokens);
    // the last allocations; nothing below allocates
    if (nfull > (int64_t)hit.size()) bm->ensure_keys();
    Seq &q = bm->seqs.emplace(seq_id, std::move(s)).first->second;
    for (int32_t b : hit) {
      bm->revive(b);
      q.blocks.push_back(b);
    }
    parent = hit.empty() ? -1 : hit.back();
    for (int64_t i = (int64_t)hit.size(); i < need; ++i) {
      const int32_t b = bm->take();
      q.blocks.push_back(b);
      if (i < nfull) {  // a full block of the prompt: findable by later prompts
        bm->register_block(b, parent, tokens + (size_t)i * B);
        parent = b;
      }
    }
    if (cached_tokens) *cached_tokens = (int)hit.size() * B;
    return PA_OK;
  });
}

int pa_bm_num_cached_blocks(const pa_bm *bm) { return bm ? bm->ncached : -1; }

int pa_bm_swap_out(pa_bm *bm, int seq_id, int64_t *pairs_out, int cap, int *n) {
  if (!bm || !n) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_STATE;
  Seq &s = it->second;
  *n = (int)s.blocks.size();
  if (cap < *n || (!pairs_out && *n > 0)) return PA_ERR_INVALID;
  for (int32_t b : s.blocks)
    if (bm->ref[b] != 1) return PA_ERR_STATE;  // shared blocks stay with their other users
  if ((int)bm->host_free.size() < *n) return PA_ERR_OOM;
  for (int i = 0; i < *n; ++i) {
    const int32_t h = bm->host_free.back();
    bm->host_free.pop_back();
    pairs_out[2 * i] = s.blocks[i];
    pairs_out[2 * i + 1] = h;
    s.blocks[i] = h;
  }
  // freed last to first, as by pa_bm_free_seq: a cached block then stays
  // longer than the blocks that continue it
  for (int i = *n - 1; i >= 0; --i) bm->drop((int32_t)pairs_out[2 * i]);
  s.swapped = true;
  return PA_OK;
}

int pa_bm_swap_in(pa_bm *bm, int seq_id, int64_t *pairs_out, int cap, int *n) {
  if (!bm || !n) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || !it->second.swapped) return PA_ERR_STATE;
  Seq &s = it->second;
  *n = (int)s.blocks.size();
  if (cap < *n || (!pairs_out && *n > 0)) return PA_ERR_INVALID;
  if (bm->nfree < *n) return PA_ERR_OOM;
  for (int i = 0; i < *n; ++i) {
    const int32_t h = s.blocks[i];
    const int32_t d = bm->take();
    pairs_out[2 * i] = h;
    pairs_out[2 * i + 1] = d;
    bm->host_free.push_back(h);
    s.blocks[i] = d;
  }
  s.swapped = false;
  return PA_OK;
}

int pa_bm_num_free_host(const pa_bm *bm) { return bm ? (int)bm->host_free.size() : -1; }

}  // extern "C"

namespace {

int64_t wasted_slots(const pa_bm *bm) {
  // Only a sequence's last block can be partly filled.  A block shared by
  // several sequences is counted once, with the largest fill among them.
  std::unordered_map<int32_t, int> fill;
  for (const auto &kv : bm->seqs) {
    const Seq &s = kv.second;
    if (s.blocks.empty() || s.swapped) continue;
    int f = s.len - (int)(s.blocks.size() - 1) * bm->block_size;
    auto it = fill.find(s.blocks.back());
    if (it == fill.end())
      fill.emplace(s.blocks.back(), f);
    else
      it->second = std::max(it->second, f);
  }
  int64_t w = 0;
  for (const auto &kv : fill) w += bm->block_size - kv.second;
  return w;
}

}  // namespace

extern "C" {

int64_t pa_bm_wasted_slots(const pa_bm *bm) {
  if (!bm) return -1;
  try {
    return wasted_slots(bm);
  } catch (...) {
    return -1;
  }
}

}  // extern "C"
