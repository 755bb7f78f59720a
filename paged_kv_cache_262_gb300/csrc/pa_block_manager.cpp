// Host block manager: free list, per-sequence block tables, reference counts,
// fork / copy-on-write / free.  Plain C++17, no GPU.
//
// Follows "vLLM High-Performance Inference Engine: PagedAttention Principles
// and Deployment Guide" ("PagedAttention Architecture Deep Dive": block table
// with ref_count, pages shared between sequences), "vLLM Guide: High-Throughput
// Multi-GPU LLM Serving with PagedAttention" ("What Is PagedAttention?": blocks
// allocated on demand, shared prefixes with copy-on-write) and "Configuring
// vLLM and PagedAttention for High Throughput Enterprise LLM Serving"
// ("High-Throughput Batching": pages go back to the free pool on <eos>).
#include <algorithm>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pagedattn.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;
  int len = 0;
};

}  // namespace

struct pa_bm {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ref;        // per block, 0 = free
  std::vector<int32_t> free_list;  // LIFO stack; back() is handed out next
  std::unordered_map<int, Seq> seqs;

  int32_t take() {
    int32_t b = free_list.back();
    free_list.pop_back();
    ref[b] = 1;
    return b;
  }
  void drop(int32_t b) {
    if (--ref[b] == 0) free_list.push_back(b);
  }
};

extern "C" {

pa_bm *pa_bm_create(int num_blocks, int block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_bm *bm = new (std::nothrow) pa_bm();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->free_list.reserve(num_blocks);
  for (int b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(b);
  return bm;
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens) {
  if (!bm || seq_id < 0 || num_tokens < 0) return PA_ERR_INVALID;
  if (bm->seqs.count(seq_id)) return PA_ERR_STATE;
  const int64_t need = ((int64_t)num_tokens + bm->block_size - 1) / bm->block_size;
  if (need > (int64_t)bm->free_list.size()) return PA_ERR_OOM;
  Seq s;
  s.len = num_tokens;
  s.blocks.reserve(need);
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  bm->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

int pa_bm_fork(pa_bm *bm, int parent_id, int child_id) {
  if (!bm || child_id < 0) return PA_ERR_INVALID;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end() || bm->seqs.count(child_id)) return PA_ERR_STATE;
  Seq c = it->second;
  for (int32_t b : c.blocks) ++bm->ref[b];
  bm->seqs.emplace(child_id, std::move(c));
  return PA_OK;
}

int pa_bm_append(pa_bm *bm, int seq_id, int64_t *slot_out, int64_t cow_pair_out[2]) {
  if (!bm || !slot_out || !cow_pair_out) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_STATE;
  Seq &s = it->second;
  const int B = bm->block_size;
  const int j = s.len;
  cow_pair_out[0] = cow_pair_out[1] = -1;
  if (j % B == 0) {  // the token opens a new block
    if (bm->free_list.empty()) return PA_ERR_OOM;
    s.blocks.push_back(bm->take());
  } else {
    int32_t &last = s.blocks[j / B];
    if (bm->ref[last] > 1) {  // shared partial block: copy on write
      if (bm->free_list.empty()) return PA_ERR_OOM;
      int32_t fresh = bm->take();
      cow_pair_out[0] = last;
      cow_pair_out[1] = fresh;
      bm->drop(last);
      last = fresh;
    }
  }
  *slot_out = (int64_t)s.blocks[j / B] * B + (j % B);
  s.len = j + 1;
  return PA_OK;
}

int pa_bm_free_seq(pa_bm *bm, int seq_id) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_STATE;
  for (int32_t b : it->second.blocks) {
    if (bm->ref[b] <= 0) return PA_ERR_STATE;  // cannot happen unless corrupted
  }
  // Return blocks last-to-first so the sequence's first block is reused first.
  const auto &bl = it->second.blocks;
  for (auto r = bl.rbegin(); r != bl.rend(); ++r) bm->drop(*r);
  bm->seqs.erase(it);
  return PA_OK;
}

int pa_bm_block_table(const pa_bm *bm, int seq_id, int32_t *out, int cap, int *n) {
  if (!bm || !n) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_STATE;
  const auto &bl = it->second.blocks;
  *n = (int)bl.size();
  if (cap < *n || (!out && *n > 0)) return PA_ERR_INVALID;
  std::copy(bl.begin(), bl.end(), out);
  return PA_OK;
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

int pa_bm_num_free(const pa_bm *bm) { return bm ? (int)bm->free_list.size() : -1; }

int64_t pa_bm_wasted_slots(const pa_bm *bm) {
  if (!bm) return -1;
  // Only a sequence's last block can be partly filled.  A block shared by
  // several sequences is counted once, with the largest fill among them.
  std::unordered_map<int32_t, int> fill;
  for (const auto &kv : bm->seqs) {
    const Seq &s = kv.second;
    if (s.blocks.empty()) continue;
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

}  // extern "C"
