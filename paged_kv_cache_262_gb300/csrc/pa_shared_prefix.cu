// Shared-prefix-aware decode.
//
// "Configuring vLLM and PagedAttention for High Throughput Enterprise LLM
// Serving" ("Zero-Copy Prefix Caching & Shared Sampling") has requests that
// share a prompt prefix point at the same physical pages, and decode is bound
// by reading the cache from HBM ("Memory Bottlenecks in Autoregressive LLM
// Inference").  Plain decode reads a shared prefix once per sharer.  Here a
// group of sequences that share their first P tokens has that prefix attended
// once, for all of the group's query rows together (sequences x query heads),
// as a dense contraction on the tensor cores; each sequence's decode then
// covers only its own keys P .. ctx-1 and merges the prefix's partial softmax
// states (m, l, o/l) exactly as split-K parts are merged.  When the groups
// alone would not fill the GPU, the prefix is cut into up to 8 key ranges of
// whole 128-key tiles, each attended by its own CTAs into its own state.
// A second level (pa_paged_attention_decode_shared_prefix2): sub-groups of
// consecutive sequences that share more leading blocks -- the samples of one
// prompt -- are decoded as one unit per (sub-group, kv head), reading those
// blocks once for all members (the sub-group mode of the decode unit).
#include <cuda_runtime.h>
#include <stdlib.h>

#include <algorithm>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

struct Layout {
  size_t decode, pre_o, pre_ml, tasks;
  size_t total() const { return decode + pre_o + pre_ml + tasks; }
};

Layout layout(const pa_decode_desc *d) {
  Layout l;
  l.decode = up256(pa::make_decode_plan(d, pa::current_sm_count()).total());
  l.pre_o = up256((size_t)pa::kMaxPrefixParts * d->num_seqs * d->num_q_heads * d->head_dim * sizeof(float));
  l.pre_ml = up256((size_t)pa::kMaxPrefixParts * d->num_seqs * d->num_q_heads * 2 * sizeof(float));
  l.tasks = d->head_dim == 128 ? up256(pa::task_workspace_bytes(d)) : 0;
  return l;
}

// The second launch as a task queue (pa_decode_tasks.cu) for sub-groups
// behind a group prefix: what is left past the prefix is short (a prompt's
// own blocks and each sample's copy-on-write block), where one CTA per unit
// spends most of its life starting and finishing (prefix sharing, 64 prompts
// x 4 samples: 55.6 us one level, 59.6 us sub-groups, 42-43 us as tasks).
// Long units stay with the one-CTA-per-unit decode (parallel sampling: 124
// us against 137-142 as tasks; one level with groups: 55.6 against 68-70).
// PA_DECODE_TASKS=0 / 1 in the environment forces the choice (comparison).
bool use_tasks(const pa_decode_desc *d, int nsg, int rows, bool subgroups_behind_prefix) {
  const char *env = getenv("PA_DECODE_TASKS");
  if (env && env[0] == '0') return false;
  if (!(env && env[0] == '1') && !subgroups_behind_prefix) return false;
  return pa::tasks_supported(d, nsg, rows);
}

// The second launch on the tensor cores (pa_decode_wide.cu), taken only with
// PA_DECODE_WIDE=1 in the environment: on these units it is slower than the
// warp-MMA kernels (parallel sampling 160 us against 123 us one CTA per unit;
// prefix sharing 84 us against 43.6 us as tasks) -- each 128-token tile
// passes through a chain of S MMA, TMEM load, a four-warp maxima exchange,
// P^T through shared memory behind a proxy fence, the P V MMA and a TMEM
// fold, and three 64 KB tiles in flight per SM do not cover that chain.
bool use_wide(const pa_decode_desc *d, int nsg, int rows) {
  const char *env = getenv("PA_DECODE_WIDE");
  if (!(env && env[0] == '1')) return false;
  return pa::wide_supported(d, nsg, rows);
}

}  // namespace

extern "C" size_t pa_shared_prefix_workspace_bytes(const pa_decode_desc *desc) {
  if (pa::validate_decode_desc(desc) != PA_OK) return 0;
  return layout(desc).total();
}

namespace {

// Both entry points: groups (one level), and optionally sub-groups (a second).
int shared_prefix(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_tables, const int32_t *context_lens, int num_groups,
                  const int32_t *group_starts, const int32_t *group_prefix_lens, const int32_t *prefix_tables,
                  int prefix_max_blocks, int max_group_size, int max_prefix_len, int num_subgroups,
                  const int32_t *subgroup_starts, const int32_t *subgroup_shared_lens, int max_subgroup_size,
                  void *out, void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream) {
  using namespace pa;
  int st = validate_decode_desc(d);
  if (st != PA_OK) return st;
  if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0 || prefix_max_blocks < 0 || num_subgroups < 0 ||
      max_subgroup_size < 0)
    return PA_ERR_INVALID;
  if (d->num_seqs == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !out || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(out))
    return PA_ERR_INVALID;
  const int G = d->num_q_heads / d->num_kv_heads;
  DecodePrefix sub{};  // the sub-group partition (the prefix states are filled in below)
  if (num_subgroups > 0) {
    if (!subgroup_starts || !subgroup_shared_lens || max_subgroup_size == 0) return PA_ERR_INVALID;
    if (d->head_dim != 128 || (long long)max_subgroup_size * G > 16) return PA_ERR_UNSUPPORTED;
    if (num_subgroups > 65535) return PA_ERR_UNSUPPORTED;
    sub.sub_start = subgroup_starts;
    sub.sub_shared = subgroup_shared_lens;
    sub.nsub = num_subgroups;
    sub.sub_rows = max_subgroup_size * G;
  }
  if (num_groups == 0) {
    if (num_subgroups > 0 && use_wide(d, num_subgroups, sub.sub_rows)) {
      const Layout l = layout(d);
      if (!workspace || workspace_bytes < l.total() || !aligned16(workspace)) return PA_ERR_WORKSPACE;
      uint8_t *tws = static_cast<uint8_t *>(workspace) + l.decode + l.pre_o + l.pre_ml;
      st = decode_tasks_clear(d, tws, stream);
      if (st != PA_OK) return st;
      return decode_wide_launch(d, q, k_pool, v_pool, block_tables, context_lens, sub, sub.sub_rows, out,
                                task_counter(d, tws), err_flag, stream);
    }
    if (num_subgroups > 0 && use_tasks(d, num_subgroups, sub.sub_rows, false)) {
      const Layout l = layout(d);
      if (!workspace || workspace_bytes < l.total() || !aligned16(workspace)) return PA_ERR_WORKSPACE;
      uint8_t *tws = static_cast<uint8_t *>(workspace) + l.decode + l.pre_o + l.pre_ml;
      st = decode_tasks_clear(d, tws, stream);
      if (st != PA_OK) return st;
      return decode_tasks_launch(d, q, k_pool, v_pool, block_tables, context_lens, sub, sub.sub_rows, out, tws,
                                 err_flag, stream);
    }
    return decode_launch(d, q, k_pool, v_pool, block_tables, context_lens, out, workspace, workspace_bytes, err_flag,
                         stream, num_subgroups > 0 ? &sub : nullptr);
  }
  if (!group_starts || !group_prefix_lens || !prefix_tables || prefix_max_blocks == 0 || max_group_size == 0 ||
      max_prefix_len == 0)
    return PA_ERR_INVALID;
  if (max_prefix_len > d->max_context_len || (int64_t)prefix_max_blocks * d->block_size < max_prefix_len)
    return PA_ERR_INVALID;
  const Layout l = layout(d);
  if (!workspace || workspace_bytes < l.total() || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *pre_o = reinterpret_cast<float *>(ws + l.decode);
  float *pre_ml = reinterpret_cast<float *>(ws + l.decode + l.pre_o);
  const int nsg = num_subgroups > 0 ? num_subgroups : d->num_seqs;
  const int rows = num_subgroups > 0 ? sub.sub_rows : G;
  const bool wide = use_wide(d, nsg, rows);
  const bool tasks = !wide && use_tasks(d, nsg, rows, num_subgroups > 0);
  // 1. each group's shared prefix, all of its rows at once, on the tensor cores,
  //    cut into key ranges so that the pass has about one CTA per SM -- or,
  //    beside the task decode (which streams on the SMs the pass leaves free;
  //    only its merge waits for the pass), about 7/16 of the SMs (prefix
  //    sharing, 64 prompts x 4 samples: a 48.2 us step with 2 key ranges, 49.4
  //    with 4, 50.1 with 1)
  const long long base = (long long)num_groups * d->num_kv_heads * (((long long)max_group_size * G + 255) / 256);
  const int sms = std::max(current_sm_count(), 1);
  int kparts = (int)std::min<long long>(kMaxPrefixParts, std::max<long long>(1, (sms + base - 1) / base));
  if (tasks) {
    const long long want = (long long)sms * 7 / 16;
    kparts = (int)std::min<long long>(kMaxPrefixParts, std::max<long long>(1, (want + base / 2) / base));
  }
  if (const char *env = getenv("PA_PREFIX_PARTS"))  // comparison: a fixed number of key ranges
    kparts = std::max(1, std::min(kMaxPrefixParts, atoi(env)));
  kparts = std::min(kparts, (max_prefix_len + 127) / 128);
  const int kpart_len = ((max_prefix_len + kparts - 1) / kparts + 127) / 128 * 128;
  kparts = (max_prefix_len + kpart_len - 1) / kpart_len;
  if (tasks || wide) {  // before the prefix pass: the second grid may start beside it
    st = decode_tasks_clear(d, ws + l.decode + l.pre_o + l.pre_ml, stream);
    if (st != PA_OK) return st;
  }
  pa_decode_desc pd = *d;
  pd.num_seqs = num_groups;
  pd.max_blocks_per_seq = prefix_max_blocks;
  pd.max_context_len = max_prefix_len;
  st = prefill_launch(&pd, q, group_starts, max_group_size, d->num_seqs, k_pool, v_pool, prefix_tables,
                      group_prefix_lens, nullptr, pre_o, pre_ml, /*causal=*/0, kparts, kparts > 1 ? kpart_len : 0,
                      err_flag, stream);
  if (st != PA_OK) return st;
  // 2. every sequence's own keys (or every sub-group's), merged with its group's prefix states
  DecodePrefix pre = sub;
  pre.grp_start = group_starts;
  pre.grp_prefix = group_prefix_lens;
  pre.ngroups = num_groups;
  pre.pre_o = pre_o;
  pre.pre_ml = pre_ml;
  pre.npre = kparts;
  if (wide)
    return decode_wide_launch(d, q, k_pool, v_pool, block_tables, context_lens, pre, rows, out,
                              task_counter(d, ws + l.decode + l.pre_o + l.pre_ml), err_flag, stream);
  if (tasks)
    return decode_tasks_launch(d, q, k_pool, v_pool, block_tables, context_lens, pre, rows, out,
                               ws + l.decode + l.pre_o + l.pre_ml, err_flag, stream);
  return decode_launch(d, q, k_pool, v_pool, block_tables, context_lens, out, ws, l.decode, err_flag, stream, &pre);
}

}  // namespace

extern "C" int pa_paged_attention_decode_shared_prefix(
    const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool, const int32_t *block_tables,
    const int32_t *context_lens, int num_groups, const int32_t *group_starts, const int32_t *group_prefix_lens,
    const int32_t *prefix_tables, int prefix_max_blocks, int max_group_size, int max_prefix_len, void *out,
    void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream) {
  return shared_prefix(d, q, k_pool, v_pool, block_tables, context_lens, num_groups, group_starts, group_prefix_lens,
                       prefix_tables, prefix_max_blocks, max_group_size, max_prefix_len, 0, nullptr, nullptr, 0, out,
                       workspace, workspace_bytes, err_flag, stream);
}

extern "C" int pa_paged_attention_decode_shared_prefix2(
    const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool, const int32_t *block_tables,
    const int32_t *context_lens, int num_groups, const int32_t *group_starts, const int32_t *group_prefix_lens,
    const int32_t *prefix_tables, int prefix_max_blocks, int max_group_size, int max_prefix_len, int num_subgroups,
    const int32_t *subgroup_starts, const int32_t *subgroup_shared_lens, int max_subgroup_size, void *out,
    void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream) {
  return shared_prefix(d, q, k_pool, v_pool, block_tables, context_lens, num_groups, group_starts, group_prefix_lens,
                       prefix_tables, prefix_max_blocks, max_group_size, max_prefix_len, num_subgroups,
                       subgroup_starts, subgroup_shared_lens, max_subgroup_size, out, workspace, workspace_bytes,
                       err_flag, stream);
}
