// Host-side helpers shared by the launchers of libpagedattn (not part of the
// public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// SM count of the current device (cached per device); <= 0 on error.
int current_sm_count();

// Encodes a 2-D bf16 tensor map over `rows` x `cols` elements (row pitch
// cols*2 bytes) with a box of box_rows x box_cols and 128-byte swizzling.
// Returns false when the driver encoder is unavailable or rejects the map.
bool encode_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, uint32_t box_cols, bool swizzle128);
// K or V pool rows of 128 bf16 as (64 columns, row, half): one box of
// box_rows rows and both 64-column halves lands as the two halves one after
// the other, each box_rows x 128 bytes, 128-byte swizzled -- the layout two
// 64-column 2-D boxes give, in one copy.
bool encode_kv_halves_3d(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// Longest context part one decode CTA streams, and most parts per sequence.
constexpr int kMaxPartPages = 512;
constexpr int kMaxParts = 256;

// Split-K plan of a decode call: every sequence's pages are cut into parts of
// part_pages pages; max_parts parts at most per sequence.
struct DecodePlan {
  int part_pages = 0;
  int max_parts = 0;
  size_t ws_o_bytes = 0;    // fp32 [S][Hkv][max_parts][G][D]
  size_t ws_ml_bytes = 0;   // fp32 [S][Hkv][max_parts][G][2]
  size_t ws_cnt_bytes = 0;  // uint64 [S][Hkv] epoch-tagged arrival counters
  size_t total() const { return ws_o_bytes + ws_ml_bytes + ws_cnt_bytes; }
};

// Validates `d` for the decode kernel; PA_OK or an error status.
int validate_decode_desc(const pa_decode_desc *d);

// The plan used by both pa_decode_workspace_bytes and the launcher.
DecodePlan make_decode_plan(const pa_decode_desc *d, int sm_count);

// A new tag for the split-K arrival counters of one decode launch: unique
// (never 0) across every launcher that may share a workspace.
unsigned int next_decode_epoch();

// Shared-prefix information for the decode kernel (see pa_shared_prefix.cu).
struct DecodePrefix {
  const int32_t *grp_start;   // device [ngroups + 1]
  const int32_t *grp_prefix;  // device [ngroups], tokens, multiples of B
  int ngroups;
  const float *pre_o;         // device [npre][S][Hq][D]
  const float *pre_ml;        // device [npre][S][Hq][2]
  int npre;                   // partial states per row (key ranges of the prefix)
  // Sub-groups (optional, nsub > 0): sequences sub_start[k] .. sub_start[k+1]-1
  // share keys 0 .. sub_shared[k]-1; one decode unit per (sub-group, kv head)
  // covering at most sub_rows query rows (member x head).
  const int32_t *sub_start;   // device [nsub + 1], a partition of 0 .. S-1
  const int32_t *sub_shared;  // device [nsub], tokens, multiples of B
  int nsub;
  int sub_rows;
};

// The newest token of every sequence, appended by the decode launch itself
// (pa_paged_attention_decode_append).
struct DecodeAppend {
  const void *new_k;     // device bf16 [S][Hkv][D]
  const void *new_v;     // device bf16 [S][Hkv][D]
  const int64_t *slots;  // device [S], the slot of position ctx-1 or < 0
};

// The decode launcher behind pa_paged_attention_decode (pre and app may be
// null; not both set).
int decode_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_tables, const int32_t *context_lens, void *out, void *workspace,
                  size_t workspace_bytes, int32_t *err_flag, void *stream, const DecodePrefix *pre,
                  const DecodeAppend *app = nullptr);

// Launches the chunked-prefill kernel (pa_prefill.cu).  causal = 0 lets every
// row see all ctx keys; with part_o/part_ml set, rows are written as fp32
// partial softmax states (o/l, m, l) instead of bf16 outputs, one state per
// key range when kparts > 1 (ranges of kpart_len keys, a multiple of 128).
int prefill_launch(const pa_decode_desc *d, const void *q, const int32_t *cu_q, int max_q_len, int total_q,
                   const void *k_pool, const void *v_pool, const int32_t *block_tables, const int32_t *context_lens,
                   void *out, float *part_o, float *part_ml, int causal, int kparts, int kpart_len,
                   int32_t *err_flag, void *stream);

// Most key ranges the shared-prefix pass splits a prefix into.
constexpr int kMaxPrefixParts = 8;

// Task decode (pa_decode_tasks.cu): parts a unit's pages are cut into at
// most, and sub-groups (or sequences) one launch takes at most.
constexpr int kTaskMaxParts = 16;
constexpr int kTaskMaxSub = 512;

// Workspace of the task decode: per-part partial states of every query row,
// arrival counters, the task counters.
size_t task_workspace_bytes(const pa_decode_desc *d);

// Whether the task decode takes this call: head_dim 128, 1 .. kTaskMaxSub
// sub-groups (at most num_seqs), at most 16 query rows a unit.
bool tasks_supported(const pa_decode_desc *d, int nsg, int rows);

// Zeroes the task decode's counters in its workspace (stream-ordered); must
// precede decode_tasks_launch on the stream.
int decode_tasks_clear(const pa_decode_desc *d, void *workspace, void *stream);

// The task decode's counter word in its workspace (zeroed by
// decode_tasks_clear); the wide-group decode takes its units from it.
unsigned int *task_counter(const pa_decode_desc *d, void *workspace);

// Whether the wide-group decode (pa_decode_wide.cu) takes this call: head_dim
// 128, 1 .. kTaskMaxSub units' sub-groups (at most num_seqs), at most 16 query
// rows a unit.
bool wide_supported(const pa_decode_desc *d, int nsg, int rows);

// The shared-prefix decode's second launch on the tensor cores: every
// (sub-group, kv head) -- or (sequence, kv head) when pre.nsub == 0 -- with
// its rows (at most 16) as the MMA N side and 128-token key tiles as M, the
// group prefix's partial states folded in.  counter: a zeroed word
// (task_counter after decode_tasks_clear).  Launched as a programmatic
// dependent of the kernel before it (it waits for that kernel before reading
// pre's states).
int decode_wide_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                       const int32_t *block_tables, const int32_t *context_lens, const DecodePrefix &pre, int rows,
                       void *out, unsigned int *counter, int32_t *err_flag, void *stream);

// The shared-prefix decode's second launch as a queue of small tasks: every
// (sub-group, kv head) -- or (sequence, kv head) when pre.nsub == 0 -- with
// the group prefix's partial states (pre) folded in.  rows bounds a unit's
// query rows (members x heads).  workspace: task_workspace_bytes(d), cleared
// by decode_tasks_clear.  Launched as a programmatic dependent of the kernel
// before it (it reads nothing that kernel writes) and followed by a merge
// launch that reads pre's states.
int decode_tasks_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                        const int32_t *block_tables, const int32_t *context_lens, const DecodePrefix &pre, int rows,
                        void *out, void *workspace, int32_t *err_flag, void *stream);

}  // namespace pa
