/*
 * pagedattn.h -- C ABI of libpagedattn, the paged KV-cache attention hot path
 * for NVIDIA GB300 (sm_103a).
 *
 * The operations follow three web pages on vLLM / PagedAttention:
 *  [ATT]  "Configuring vLLM and PagedAttention for High Throughput Enterprise
 *         LLM Serving", section "Architectural Foundations: PagedAttention &
 *         Virtual Memory": KV cache split into blocks of B tokens drawn from a
 *         global physical page pool; a block table maps logical blocks to
 *         physical pages; attention weights
 *         A_ij = exp(q_i.k_j/sqrt(d)) / sum_m exp(q_i.k_m/sqrt(d)); the kernel
 *         fetches k_j from page BlockTable[j / B].
 *  [PHASE] same page, "Memory Bottlenecks in Autoregressive LLM Inference":
 *         prefill writes K/V for every position; decode reads the whole cache
 *         from HBM for each new token (bandwidth bound).
 *  [CHUNK] same page, "High-Throughput Batching: Continuous Batching & Chunked
 *         Prefill": prompts split into 512/1024-token chunks that ride along
 *         with decode iterations; pages returned to the free pool on <eos>.
 *  [SHARE] same page, "Zero-Copy Prefix Caching & Shared Sampling", and
 *         "vLLM Guide: High-Throughput Multi-GPU LLM Serving with
 *         PagedAttention", section "What Is PagedAttention?": blocks allocated
 *         on demand; shared prefixes (system prompts, few-shot examples,
 *         earlier turns of a conversation) point at the same physical pages,
 *         with copy-on-write.
 *  [TABLE] "vLLM High-Performance Inference Engine: PagedAttention Principles
 *         and Deployment Guide", section "PagedAttention Architecture Deep
 *         Dive": block table with per-page ref_count.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pools: k_pool and v_pool are bf16 [num_blocks][num_kv_heads][block_size]
 *    [head_dim], row-major, one tensor per layer.  One (block, kv head) is a
 *    contiguous block_size*head_dim*2-byte run.
 *  - Block tables: int32 [num_seqs][max_blocks_per_seq]; entry i of row s is the
 *    physical block holding tokens i*B .. i*B+B-1 of sequence s.  Token j of a
 *    sequence sits in block table[s][j / B] at offset j % B.
 *  - Slots: int64, slot = block * block_size + offset; slot < 0 = no write.
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Every device pointer is owned by the caller; the library allocates no
 *    device memory.  Pointers marked "device" must be device memory of the
 *    current device; bf16 tensors must be 16-byte aligned.
 *  - Every GPU call is asynchronous and ordered on `stream` (a cudaStream_t
 *    passed as void*, NULL = legacy default stream).  The return value reports
 *    host-side validation and launch errors only.
 *  - Errors found on the device (bad context length, page or slot id) are
 *    or-ed into *err_flag (device int32, may be NULL) as PA_DEVERR_* bits and
 *    nothing traps.  Attention rows of a sequence or chunk with a bad context
 *    length are written as zeros; a block-table entry outside the pool is not
 *    read (its keys are left out by decode; a prefill tile holding it computes
 *    on whatever shared memory held), so rows that need it are unspecified;
 *    a bad slot or copy pair writes nothing.  The flag is never cleared by the
 *    library.
 *  - Attention reads slot j of a sequence only for j < its context length:
 *    slots past a context (the tail of its last block, blocks no table uses)
 *    may hold any bits, NaN included, without reaching the output.
 *  - Every GPU call may be captured into a CUDA graph (stream capture): a
 *    replay re-runs it with the arguments, launch plan and tensor maps bound
 *    at capture.  Split-K decode resets its arrival counters itself, so
 *    replays need no workspace clearing; the allocation-free decode wants its
 *    first call outside a capture (see below).
 *  - Thread safety: calls are re-entrant; the only global state is a
 *    per-device cache of SM count and of the driver's tensor-map encoder.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID = -1,     /* bad argument (null pointer, size, alignment) */
  PA_ERR_UNSUPPORTED = -2, /* valid but not built (head_dim, block_size, GQA group) */
  PA_ERR_CUDA = -3,        /* CUDA runtime / launch error */
  PA_ERR_OOM = -4,         /* block manager: no free block, or no host memory */
  PA_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required */
  PA_ERR_STATE = -6        /* block manager: unknown / duplicate sequence id,
                              reference count underflow */
} pa_status;

/* Device error bits or-ed into *err_flag. */
#define PA_DEVERR_CTX 1      /* context_len <= 0, > max_blocks_per_seq*B or > max_context_len */
#define PA_DEVERR_PAGE 2     /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 4     /* slot >= num_blocks * block_size */
#define PA_DEVERR_PAIR 8     /* copy pair with a block id outside [0, num_blocks) */
#define PA_DEVERR_TIMEOUT 16 /* an on-chip wait gave up (bounded waits only) */

/* Shape of one paged-attention call.  head_dim in {64, 128}; block_size in
 * {16, 32}; num_q_heads a multiple of num_kv_heads with a group of at most 16.
 * max_context_len bounds every context_lens[s] of the call (it sizes the
 * grid); scale multiplies q.k (1/sqrt(head_dim) per [ATT]). */
typedef struct pa_decode_desc {
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  int max_blocks_per_seq;
  int max_context_len;
  float scale;
} pa_decode_desc;

/* Library version string. */
const char *pa_version(void);

/* Human-readable name of a pa_status value. */
const char *pa_status_string(int status);

/* Bytes of device workspace pa_paged_attention_decode needs for `desc` on the
 * current device (0 when no context is split).  The workspace holds split-K
 * partial results and one 64-bit arrival counter per (sequence, kv head)
 * tagged with a per-call epoch, so it needs no initialisation and may be
 * reused across calls of any shape.  Returns 0 for an invalid desc. */
size_t pa_decode_workspace_bytes(const pa_decode_desc *desc);

/* Paged decode attention [ATT][PHASE]: for every sequence s and query head h,
 *   out[s][h] = sum_j softmax_j(scale * q[s][h] . k_j) v_j,  j = 0..ctx_s-1,
 * with k_j, v_j read from block block_tables[s][j / B], offset j % B of kv head
 * h / G.  ctx_s = context_lens[s] includes the token generated this step, whose
 * K/V must already be in the cache (pa_reshape_and_cache).  Softmax in fp32
 * with a running max; bf16 output.
 *   q            device bf16 [num_seqs][num_q_heads][head_dim]
 *   k_pool,v_pool device bf16 pools (layout above)
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens device int32 [num_seqs]
 *   out          device bf16 [num_seqs][num_q_heads][head_dim]
 *   workspace    device, >= pa_decode_workspace_bytes(desc) (may be NULL when
 *                that is 0), 16-byte aligned, any contents; calls that may
 *                overlap on the GPU must not share one
 *   err_flag     device int32 or NULL
 * Returns PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE or
 * PA_ERR_CUDA.  num_seqs == 0 launches nothing. */
int pa_paged_attention_decode(const pa_decode_desc *desc, const void *q, const void *k_pool,
                              const void *v_pool, const int32_t *block_tables,
                              const int32_t *context_lens, void *out, void *workspace,
                              size_t workspace_bytes, int32_t *err_flag, void *stream);

/* Decode attention with the step's cache write in the same launch: the
 * result of pa_reshape_and_cache of one new token per sequence followed by
 * pa_paged_attention_decode, bit for bit, in one kernel launch.  Sequence s's
 * new token is the last one it attends to, position ctx_s - 1 [ATT][PHASE];
 * its K/V go to the next free slot of the sequence's last block [SHARE].
 *   new_k, new_v  device bf16 [num_seqs][num_kv_heads][head_dim], 16-byte
 *                 aligned: the new token's K and V
 *   slot_mapping  device int64 [num_seqs]: the slot of position ctx_s - 1,
 *                 block_tables[s][(ctx_s-1)/B] * B + (ctx_s-1) % B, or < 0 for
 *                 no write (attention then reads what the slot holds)
 *   k_pool, v_pool are written (that slot of every kv head) and read.
 * A slot >= 0 that is not the slot of position ctx_s - 1 (outside the pool or
 * elsewhere in it) sets PA_DEVERR_SLOT and writes nothing; so does nothing a
 * sequence with a bad context length.  The block holding position ctx_s - 1
 * must not be read at that offset by another sequence of the call (a block
 * shared by several sequences is copied before it is written: copy-on-write).
 * Other arguments, the workspace and the errors as in
 * pa_paged_attention_decode. */
int pa_paged_attention_decode_append(const pa_decode_desc *desc, const void *q, const void *new_k,
                                     const void *new_v, const int64_t *slot_mapping, void *k_pool, void *v_pool,
                                     const int32_t *block_tables, const int32_t *context_lens, void *out,
                                     void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream);

/* Bytes of device workspace pa_paged_attention_decode_shared_prefix needs for
 * `desc` on the current device (decode split-K scratch plus up to eight fp32
 * partial softmax states per (sequence, query head), one per key range of the
 * prefix); 0 for an invalid desc. */
size_t pa_shared_prefix_workspace_bytes(const pa_decode_desc *desc);

/* Shared-prefix-aware decode [ATT][PHASE][SHARE]: the same result as
 * pa_paged_attention_decode (within rounding), for batches in which groups of
 * sequences point at the same physical pages for a common prefix (shared
 * system prompts, parallel samples, beam candidates).  Group k is the
 * sequences group_starts[k] .. group_starts[k+1]-1 (consecutive, groups
 * disjoint and ordered; sequences outside every group are decoded normally);
 * they share their first group_prefix_lens[k] tokens, a positive multiple of
 * block_size, held in blocks prefix_tables[k][0 ..] -- the same blocks that
 * lead every member's own block-table row.  The prefix is attended once for
 * all of the group's query rows on the tensor cores (fp32 partial softmax
 * states, the prefix cut into up to 8 key ranges when the groups alone would
 * not fill the GPU), then each sequence attends its own keys prefix .. ctx-1
 * and merges.
 *   group_starts       device int32 [num_groups + 1]
 *   group_prefix_lens  device int32 [num_groups], <= each member's context
 *   prefix_tables      device int32 [num_groups][prefix_max_blocks]
 *   max_group_size     bound on every group's size (sizes the grid)
 *   max_prefix_len     bound on every group_prefix_lens[k], <= max_context_len
 *   workspace          >= pa_shared_prefix_workspace_bytes(desc), any contents
 * head_dim must be 128 and the GQA group 1, 2, 4, 8 or 16 when num_groups > 0;
 * num_groups == 0 is plain decode.  Other arguments and errors as in
 * pa_paged_attention_decode; a prefix length that is not a multiple of B or
 * exceeds a member's context sets PA_DEVERR_CTX for that member. */
int pa_paged_attention_decode_shared_prefix(const pa_decode_desc *desc, const void *q, const void *k_pool,
                                            const void *v_pool, const int32_t *block_tables,
                                            const int32_t *context_lens, int num_groups,
                                            const int32_t *group_starts, const int32_t *group_prefix_lens,
                                            const int32_t *prefix_tables, int prefix_max_blocks,
                                            int max_group_size, int max_prefix_len, void *out, void *workspace,
                                            size_t workspace_bytes, int32_t *err_flag, void *stream);

/* Shared-prefix decode with a second level of sharing [ATT][SHARE]: the
 * groups of pa_paged_attention_decode_shared_prefix (their prefixes attended
 * once on the tensor cores), and a partition of all sequences into
 * consecutive sub-groups whose members share more leading blocks -- the
 * samples of one prompt under parallel sampling share the prompt's pages,
 * and only the blocks written since each copy-on-write are their own.
 * Sub-group k is sequences subgroup_starts[k] .. subgroup_starts[k+1]-1
 * (subgroup_starts[0] = 0, subgroup_starts[num_subgroups] = num_seqs), whose
 * block-table rows agree on keys 0 .. subgroup_shared_lens[k]-1 (a multiple
 * of block_size, at least the prefix length of the group that holds them (0
 * outside every group), at most each member's context).  Decode runs one unit
 * per (sub-group, kv head): the sub-group's shared keys past the group prefix
 * are read once for all of its members' query rows, each member's remaining
 * keys for that member's rows only, and the group prefix's states are folded
 * in.  Same result as pa_paged_attention_decode (within rounding).
 *   subgroup_starts       device int32 [num_subgroups + 1]
 *   subgroup_shared_lens  device int32 [num_subgroups]
 *   max_subgroup_size     bound on every sub-group's size; times the GQA group
 *                         size at most 16
 * head_dim must be 128; the members of a sub-group must lie in one group (or
 * in none).  A sub-group with an invalid shared length or a member with a bad
 * context, or more than 512 blocks to read in all (shared plus every member's
 * own), gets zero rows and PA_DEVERR_CTX.  num_subgroups == 0 is
 * pa_paged_attention_decode_shared_prefix.  Other arguments, the workspace
 * (pa_shared_prefix_workspace_bytes) and errors as there. */
int pa_paged_attention_decode_shared_prefix2(const pa_decode_desc *desc, const void *q, const void *k_pool,
                                             const void *v_pool, const int32_t *block_tables,
                                             const int32_t *context_lens, int num_groups,
                                             const int32_t *group_starts, const int32_t *group_prefix_lens,
                                             const int32_t *prefix_tables, int prefix_max_blocks, int max_group_size,
                                             int max_prefix_len, int num_subgroups, const int32_t *subgroup_starts,
                                             const int32_t *subgroup_shared_lens, int max_subgroup_size, void *out,
                                             void *workspace, size_t workspace_bytes, int32_t *err_flag,
                                             void *stream);

/* Size of the fixed device scratch array of pa_paged_attention_decode_noalloc
 * (8 MiB, held on every GPU that loads the library until the process exits). */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Paged decode attention that allocates nothing and takes no workspace.  No
 * page describes this call; it exists for callers that cannot allocate device
 * memory (a plugin whose host framework owns all device memory, a path where
 * cudaMalloc's implicit synchronisation is not allowed, memory fixed at
 * start-up).  Same arguments, results and errors as pa_paged_attention_decode
 * without the workspace pair: the split-K scratch is a file-scope device array
 * of PA_NOALLOC_SCRATCH_BYTES.  Calls no cudaMalloc/cudaFree and no allocating
 * library routine.
 *  - Returns PA_ERR_WORKSPACE, before any launch, when the shape needs more
 *    scratch than PA_NOALLOC_SCRATCH_BYTES (pa_decode_workspace_bytes(desc)
 *    tells how much it needs).
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress) and caches it with the id of the
 *    device's context; make that first call before any stream capture.  A
 *    call under a different context (after cudaDeviceReset, say) looks the
 *    address up again, so the first call after a reset must also come before
 *    any capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents; nothing in it has to start at zero (its arrival counters are
 *    tagged per call).  Calls that may overlap on the GPU race on the array:
 *    order them on one stream or serialise them. */
int pa_paged_attention_decode_noalloc(const pa_decode_desc *desc, const void *q,
                                      const void *k_pool, const void *v_pool,
                                      const int32_t *block_tables, const int32_t *context_lens,
                                      void *out, int32_t *err_flag, void *stream);

/* Causal chunked-prefill attention [PHASE][CHUNK] on the tensor cores.
 * Chunk r (r < desc->num_seqs) has C_r = cu_q[r+1] - cu_q[r] query tokens and
 * context ctx_r = context_lens[r] that INCLUDES the chunk (its K/V must already
 * be cached, e.g. by pa_reshape_and_cache).  Query row i of chunk r sits at
 * position ctx_r - C_r + i and attends keys 0 .. ctx_r - C_r + i of the
 * chunk's block-table row:
 *   out[cu_q[r]+i][h] = sum_j softmax_j(scale * q[cu_q[r]+i][h] . k_j) v_j.
 * QK^T and PV run as tcgen05 MMAs (bf16 in, fp32 accumulate in TMEM); softmax
 * in fp32; bf16 output.
 *   q          device bf16 [total_q][num_q_heads][128]
 *   cu_q       device int32 [R + 1], non-decreasing, cu_q[R] <= total_q
 *   max_q_len  bound on every C_r (sizes the grid); total_q = rows of q / out
 *   out        device bf16 [total_q][num_q_heads][128]; rows outside every
 *              chunk are not written
 * head_dim must be 128 and the GQA group size 1, 2, 4, 8 or 16.  A chunk
 * with C_r > ctx_r, ctx_r > max_context_len or a row range outside
 * [0, total_q) sets PA_DEVERR_CTX (its rows are zeroed when in range).  Other
 * arguments and errors as in pa_paged_attention_decode (no workspace). */
int pa_paged_attention_prefill_chunk(const pa_decode_desc *desc, const void *q,
                                     const int32_t *cu_q, int max_q_len, int total_q,
                                     const void *k_pool, const void *v_pool,
                                     const int32_t *block_tables, const int32_t *context_lens,
                                     void *out, int32_t *err_flag, void *stream);

/* The attention of one continuous-batching step [CHUNK] in one launch: the
 * causal chunked prefill of prefill_desc->num_seqs chunks and the decode of
 * decode_desc->num_seqs sequences over the same pools, run side by side (the
 * tensor-bound prefill tiles and the HBM-bound decode units share the GPU
 * instead of taking turns).  The results are those of
 *   pa_paged_attention_prefill_chunk(prefill_desc, prefill_q, cu_q, max_q_len,
 *       total_q, k_pool, v_pool, prefill_tables, prefill_context_lens,
 *       prefill_out, ...)
 *   pa_paged_attention_decode(decode_desc, decode_q, k_pool, v_pool,
 *       decode_tables, decode_context_lens, decode_out, workspace, ...)
 * bit for bit, with the arguments, layouts and errors of those two calls
 * (the workspace: pa_decode_workspace_bytes(decode_desc)).  Both descs must
 * describe the same pools (num_q_heads, num_kv_heads, head_dim = 128,
 * block_size, num_blocks) and the GQA group must be 1, 2, 4, 8 or 16;
 * otherwise PA_ERR_INVALID / PA_ERR_UNSUPPORTED.  Either part may be empty
 * (num_seqs == 0, or no prefill rows).  The K/V of every token attended must
 * already be cached (pa_reshape_and_cache). */
int pa_paged_attention_mixed(const pa_decode_desc *prefill_desc, const void *prefill_q, const int32_t *cu_q,
                             int max_q_len, int total_q, const int32_t *prefill_tables,
                             const int32_t *prefill_context_lens, void *prefill_out,
                             const pa_decode_desc *decode_desc, const void *decode_q, const int32_t *decode_tables,
                             const int32_t *decode_context_lens, void *decode_out, void *workspace,
                             size_t workspace_bytes, const void *k_pool, const void *v_pool, int32_t *err_flag,
                             void *stream);

/* Writes the K/V of num_tokens new tokens into their cache slots [PHASE][SHARE]:
 *   k_pool[slot / B][h][slot % B][:] = k[t][h][:]  (same for v), for t in order.
 * Bit-exact copy.  slot < 0: token skipped.  slot >= num_blocks*B: skipped and
 * PA_DEVERR_SLOT set.  Two tokens with the same slot: unspecified which wins.
 *   k, v          device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping  device int64 [num_tokens] */
int pa_reshape_and_cache(const void *k, const void *v, void *k_pool, void *v_pool,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, int32_t *err_flag,
                         void *stream);

/* Copy-on-write page copies [SHARE][TABLE]: for every layer l and pair i,
 *   block pairs[i][1] of k_pools[l] and v_pools[l] := block pairs[i][0].
 * A block is block_bytes = num_kv_heads*block_size*head_dim*2 contiguous bytes
 * (a multiple of 16).  Bit-exact.  Destinations must be distinct and must not
 * also be sources within one call (the copies run concurrently).
 *   k_pools, v_pools  HOST arrays of num_layers device pointers (1..256 layers)
 *   block_pairs       device int64 [num_pairs][2] (src, dst)
 * A pair with an id outside [0, num_blocks) is skipped with PA_DEVERR_PAIR. */
int pa_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                   const int64_t *block_pairs, int num_pairs, int num_blocks, size_t block_bytes,
                   int32_t *err_flag, void *stream);

/* Block moves between two pools for preemptive swapping [CHUNK] (a paused
 * request's pages go to host RAM and come back later): for every layer l and
 * pair i, block pairs[i][1] of dst_*_pools[l] := block pairs[i][0] of
 * src_*_pools[l], K and V.  Either side may be device memory or pinned host
 * memory the GPU can address (cudaHostAlloc / cudaHostRegister; on
 * Grace-Blackwell the kernel reads and writes it over the chip-to-chip link).
 * Bit-exact.  Destination blocks must be distinct.
 *   *_pools      HOST arrays of num_layers pointers (1..256 layers)
 *   block_pairs  device int64 [num_pairs][2] (src block, dst block)
 *   src_num_blocks / dst_num_blocks  blocks in each source / destination pool
 *   block_bytes  num_kv_heads*block_size*head_dim*2, a multiple of 16
 * A pair outside either pool is skipped with PA_DEVERR_PAIR. */
int pa_swap_blocks(void *const *src_k_pools, void *const *src_v_pools, void *const *dst_k_pools,
                   void *const *dst_v_pools, int num_layers, const int64_t *block_pairs, int num_pairs,
                   int src_num_blocks, int dst_num_blocks, size_t block_bytes, int32_t *err_flag,
                   void *stream);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------ */

/* HBM bandwidth probe, the ceiling the decode kernels are measured against
 * [PHASE] (decode streams the cache from HBM).
 *  mode 0: reads `bytes` from src with 16-byte vector loads and writes nothing
 *          (sink: a device 16-byte word, written only if the loads' XOR equals
 *          a fixed constant -- never with random data -- so that no load can
 *          be dropped); 8 CTAs of 256 threads per SM stride over the buffer,
 *          8 independent loads in flight per thread.
 *  mode 1: copies src to dst with 16-byte vector loads and stores (read +
 *          write bytes), same grid.
 *  mode 2: reads `bytes` from src through the TMA engine (bulk copies of 16 KB
 *          into an 8-slot shared-memory ring, one CTA per SM), the path the
 *          decode kernels' page gathers take; its bounded waits report
 *          PA_DEVERR_TIMEOUT into *err_flag (device int32, may be NULL).
 *  mode 3: reads like paged decode: 4 KB runs (a (block, kv head) of 16
 *          tokens x 128 bf16) as K/V pairs at pseudo-random places (a
 *          permutation of the runs of each half of src), with the decode
 *          kernel's concurrency (2 CTAs of 4 warps per SM, three 8 KB slots a
 *          warp); reads the largest power-of-two number of runs fitting each
 *          half (bytes read: 2 x 4096 x that number, which the caller counts);
 *          timeouts as in mode 2.
 * src, dst, sink device memory, 16-byte aligned (dst only for mode 1, sink
 * only for mode 0); bytes a nonzero multiple of 16; use a buffer several times
 * the L2 (129 MB) so the stream comes from HBM.  PA_ERR_INVALID on bad
 * arguments; asynchronous on stream (time it with events). */
int pa_hbm_probe(const void *src, void *dst, size_t bytes, int mode, void *sink, int32_t *err_flag, void *stream);

/* Self-test of the bounded on-chip wait.  Every kernel of this library waits
 * on shared-memory mbarriers (for TMA copies and tensor-core MMAs) with a
 * bound of about 2 s, after which it sets PA_DEVERR_TIMEOUT in *err_flag,
 * skips the rest of its work and returns, so that a stuck wait cannot hang
 * the GPU.  This launches one warp that waits, through the same bounded-wait
 * routine and with the same reporting, on an mbarrier nothing arrives on, for
 * at most limit_cycles SM cycles (1 .. the library's own bound, 4e9), then
 * sets *done (device int32) to 1.  Expected result: PA_DEVERR_TIMEOUT in
 * *err_flag (device int32, may be NULL), *done == 1, and a usable context.
 * No page describes this call. */
int pa_selftest_bounded_wait(long long limit_cycles, int32_t *err_flag, int32_t *done, void *stream);

/* ------------------------------------------------------------------------
 * Host block manager [TABLE][SHARE][CHUNK] (plain C++, no GPU): a free list
 * of num_blocks physical blocks of block_size tokens, per-sequence block
 * tables, per-block reference counts.  Blocks are allocated on demand (a
 * sequence of n tokens holds ceil(n / B) blocks), shared by fork, copied on
 * write when a sharer appends into a block with ref_count > 1, and returned to
 * the free pool when the last reference is dropped.  Free blocks that hold no
 * prefix-cache content are handed out first, most recently freed first
 * (initially in increasing id order); free blocks still in the prefix cache
 * only after them, least recently freed first.  Not thread safe.
 * No C++ exception leaves these calls: a failed host allocation returns
 * PA_ERR_OOM (NULL from the create calls, -1 from pa_bm_wasted_slots) and
 * leaves the manager as it was before the call.
 * ------------------------------------------------------------------------ */
typedef struct pa_bm pa_bm;

/* NULL on bad arguments (num_blocks <= 0 or block_size <= 0) or no memory. */
pa_bm *pa_bm_create(int num_blocks, int block_size);

/* The same with num_host_blocks (>= 0) host blocks for swapped-out sequences. */
pa_bm *pa_bm_create_with_host(int num_blocks, int num_host_blocks, int block_size);
void pa_bm_destroy(pa_bm *bm);

/* New sequence seq_id (>= 0, unused) holding num_tokens (>= 0) tokens:
 * allocates ceil(num_tokens / B) blocks.  Its token ids are not known, so
 * none of its blocks enters the prefix cache (pa_bm_add_seq_tokens admits a
 * prompt by its ids).  PA_ERR_OOM leaves no trace. */
int pa_bm_add_seq(pa_bm *bm, int seq_id, int num_tokens);

/* child shares every block of parent (ref_count + 1 each), same length. */
int pa_bm_fork(pa_bm *bm, int parent_id, int child_id);

/* Appends one token to seq_id.  *slot_out gets its slot.  If the token starts
 * a new block, a free block is taken.  If it lands in a block with ref_count >
 * 1, a fresh block is taken, cow_pair_out = {old, new} is returned for
 * pa_copy_blocks, and the old block's ref_count drops by one; otherwise
 * cow_pair_out = {-1, -1}.  PA_ERR_OOM leaves the sequence unchanged. */
int pa_bm_append(pa_bm *bm, int seq_id, int64_t *slot_out, int64_t cow_pair_out[2]);

/* pa_bm_append with the token's id [SHARE].  While every token id of seq_id is known
 * (it was admitted by pa_bm_add_seq_tokens, or forked from such a sequence,
 * and every append since gave its id), a block this token fills is
 * registered in the prefix cache like a prompt's full block -- when the
 * blocks before it are registered, so that a lookup from the start can
 * reach it -- and a later prompt that repeats the sequence (the next turn of
 * a conversation: earlier prompt, generated answer, new message) finds it.
 * Its K/V are valid once this step's cache write of the token has run.
 * pa_bm_append (no id) ends the tracking: none of the sequence's later
 * blocks is registered. */
int pa_bm_append_token(pa_bm *bm, int seq_id, int32_t token, int64_t *slot_out, int64_t cow_pair_out[2]);

/* One decode step's appends in one call: one token onto each of
 * seq_ids[0..n-1] (distinct, resident sequences), in that order, exactly as
 * n calls of pa_bm_append_token (tokens[n] given) or pa_bm_append (tokens
 * NULL) would do them.  slots_out[n] gets each token's slot and
 * cow_pairs_out[n][2] each copy-on-write pair ({-1, -1} for none).
 * Everything is checked before anything changes: PA_ERR_STATE (an unknown or
 * swapped-out id), PA_ERR_INVALID (a repeated id, null pointers, n < 0) and
 * PA_ERR_OOM (the step needs more free blocks than there are) leave the
 * manager and the output arrays untouched.  n == 0 does nothing. */
int pa_bm_append_batch(pa_bm *bm, const int32_t *seq_ids, const int32_t *tokens, int n, int64_t *slots_out,
                       int64_t *cow_pairs_out);

/* Drops seq_id: every block's ref_count - 1, blocks reaching 0 go back to the
 * free list (the <eos> path of [CHUNK]). */
int pa_bm_free_seq(pa_bm *bm, int seq_id);

/* Copies seq_id's block table into out[0..cap-1]; *n = its length.  Returns
 * PA_ERR_INVALID if cap < *n (nothing copied beyond cap). */
int pa_bm_block_table(const pa_bm *bm, int seq_id, int32_t *out, int cap, int *n);

/* The block tables of seq_ids[0..n-1] as one row-major int32 matrix
 * out[n][max_blocks], the layout the attention calls take: row i holds
 * sequence i's blocks, then pad up to max_blocks (the kernels never read
 * past ceil(context_len / B) entries of a row).  context_lens_out[n] (may
 * be NULL) gets each sequence's length in tokens.  PA_ERR_STATE (an unknown
 * or swapped-out id) and PA_ERR_INVALID (a table longer than max_blocks,
 * null pointers) are returned before anything is written. */
int pa_bm_block_tables(const pa_bm *bm, const int32_t *seq_ids, int n, int32_t *out, int max_blocks, int32_t pad,
                       int32_t *context_lens_out);

/* Automatic prefix caching [SHARE]: like pa_bm_add_seq for a prompt of
 * num_tokens token ids, but every full block of the prompt is registered by
 * content (the block before it and its block_size token ids, compared
 * exactly), and a new prompt reuses the longest chain of registered full
 * blocks from its start (ref_count + 1 each; a registered block keeps its
 * content after its last user frees it, until the block is handed out
 * again; then every registered block that continued it -- its K/V were
 * computed after the old content -- leaves the cache with it).  The first
 * call allocates num_blocks * block_size token ids of host memory for the
 * cache's keys.  *cached_tokens (may be NULL) gets the number of leading tokens
 * whose K/V are already in the cache: the caller writes and prefills only
 * tokens cached_tokens .. num_tokens-1.  A block registered here holds valid
 * K/V once this sequence's prefill of it has run.  PA_ERR_OOM leaves no
 * trace. */
int pa_bm_add_seq_tokens(pa_bm *bm, int seq_id, const int32_t *tokens, int num_tokens, int *cached_tokens);

/* Number of blocks currently registered in the prefix cache (free ones
 * included). */
int pa_bm_num_cached_blocks(const pa_bm *bm);

/* Moves seq_id to host blocks (preemption): every block must be unshared
 * (ref_count 1, else PA_ERR_STATE).  Writes *n (device block, host block)
 * pairs for pa_swap_blocks (device pools -> host pools) into pairs_out
 * [cap][2] and frees the device blocks.  PA_ERR_OOM (not enough free host
 * blocks) and PA_ERR_INVALID (cap < *n) leave everything unchanged.  While
 * swapped, the sequence cannot be forked, appended to or listed. */
int pa_bm_swap_out(pa_bm *bm, int seq_id, int64_t *pairs_out, int cap, int *n);

/* Brings a swapped-out seq_id back: new device blocks, *n (host block, device
 * block) pairs for pa_swap_blocks (host pools -> device pools); the host
 * blocks are freed.  PA_ERR_OOM leaves everything unchanged. */
int pa_bm_swap_in(pa_bm *bm, int seq_id, int64_t *pairs_out, int cap, int *n);

/* Number of free host blocks. */
int pa_bm_num_free_host(const pa_bm *bm);

/* Tokens held by seq_id, or -1 if unknown. */
int pa_bm_seq_len(const pa_bm *bm, int seq_id);

/* Reference count of a block (0 = free), -1 if out of range. */
int pa_bm_ref_count(const pa_bm *bm, int block);

/* Number of free blocks. */
int pa_bm_num_free(const pa_bm *bm);

/* Unused token slots in allocated blocks over all live sequences (each shared
 * block counted once), i.e. internal fragmentation in tokens. */
int64_t pa_bm_wasted_slots(const pa_bm *bm);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
