// Paged decode attention for sm_103a.
//
// Computes, for every sequence s and query head h, the attention of
// "Configuring vLLM and PagedAttention for High Throughput Enterprise LLM
// Serving" ("Architectural Foundations: PagedAttention & Virtual Memory"):
//   out = sum_j softmax_j(scale * q.k_j) v_j,  k_j, v_j in block BlockTable[j / B]
// over the whole cached context -- the bandwidth-bound decode phase of
// "Memory Bottlenecks in Autoregressive LLM Inference" on the same page.
//
// Design (one CTA per (context part, kv head, sequence), 4 warps):
//  * The part's block-table entries are staged once in shared memory.
//  * Each warp owns every 4th page of the part and a private ring of NST
//    shared-memory slots.  Lane 0 gathers a page's K and V runs (B rows x D
//    bf16 each, one (block, kv head) run is contiguous in the pool) with 2-D TMA
//    loads (128-byte swizzle, L2 evict-first) that complete on the slot's
//    mbarrier.  No warp ever waits for another warp while streaming.
//  * QK^T and PV are warp MMAs (m16n8k16, bf16 in, fp32 accumulate): tokens are
//    the M side of S^T = K Q^T (the G query heads of the kv head are the N side,
//    so one K page read serves the whole GQA group), and d is the M side of
//    O^T = V^T P^T.  The probabilities move from the S^T accumulator to the PV
//    operand with movmatrix (no shared-memory round trip).
//  * Online softmax in fp32 (running max and sum, base-2 exponent).  The
//    probabilities are rounded to bf16 once and the same rounded values feed
//    both the PV product and the running sum.
//  * Warps are merged in shared memory at the end; a context cut into several
//    parts writes (o/l, m, l) per part to the workspace, and the last CTA of a
//    (sequence, kv head) to arrive (atomic counter, no waiting) merges the
//    parts in part order -- deterministic, one launch.  The counter carries a
//    per-call epoch tag, so stale workspace contents never need clearing.
//  * When the grid fills a few waves of the resident slots, CTAs map to
//    sequences longest context first (an in-kernel rank over the lengths).
//  * Every mbarrier wait is bounded; a timeout sets PA_DEVERR_TIMEOUT.
//  * Shared-prefix launches: a sequence in a group starts at the end of the
//    group's prefix, whose partial softmax states a tensor-core pass wrote
//    before; they are loaded before streaming and folded in at the end.
//  * Sub-group mode (shared-prefix decode, second level): one CTA per
//    (sub-group, kv head) streams the blocks the members share once for all
//    of their query rows (member x head as the MMA N side, up to 16), then
//    each member's own blocks with the other members' columns masked.
//  * Optionally (decode with append) the CTA that streams a sequence's last
//    page also stores the step's new token (K/V at position ctx-1) into its
//    slot of the pools and patches that row of its shared-memory copy of the
//    page before the products -- the cache write of the decode step rides in
//    the attention launch instead of a launch of its own.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>

#include "pa_decode_body.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

template <int D, int B, int NT, int NW, int NST, bool PRE, bool APP, bool GRP>
__global__ void __launch_bounds__(NW * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  decode_unit<D, B, NT, NW, NST, PRE, APP, GRP, D == 128>(&tmK, &tmV, a, lin, threadIdx.x, smem, 0);
}

template <int D, int B, int NT, bool PRE, bool APP, bool GRP = false, int NST16 = 3>
int launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a, dim3 grid,
                  cudaStream_t st) {
  // 16-token pages: 3 slots a warp (96 KB, 2 CTAs per SM), or NST16 = 2 (64
  // KB, 3 CTAs per SM) when the caller asks; 32-token pages: 1 slot a warp
  // (64 KB, 3 CTAs per SM) -- with 2 slots a CTA would hold 128 KB and one
  // CTA per SM could not hide its own set-up and merge.  The shared-prefix
  // launch, whose own key ranges are typically short, takes 2 slots with
  // 16-token pages: more CTAs in flight hide the set-up of short units
  // (prefix sharing: 72.6 -> 61.1 us).
  constexpr int NW = 4;
  constexpr int NST = (B == 16) ? (PRE ? 2 : NST16) : 1;
  using L = DecodeSmem<D, B, NW, NST>;
  static_assert(L::kAlloc <= 227 * 1024, "decode shared memory over the per-CTA limit");
  auto kern = decode_kernel<D, B, NT, NW, NST, PRE, APP, GRP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  kern<<<grid, NW * 32, L::kAlloc, st>>>(tk, tv, a);
  return launch_status(cudaGetLastError());
}

template <int D, int B>
int dispatch_nt(int G, const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a, dim3 grid,
                cudaStream_t st) {
  // Separate instances keep the plain decode's registers: the shared-prefix
  // launch (prefix states prefetched), the sub-group launch and the decode
  // with append.
  // A launch whose units all fit one wave at 2 CTAs per SM takes 2 slots a
  // warp (32K contexts, 256 units of 512 pages: 165.1 -> 160.1 us); more
  // units keep 3 (Llama-3-8B-shaped decode, 512 units: 51.2 us, 53.3 with 2;
  // parallel sampling, 512 sub-group units: 120.7 us, 124.6 with 2).
  const bool one_wave = (long long)grid.x * grid.y * grid.z <= 2ll * current_sm_count();
  if constexpr (D == 128)
    if (a.nsub > 0) {
      if (B == 16 && one_wave)
        return a.sub_rows <= 8 ? launch_decode<D, B, 1, false, false, true, 2>(tk, tv, a, grid, st)
                               : launch_decode<D, B, 2, false, false, true, 2>(tk, tv, a, grid, st);
      return a.sub_rows <= 8 ? launch_decode<D, B, 1, false, false, true>(tk, tv, a, grid, st)
                             : launch_decode<D, B, 2, false, false, true>(tk, tv, a, grid, st);
    }
  if (a.ngroups > 0)
    return G <= 8 ? launch_decode<D, B, 1, true, false>(tk, tv, a, grid, st)
                  : launch_decode<D, B, 2, true, false>(tk, tv, a, grid, st);
  if (B == 16 && G <= 8 && one_wave) {
    if (a.app_slots) return launch_decode<D, B, 1, false, true, false, 2>(tk, tv, a, grid, st);
    return launch_decode<D, B, 1, false, false, false, 2>(tk, tv, a, grid, st);
  }
  if (a.app_slots)
    return G <= 8 ? launch_decode<D, B, 1, false, true>(tk, tv, a, grid, st)
                  : launch_decode<D, B, 2, false, true>(tk, tv, a, grid, st);
  return G <= 8 ? launch_decode<D, B, 1, false, false>(tk, tv, a, grid, st)
                : launch_decode<D, B, 2, false, false>(tk, tv, a, grid, st);
}

}  // namespace
}  // namespace pa

namespace pa {

int decode_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_tables, const int32_t *context_lens, void *out, void *workspace,
                  size_t workspace_bytes, int32_t *err_flag, void *stream, const DecodePrefix *pre,
                  const DecodeAppend *app) {
  int st = validate_decode_desc(d);
  if (st != PA_OK) return st;
  if (d->num_seqs == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (app && (pre || !app->new_k || !app->new_v || !app->slots || !aligned16(app->new_k) || !aligned16(app->new_v)))
    return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PA_ERR_INVALID;
  if (d->num_seqs > 65535 || d->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const DecodePlan plan = make_decode_plan(d, sms);
  if (plan.total() > 0 && (!workspace || workspace_bytes < plan.total() || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  const uint64_t rows = (uint64_t)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tk, tv;  // head_dim 128: a page's two 64-column halves in one copy
  if (d->head_dim == 128 ? !encode_kv_halves_3d(&tk, k_pool, rows, d->block_size) ||
                               !encode_kv_halves_3d(&tv, v_pool, rows, d->block_size)
                         : !encode_2d_bf16(&tk, k_pool, rows, d->head_dim, d->block_size, 64, true) ||
                               !encode_2d_bf16(&tv, v_pool, rows, d->head_dim, d->block_size, 64, true))
    return PA_ERR_CUDA;
  DecodeArgs a;
  fill_decode_args(&a, d, plan, q, block_tables, context_lens, out, workspace, err_flag,
                   (long long)sms * (d->block_size == 16 ? 2 : 3));
  a.grp_start = pre ? pre->grp_start : nullptr;
  a.grp_prefix = pre ? pre->grp_prefix : nullptr;
  a.ngroups = pre ? pre->ngroups : 0;
  a.pre_o = pre ? pre->pre_o : nullptr;
  a.pre_ml = pre ? pre->pre_ml : nullptr;
  a.npre = pre ? pre->npre : 0;
  a.sub_start = pre ? pre->sub_start : nullptr;
  a.sub_shared = pre ? pre->sub_shared : nullptr;
  a.nsub = pre ? pre->nsub : 0;
  a.sub_rows = pre ? pre->sub_rows : 0;
  if (a.nsub > 0 && (d->head_dim != 128 || a.sub_rows > 16 || a.sub_rows <= 0)) return PA_ERR_UNSUPPORTED;
  a.app_k = app ? static_cast<const uint4 *>(app->new_k) : nullptr;
  a.app_v = app ? static_cast<const uint4 *>(app->new_v) : nullptr;
  a.app_slots = app ? app->slots : nullptr;
  a.kp = app ? static_cast<uint4 *>(const_cast<void *>(k_pool)) : nullptr;
  a.vp = app ? static_cast<uint4 *>(const_cast<void *>(v_pool)) : nullptr;
  // one CTA per (part, kv head, sequence); sub-groups: per (kv head, sub-group)
  const dim3 grid(a.nsub > 0 ? 1 : plan.max_parts, d->num_kv_heads, a.nsub > 0 ? a.nsub : d->num_seqs);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->head_dim == 128)
    return d->block_size == 16 ? dispatch_nt<128, 16>(a.G, tk, tv, a, grid, s)
                               : dispatch_nt<128, 32>(a.G, tk, tv, a, grid, s);
  return d->block_size == 16 ? dispatch_nt<64, 16>(a.G, tk, tv, a, grid, s)
                             : dispatch_nt<64, 32>(a.G, tk, tv, a, grid, s);
}

}  // namespace pa

extern "C" int pa_paged_attention_decode(const pa_decode_desc *d, const void *q, const void *k_pool,
                                         const void *v_pool, const int32_t *block_tables,
                                         const int32_t *context_lens, void *out, void *workspace,
                                         size_t workspace_bytes, int32_t *err_flag, void *stream) {
  return pa::decode_launch(d, q, k_pool, v_pool, block_tables, context_lens, out, workspace, workspace_bytes,
                           err_flag, stream, nullptr, nullptr);
}

extern "C" int pa_paged_attention_decode_append(const pa_decode_desc *d, const void *q, const void *new_k,
                                                const void *new_v, const int64_t *slot_mapping, void *k_pool,
                                                void *v_pool, const int32_t *block_tables,
                                                const int32_t *context_lens, void *out, void *workspace,
                                                size_t workspace_bytes, int32_t *err_flag, void *stream) {
  if (!new_k || !new_v || !slot_mapping) return PA_ERR_INVALID;
  const pa::DecodeAppend app{new_k, new_v, slot_mapping};
  return pa::decode_launch(d, q, k_pool, v_pool, block_tables, context_lens, out, workspace, workspace_bytes,
                           err_flag, stream, nullptr, &app);
}
