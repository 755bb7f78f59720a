// Causal chunked-prefill attention over the paged KV cache, on the tcgen05
// tensor cores of sm_103a.
//
// Follows "Configuring vLLM and PagedAttention for High Throughput Enterprise
// LLM Serving": the prefill phase attends every prompt position at once and is
// compute bound ("Memory Bottlenecks in Autoregressive LLM Inference"); long
// prompts are processed in chunks (512 or 1024 tokens) that ride along with
// decode iterations ("High-Throughput Batching: Continuous Batching & Chunked
// Prefill"); keys and values are read through the block table,
// P_physical = BlockTable[j / B] ("Architectural Foundations").  A chunk of C
// query tokens over a context of ctx tokens (the chunk included) places query
// row i at position ctx - C + i; it attends keys 0 .. ctx - C + i.
//
// One CTA per (pair of query tiles, kv head, chunk).  A query tile is 128 MMA
// rows: 128/G consecutive positions x the G query heads that share the kv
// head; the CTA holds two consecutive tiles (A and B), so every K/V tile it
// loads serves 256 rows.  Roles (12 warps, three warpgroups):
//   warps 0-3  tile A: load its Q rows, softmax of one row each (TMEM lane =
//              row), write P (bf16) back into TMEM over its S, rescale O,
//              store the output;
//   warps 4-7  the same for tile B;
//   warp 8     gathers 128-key K and V tiles with 2-D TMA (128-byte
//              swizzle; one lane per page) into two-stage K and V rings; a K
//              stage is refilled once both S MMAs of its tile are done, a V
//              stage once both PV MMAs are;
//   warp 9     owns the TMEM allocation and issues the MMAs in the order
//              S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...:
//              S = Q K^T (A and B from shared memory, fp32 into TMEM) and
//              O += P V (P from TMEM, V MN-major from shared memory);
//   warps 10-11 idle (they complete the third warpgroup, whose registers go
//              to the softmax warpgroups).
// MMAs issued by one thread complete in order, so an S MMA that reuses the
// TMEM columns of the previous tile's P runs after the PV MMA that read them,
// and a completed S tells the softmax that the previous PV is done.
// The softmax keeps a running max per row in base 2 and rescales O only when
// the max grows by more than 8 (2^8); until then probabilities are taken
// against the stale max, which the final normalisation by the same running
// sum makes exact.  Value rows of keys past the context are zeroed in shared
// memory before they meet a zero probability (unused cache slots may hold
// NaNs).  Chunks start in order of decreasing context.  Every wait is
// bounded; a timeout sets PA_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pa_internal.h"
#include "pa_prefill_body.cuh"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

template <int B, int G, bool PARTIAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const PrefillArgs a) {
  // The partial-state pass (a group's shared prefix) lets a programmatic
  // dependent start beside it at once: the shared-prefix decode's task grid
  // reads nothing this pass writes.
  if constexpr (PARTIAL) asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  prefill_tile<B, G, PARTIAL>(&tmK, &tmV, a, blockIdx.x, blockIdx.y, blockIdx.z, gridDim.x, smem);
}

template <int B, int G>
int launch_prefill(const CUtensorMap &tk, const CUtensorMap &tv, const PrefillArgs &a, dim3 grid,
                   cudaStream_t st) {
  // partial states (the shared-prefix pass) or bf16 rows: separate kernels,
  // so that each keeps its own register allocation
  auto kern = a.part_o ? prefill_kernel<B, G, true> : prefill_kernel<B, G, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return PA_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PA_ERR_CUDA;
  if (fa.numRegs < kRegsLaunch) return PA_ERR_UNSUPPORTED;  // the register split would not fit
  kern<<<grid, kThreads, kSmem, st>>>(tk, tv, a);
  return launch_status(cudaGetLastError());
}

template <int B>
int dispatch_g(int G, const CUtensorMap &tk, const CUtensorMap &tv, const PrefillArgs &a, dim3 grid,
               cudaStream_t st) {
  switch (G) {
    case 1: return launch_prefill<B, 1>(tk, tv, a, grid, st);
    case 2: return launch_prefill<B, 2>(tk, tv, a, grid, st);
    case 4: return launch_prefill<B, 4>(tk, tv, a, grid, st);
    case 8: return launch_prefill<B, 8>(tk, tv, a, grid, st);
    case 16: return launch_prefill<B, 16>(tk, tv, a, grid, st);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace

int prefill_launch(const pa_decode_desc *d, const void *q, const int32_t *cu_q, int max_q_len, int total_q,
                   const void *k_pool, const void *v_pool, const int32_t *block_tables, const int32_t *context_lens,
                   void *out, float *part_o, float *part_ml, int causal, int kparts, int kpart_len,
                   int32_t *err_flag, void *stream) {
  PrefillArgs a;
  dim3 grid;
  int st = prepare_prefill(d, q, cu_q, max_q_len, total_q, k_pool, v_pool, block_tables, context_lens, out, part_o,
                           part_ml, causal, kparts, kpart_len, err_flag, &a, &grid);
  if (st != PA_OK || grid.x == 0) return st;
  const uint64_t rows = (uint64_t)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tk, tv;
  if (!encode_2d_bf16(&tk, k_pool, rows, 128, d->block_size, 64, true) ||
      !encode_2d_bf16(&tv, v_pool, rows, 128, d->block_size, 64, true))
    return PA_ERR_CUDA;
  const int G = d->num_q_heads / d->num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d->block_size == 16 ? dispatch_g<16>(G, tk, tv, a, grid, s) : dispatch_g<32>(G, tk, tv, a, grid, s);
}

}  // namespace pa

extern "C" int pa_paged_attention_prefill_chunk(const pa_decode_desc *d, const void *q, const int32_t *cu_q,
                                                int max_q_len, int total_q, const void *k_pool,
                                                const void *v_pool, const int32_t *block_tables,
                                                const int32_t *context_lens, void *out, int32_t *err_flag,
                                                void *stream) {
  return pa::prefill_launch(d, q, cu_q, max_q_len, total_q, k_pool, v_pool, block_tables, context_lens, out,
                            nullptr, nullptr, 1, 1, 0, err_flag, stream);
}
