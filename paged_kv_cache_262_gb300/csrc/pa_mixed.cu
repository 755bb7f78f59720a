// One launch for the attention of a continuous-batching step on sm_103a: the
// causal chunked prefill of the step's prompt chunks and the decode of its
// generating sequences, side by side.
//
// "Configuring vLLM and PagedAttention for High Throughput Enterprise LLM
// Serving" ("High-Throughput Batching: Continuous Batching & Chunked
// Prefill"): a long prompt is cut into chunks that share each engine
// iteration with the decode tokens, so that prefill compute rides along with
// the memory-bound decode ("Memory Bottlenecks in Autoregressive LLM
// Inference").  On the GPU the two halves stress different units: the prefill
// tiles keep the tensor cores busy, the decode units stream the cache from
// HBM.  Run one after the other, each leaves the other's unit idle; here every
// CTA of one grid takes one role:
//  * a prefill CTA runs one pair of 128-row query tiles of one kv head of
//    one chunk, exactly the prefill kernel's CTA (pa_prefill_body.cuh);
//  * a decode CTA runs three independent decode units of four warps each
//    (one (sequence part, kv head) apiece, the decode kernel's CTA,
//    pa_decode_body.cuh), each with its own shared memory and named barrier;
//    three units in 205 KB match the prefill CTA's footprint, so an SM holds
//    either one prefill CTA or three decode units.
// The roles are interleaved evenly in dispatch order, so that both queues
// drain together and the HBM-bound and tensor-bound CTAs share the GPU for the
// whole step.  Results are those of pa_paged_attention_prefill_chunk and
// pa_paged_attention_decode with the same arguments, bit for bit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include "pa_decode_body.cuh"
#include "pa_internal.h"
#include "pa_prefill_body.cuh"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

constexpr int kUnitsPerCta = kThreads / 128;  // decode units (4 warps each) in one mixed-step CTA

template <int B>
struct MixedSmem {
  // 16-token pages: two ring slots a warp (three units must fit one CTA);
  // 32-token pages: one, as in the decode kernel.
  static constexpr int kDecodeStages = B == 16 ? 2 : 1;
  using L = DecodeSmem<128, B, 4, kDecodeStages>;
  static constexpr int kUnitStride = (L::kBytes + 1023) & ~1023;
  static constexpr int kDecodeBytes = kUnitsPerCta * kUnitStride + 1024;  // + alignment slack
  static constexpr int kBytes = kDecodeBytes > kSmem ? kDecodeBytes : kSmem;
  static_assert(kBytes <= 227 * 1024, "mixed-step shared memory over the per-CTA limit");
};

// Dispatch order of the two roles (PA_MIXED_ORDER: interleave, decode-first,
// prefill-first; the last two are for comparison).
enum MixedOrder { kInterleave = 0, kDecodeFirst = 1, kPrefillFirst = 2 };

struct MixedPlan {
  int n_prefill;     // prefill CTAs: gx * gy * gz
  int n_decode;      // decode CTAs: ceil(decode_units / kUnitsPerCta)
  int decode_units;  // sequences x kv heads x split parts
  int gx, gy;        // prefill grid (bx fastest), as the prefill kernel's
  int order;         // MixedOrder
};

template <int B, int G>
__global__ void __launch_bounds__(kThreads, 1)
    mixed_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmK3, const __grid_constant__ CUtensorMap tmV3,
                 const PrefillArgs pf, const DecodeArgs dc, const MixedPlan m) {
  // tmK / tmV: 64-column boxes (prefill tiles); tmK3 / tmV3: a page's two
  // halves in one copy (decode units)
  using M = MixedSmem<B>;
  constexpr int NT = G <= 8 ? 1 : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int b = blockIdx.x;
  int before;  // decode CTAs ahead of this one in dispatch order
  bool decode;
  if (m.order == kDecodeFirst) {
    decode = b < m.n_decode;
    before = min(b, m.n_decode);
  } else if (m.order == kPrefillFirst) {
    decode = b >= m.n_prefill;
    before = max(0, b - m.n_prefill);
  } else {  // CTA b is a decode CTA when the even spread of n_decode over the grid steps at b
    const long long n = (long long)m.n_prefill + m.n_decode;
    before = (int)((long long)b * m.n_decode / n);
    decode = (int)((long long)(b + 1) * m.n_decode / n) > before;
  }
  if (decode) {
    const int sub = threadIdx.x >> 7;
    const int lin = before * kUnitsPerCta + sub;
    if (lin < m.decode_units)
      decode_unit<128, B, NT, 4, M::kDecodeStages, false, false, false, true>(
          &tmK3, &tmV3, dc, lin, threadIdx.x & 127, smem + sub * M::kUnitStride, 1 + sub);
    return;
  }
  const int p = b - before;  // prefill CTA number, in the prefill kernel's launch order
  const int bx = p % m.gx, rest = p / m.gx;
  prefill_tile<B, G, false>(&tmK, &tmV, pf, bx, rest % m.gy, rest / m.gy, m.gx, smem);
}

template <int B, int G>
int launch_mixed(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk3, const CUtensorMap &tv3,
                 const PrefillArgs &pf, const DecodeArgs &dc, const MixedPlan &m, cudaStream_t st) {
  using M = MixedSmem<B>;
  auto kern = mixed_kernel<B, G>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, M::kBytes) != cudaSuccess)
    return PA_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PA_ERR_CUDA;
  if (fa.numRegs < kRegsLaunch) return PA_ERR_UNSUPPORTED;  // the prefill register split would not fit
  kern<<<m.n_prefill + m.n_decode, kThreads, M::kBytes, st>>>(tk, tv, tk3, tv3, pf, dc, m);
  return launch_status(cudaGetLastError());
}

template <int B>
int dispatch_mixed(int G, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk3, const CUtensorMap &tv3,
                   const PrefillArgs &pf, const DecodeArgs &dc, const MixedPlan &m, cudaStream_t st) {
  switch (G) {
    case 1: return launch_mixed<B, 1>(tk, tv, tk3, tv3, pf, dc, m, st);
    case 2: return launch_mixed<B, 2>(tk, tv, tk3, tv3, pf, dc, m, st);
    case 4: return launch_mixed<B, 4>(tk, tv, tk3, tv3, pf, dc, m, st);
    case 8: return launch_mixed<B, 8>(tk, tv, tk3, tv3, pf, dc, m, st);
    case 16: return launch_mixed<B, 16>(tk, tv, tk3, tv3, pf, dc, m, st);
    default: return PA_ERR_UNSUPPORTED;
  }
}

bool same_cache(const pa_decode_desc *a, const pa_decode_desc *b) {
  return a->num_q_heads == b->num_q_heads && a->num_kv_heads == b->num_kv_heads && a->head_dim == b->head_dim &&
         a->block_size == b->block_size && a->num_blocks == b->num_blocks;
}

}  // namespace
}  // namespace pa

extern "C" int pa_paged_attention_mixed(const pa_decode_desc *prefill_desc, const void *prefill_q,
                                        const int32_t *cu_q, int max_q_len, int total_q,
                                        const int32_t *prefill_tables, const int32_t *prefill_context_lens,
                                        void *prefill_out, const pa_decode_desc *decode_desc, const void *decode_q,
                                        const int32_t *decode_tables, const int32_t *decode_context_lens,
                                        void *decode_out, void *workspace, size_t workspace_bytes,
                                        const void *k_pool, const void *v_pool, int32_t *err_flag, void *stream) {
  using namespace pa;
  if (!prefill_desc || !decode_desc) return PA_ERR_INVALID;
  int st = validate_decode_desc(decode_desc);
  if (st != PA_OK) return st;
  if (!same_cache(prefill_desc, decode_desc)) return PA_ERR_INVALID;
  PrefillArgs pf{};
  dim3 pgrid;
  st = prepare_prefill(prefill_desc, prefill_q, cu_q, max_q_len, total_q, k_pool, v_pool, prefill_tables,
                       prefill_context_lens, prefill_out, nullptr, nullptr, 1, 1, 0, err_flag, &pf, &pgrid);
  if (st != PA_OK) return st;
  const pa_decode_desc *d = decode_desc;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  DecodePlan plan{};
  DecodeArgs dc{};
  long long units = 0;
  if (d->num_seqs > 0) {
    if (!decode_q || !decode_tables || !decode_context_lens || !decode_out || !k_pool || !v_pool)
      return PA_ERR_INVALID;
    if (!aligned16(decode_q) || !aligned16(decode_out) || !aligned16(k_pool) || !aligned16(v_pool))
      return PA_ERR_INVALID;
    plan = make_decode_plan(d, sms);
    if (plan.total() > 0 && (!workspace || workspace_bytes < plan.total() || !aligned16(workspace)))
      return PA_ERR_WORKSPACE;
    fill_decode_args(&dc, d, plan, decode_q, decode_tables, decode_context_lens, decode_out, workspace, err_flag,
                     (long long)sms * kUnitsPerCta);
    units = (long long)d->num_seqs * d->num_kv_heads * plan.max_parts;
  }
  const long long n_prefill = (long long)pgrid.x * pgrid.y * pgrid.z;
  const long long n_decode = (units + kUnitsPerCta - 1) / kUnitsPerCta;
  if (n_prefill + n_decode == 0) return PA_OK;
  if (n_prefill + n_decode > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  MixedPlan m;
  m.n_prefill = (int)n_prefill;
  m.n_decode = (int)n_decode;
  m.decode_units = (int)units;
  m.gx = pgrid.x ? (int)pgrid.x : 1;
  m.gy = pgrid.y ? (int)pgrid.y : 1;
  m.order = kInterleave;
  const char *env = getenv("PA_MIXED_ORDER");
  if (env && !strcmp(env, "decode-first")) m.order = kDecodeFirst;
  if (env && !strcmp(env, "prefill-first")) m.order = kPrefillFirst;
  const uint64_t rows = (uint64_t)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tk, tv, tk3, tv3;
  if (!encode_2d_bf16(&tk, k_pool, rows, 128, d->block_size, 64, true) ||
      !encode_2d_bf16(&tv, v_pool, rows, 128, d->block_size, 64, true) ||
      !encode_kv_halves_3d(&tk3, k_pool, rows, d->block_size) || !encode_kv_halves_3d(&tv3, v_pool, rows, d->block_size))
    return PA_ERR_CUDA;
  const int G = d->num_q_heads / d->num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d->block_size == 16 ? dispatch_mixed<16>(G, tk, tv, tk3, tv3, pf, dc, m, s)
                             : dispatch_mixed<32>(G, tk, tv, tk3, tv3, pf, dc, m, s);
}
