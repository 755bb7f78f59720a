// Cache writes of libpagedattn: reshape_and_cache (new tokens' K/V into their
// slots) and copy_blocks (copy-on-write page copies).  Both are bit-exact
// 16-byte vector copies; both are HBM/launch bound.
//
// reshape_and_cache follows "Configuring vLLM and PagedAttention for High
// Throughput Enterprise LLM Serving" ("Architectural Foundations": pages are
// allocated on demand from a global pool and addressed through the block
// table; "Memory Bottlenecks": K/V are produced for every token position).
// copy_blocks follows "vLLM Guide: High-Throughput Multi-GPU LLM Serving with
// PagedAttention" ("What Is PagedAttention?": shared blocks with copy-on-write)
// and the ref_count column of the block-table example in "vLLM
// High-Performance Inference Engine: PagedAttention Principles and Deployment
// Guide" ("PagedAttention Architecture Deep Dive").  swap_blocks moves whole
// blocks between HBM and pinned host memory for preemptive swapping
// ("Configuring vLLM and PagedAttention ...", question on KV cache offloading:
// the least recently started request's pages go to host RAM and come back
// later); on Grace-Blackwell the kernel reads and writes the pinned host pool
// directly over the chip-to-chip link.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pa_internal.h"
#include "pagedattn.h"

namespace pa {
namespace {

// One thread per 16-byte chunk of one (token, kv head) row, K and V together.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             uint4 *__restrict__ kp, uint4 *__restrict__ vp,
                             const int64_t *__restrict__ slots, int64_t total, int hc, int C, int B,
                             int64_t nslots, int32_t *err) {
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / hc;
    const int rem = (int)(idx - t * hc);
    const int h = rem / C, c = rem - h * C;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= nslots) {
      if (err && rem == 0) atomicOr(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / B, off = slot - blk * B;
    const int64_t H = hc / C;
    const int64_t dst = ((blk * H + h) * B + off) * C + c;
    const uint4 kv = __ldg(k + idx);
    const uint4 vv = __ldg(v + idx);
    kp[dst] = kv;
    vp[dst] = vv;
  }
}

constexpr int kCopyLayers = 128;  // layers per launch (kernel-parameter space)

struct CopyPtrs {
  uint4 *k[kCopyLayers];
  uint4 *v[kCopyLayers];
};

// grid (pair, layer, K|V); each CTA copies one block of one pool.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const __grid_constant__ CopyPtrs ptrs, const int64_t *__restrict__ pairs,
                       int num_blocks, int64_t chunks, int32_t *err) {
  const int pair = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
  const int64_t src = __ldg(pairs + 2 * (int64_t)pair), dst = __ldg(pairs + 2 * (int64_t)pair + 1);
  if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
    if (err && threadIdx.x == 0 && layer == 0 && which == 0) atomicOr(err, PA_DEVERR_PAIR);
    return;
  }
  uint4 *base = which ? ptrs.v[layer] : ptrs.k[layer];
  const uint4 *__restrict__ s = base + src * chunks;
  uint4 *__restrict__ d = base + dst * chunks;
  constexpr int U = 4;
  int64_t i = threadIdx.x;
  for (; i + (U - 1) * 256 < chunks; i += U * 256) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = __ldcs(s + i + u * 256);
#pragma unroll
    for (int u = 0; u < U; ++u) __stcs(d + i + u * 256, r[u]);
  }
  for (; i < chunks; i += 256) __stcs(d + i, __ldcs(s + i));
}

constexpr int kSwapLayers = 64;  // layers per launch (kernel-parameter space)

struct SwapPtrs {
  const uint4 *src_k[kSwapLayers];
  const uint4 *src_v[kSwapLayers];
  uint4 *dst_k[kSwapLayers];
  uint4 *dst_v[kSwapLayers];
};

// grid (pair, layer, K|V); each CTA moves one block from the source pool to
// the destination pool (either may be pinned host memory addressed by the GPU).
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(const __grid_constant__ SwapPtrs ptrs, const int64_t *__restrict__ pairs, int src_blocks,
                       int dst_blocks, int64_t chunks, int32_t *err) {
  const int pair = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
  const int64_t src = __ldg(pairs + 2 * (int64_t)pair), dst = __ldg(pairs + 2 * (int64_t)pair + 1);
  if (src < 0 || dst < 0 || src >= src_blocks || dst >= dst_blocks) {
    if (err && threadIdx.x == 0 && layer == 0 && which == 0) atomicOr(err, PA_DEVERR_PAIR);
    return;
  }
  const uint4 *__restrict__ s = (which ? ptrs.src_v[layer] : ptrs.src_k[layer]) + src * chunks;
  uint4 *__restrict__ d = (which ? ptrs.dst_v[layer] : ptrs.dst_k[layer]) + dst * chunks;
  constexpr int U = 4;
  int64_t i = threadIdx.x;
  for (; i + (U - 1) * 256 < chunks; i += U * 256) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = __ldcs(s + i + u * 256);
#pragma unroll
    for (int u = 0; u < U; ++u) __stcs(d + i + u * 256, r[u]);
  }
  for (; i < chunks; i += 256) __stcs(d + i, __ldcs(s + i));
}

}  // namespace
}  // namespace pa

extern "C" int pa_swap_blocks(void *const *src_k_pools, void *const *src_v_pools, void *const *dst_k_pools,
                              void *const *dst_v_pools, int num_layers, const int64_t *block_pairs, int num_pairs,
                              int src_num_blocks, int dst_num_blocks, size_t block_bytes, int32_t *err_flag,
                              void *stream) {
  using namespace pa;
  if (num_layers <= 0 || num_layers > 256 || num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 ||
      block_bytes == 0 || block_bytes % 16 != 0)
    return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!src_k_pools || !src_v_pools || !dst_k_pools || !dst_v_pools || !block_pairs) return PA_ERR_INVALID;
  for (int l = 0; l < num_layers; ++l)
    if (!src_k_pools[l] || !src_v_pools[l] || !dst_k_pools[l] || !dst_v_pools[l] || !aligned16(src_k_pools[l]) ||
        !aligned16(src_v_pools[l]) || !aligned16(dst_k_pools[l]) || !aligned16(dst_v_pools[l]))
      return PA_ERR_INVALID;
  for (int l0 = 0; l0 < num_layers; l0 += kSwapLayers) {
    const int nl = std::min(kSwapLayers, num_layers - l0);
    SwapPtrs p{};
    for (int l = 0; l < nl; ++l) {
      p.src_k[l] = static_cast<const uint4 *>(src_k_pools[l0 + l]);
      p.src_v[l] = static_cast<const uint4 *>(src_v_pools[l0 + l]);
      p.dst_k[l] = static_cast<uint4 *>(dst_k_pools[l0 + l]);
      p.dst_v[l] = static_cast<uint4 *>(dst_v_pools[l0 + l]);
    }
    swap_blocks_kernel<<<dim3(num_pairs, nl, 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        p, block_pairs, src_num_blocks, dst_num_blocks, (int64_t)(block_bytes / 16), err_flag);
    const int st = launch_status(cudaGetLastError());
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

extern "C" int pa_reshape_and_cache(const void *k, const void *v, void *k_pool, void *v_pool,
                                    const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                    int head_dim, int block_size, int num_blocks, int32_t *err_flag,
                                    void *stream) {
  using namespace pa;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID;
  if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID;
  const int C = head_dim / 8;
  const int hc = num_kv_heads * C;
  const int64_t total = (int64_t)num_tokens * hc;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const int64_t want = (total + 255) / 256;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 16));
  reshape_and_cache_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), static_cast<uint4 *>(k_pool),
      static_cast<uint4 *>(v_pool), slot_mapping, total, hc, C, block_size,
      (int64_t)num_blocks * block_size, err_flag);
  return launch_status(cudaGetLastError());
}

extern "C" int pa_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                              const int64_t *block_pairs, int num_pairs, int num_blocks,
                              size_t block_bytes, int32_t *err_flag, void *stream) {
  using namespace pa;
  if (num_layers <= 0 || num_layers > 256 || num_pairs < 0 || num_blocks <= 0 || block_bytes == 0)
    return PA_ERR_INVALID;
  if (block_bytes % 16 != 0) return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!k_pools || !v_pools || !block_pairs) return PA_ERR_INVALID;
  if (num_pairs > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  for (int l = 0; l < num_layers; ++l)
    if (!k_pools[l] || !v_pools[l] || !aligned16(k_pools[l]) || !aligned16(v_pools[l]))
      return PA_ERR_INVALID;
  for (int l0 = 0; l0 < num_layers; l0 += kCopyLayers) {
    const int nl = std::min(kCopyLayers, num_layers - l0);
    CopyPtrs p{};
    for (int l = 0; l < nl; ++l) {
      p.k[l] = static_cast<uint4 *>(k_pools[l0 + l]);
      p.v[l] = static_cast<uint4 *>(v_pools[l0 + l]);
    }
    copy_blocks_kernel<<<dim3(num_pairs, nl, 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        p, block_pairs, num_blocks, (int64_t)(block_bytes / 16), err_flag);
    const int st = launch_status(cudaGetLastError());
    if (st != PA_OK) return st;
  }
  return PA_OK;
}
