// Diagnostics of libpagedattn: the HBM bandwidth probe that the decode
// kernels' roofline is read against, and a self-test of the bounded on-chip
// wait that every kernel of the library relies on.
//
// Decode is a read stream: "Configuring vLLM and PagedAttention for High
// Throughput Enterprise LLM Serving" ("Memory Bottlenecks in Autoregressive
// LLM Inference") has each new token read every cached key and value from
// HBM.  A copy benchmark (read + write) pays for the DRAM's read/write
// turnarounds, which a read stream does not, so the probe measures both: a
// read-only stream of 16-byte vector loads and a 16-byte vector copy.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 8;     // independent 16-byte loads in flight per thread
constexpr int kProbeCtasPerSm = 8;  // 2048 threads per SM

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Reads n 16-byte words.  The loads feed an XOR that is stored only when it
// equals `never` (with random data, never), so nothing is written yet no load
// can be dropped.
__global__ void __launch_bounds__(kProbeThreads) hbm_read_kernel(const uint4 *__restrict__ src, size_t n,
                                                                 uint4 *sink, uint32_t never) {
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kProbeUnroll - 1) * stride < n; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n; i += stride) {
    const uint4 v = ld_stream(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == never) *sink = make_uint4(acc, blockIdx.x, threadIdx.x, 0u);
}

// dst := src, n 16-byte words.
__global__ void __launch_bounds__(kProbeThreads) hbm_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                                 size_t n) {
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
  for (; i + (kProbeUnroll - 1) * stride < n; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < n; i += stride) __stcs(dst + i, ld_stream(src + i));
}

// Reads n_bytes through the TMA engine: bulk copies (cp.async.bulk) of
// kBulkChunk bytes from global into a ring of kBulkSlots shared-memory slots,
// the path the decode kernels' page gathers take.  Chunk c goes to CTA
// c mod gridDim.x; one thread issues, reusing a slot once its copy has landed.
constexpr int kBulkChunk = 16384;
constexpr int kBulkSlots = 8;
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__global__ void __launch_bounds__(32) hbm_bulk_read_kernel(const uint8_t *__restrict__ src, size_t n_bytes,
                                                           int32_t *err) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t bars[kBulkSlots];
  if (threadIdx.x != 0) return;
  for (int i = 0; i < kBulkSlots; ++i) mbar_init(&bars[i], 1);
  fence_mbar_init();
  const size_t nchunks = (n_bytes + kBulkChunk - 1) / kBulkChunk;
  long long k = 0;  // this CTA's copies issued so far
  for (size_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++k) {
    const int slot = (int)(k % kBulkSlots);
    if (k >= kBulkSlots && !mbar_wait(&bars[slot], (uint32_t)(((k / kBulkSlots) - 1) & 1))) {
      if (err) atomicOr(err, PA_DEVERR_TIMEOUT);
      break;  // the copies still in flight are waited for below
    }
    const size_t off = c * kBulkChunk;
    const uint32_t bytes = (uint32_t)(n_bytes - off < (size_t)kBulkChunk ? n_bytes - off : (size_t)kBulkChunk);
    mbar_arrive_expect_tx(&bars[slot], bytes);
    bulk_load(ring + slot * kBulkChunk, src + off, bytes, &bars[slot]);
  }
  // the last use of every slot: its copy must land before the CTA exits
  for (long long j = k - kBulkSlots < 0 ? 0 : k - kBulkSlots; j < k; ++j)
    if (!mbar_wait(&bars[j % kBulkSlots], (uint32_t)((j / kBulkSlots) & 1)) && err) atomicOr(err, PA_DEVERR_TIMEOUT);
}

// Reads like paged decode: K and V runs of 4 KB (one (block, kv head) of 16
// tokens x 128 bf16) at scattered places, with the decode kernel's
// concurrency -- 2 CTAs per SM, 4 warps each, every warp a ring of three 8 KB
// slots (a K run and a V run).  The buffer's first half holds the K runs, the
// second the V runs; run i of a warp's stream is at (i * 0x9E3779B1) mod the
// number of runs in a half (a power of two: a permutation), so consecutive
// reads land far apart as a block table's scattered pages do.
constexpr int kGatherRun = 4096;
constexpr int kGatherSlots = 3;
__global__ void __launch_bounds__(128) hbm_gather_kernel(const uint8_t *__restrict__ src, uint32_t runs_log2,
                                                         int per_warp, int32_t *err) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t bars[4 * kGatherSlots];
  uint8_t *ring = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t *mb = bars + warp * kGatherSlots;
  uint8_t *slots = ring + warp * kGatherSlots * 2 * kGatherRun;
  if (lane == 0) {
    for (int i = 0; i < kGatherSlots; ++i) mbar_init(&mb[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t mask = (1u << runs_log2) - 1u;
  const size_t half = (size_t)kGatherRun << runs_log2;
  const uint32_t base = (uint32_t)(blockIdx.x * 4 + warp) * (uint32_t)per_warp;
  auto issue = [&](int i) {
    const size_t r = (size_t)(((base + (uint32_t)i) * 0x9E3779B1u) & mask) * kGatherRun;
    uint64_t *b = &mb[i % kGatherSlots];
    uint8_t *d = slots + (i % kGatherSlots) * 2 * kGatherRun;
    mbar_arrive_expect_tx(b, 2 * kGatherRun);
    bulk_load(d, src + r, kGatherRun, b);
    bulk_load(d + kGatherRun, src + half + r, kGatherRun, b);
  };
  if (lane == 0)
    for (int i = 0; i < kGatherSlots && i < per_warp; ++i) issue(i);
  int i = 0;
  for (; i < per_warp; ++i) {
    if (!__all_sync(0xffffffffu, mbar_wait(&mb[i % kGatherSlots], (uint32_t)((i / kGatherSlots) & 1)))) {
      if (lane == 0 && err) atomicOr(err, PA_DEVERR_TIMEOUT);
      break;
    }
    if (lane == 0 && i + kGatherSlots < per_warp) issue(i + kGatherSlots);
  }
  for (int k = i + 1; k < per_warp && k < i + kGatherSlots; ++k)  // after a timeout: copies in flight land
    mbar_wait(&mb[k % kGatherSlots], (uint32_t)((k / kGatherSlots) & 1));
}

// One warp waits, as every streaming warp of the decode kernel does, on an
// mbarrier that nothing arrives on; the wait gives up after limit_cycles and
// the kernel reports PA_DEVERR_TIMEOUT, then returns.  *done is set last, so
// the host can tell the kernel ran to its end.
__global__ void __launch_bounds__(32) bounded_wait_kernel(long long limit_cycles, int32_t *err, int32_t *done) {
  __shared__ uint64_t bar;
  const int lane = threadIdx.x;
  if (lane == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_limit(&bar, 0u, limit_cycles));
  if (!ok && lane == 0 && err) atomicOr(err, PA_DEVERR_TIMEOUT);
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    *done = 1;
  }
}

}  // namespace
}  // namespace pa

extern "C" int pa_hbm_probe(const void *src, void *dst, size_t bytes, int mode, void *sink, int32_t *err_flag,
                            void *stream) {
  using namespace pa;
  if (!src || bytes == 0 || (bytes & 15) || !aligned16(src)) return PA_ERR_INVALID;
  if (mode < 0 || mode > 3) return PA_ERR_INVALID;
  if (mode == 0 && (!sink || !aligned16(sink))) return PA_ERR_INVALID;
  if (mode == 1 && (!dst || !aligned16(dst))) return PA_ERR_INVALID;
  // mode 3: the largest power-of-two number of 4 KB runs that fits each half of the buffer
  uint32_t lg = 0;
  while (lg < 30 && ((size_t)kGatherRun << (lg + 1)) * 2 <= bytes) ++lg;
  if (mode == 3 && ((size_t)kGatherRun << lg) * 2 > bytes) return PA_ERR_INVALID;
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const size_t n = bytes / 16;
  const size_t want = (n + kProbeThreads - 1) / kProbeThreads;
  const unsigned grid = (unsigned)(want < (size_t)sms * kProbeCtasPerSm ? want : (size_t)sms * kProbeCtasPerSm);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mode == 2) {
    constexpr int kRing = kBulkSlots * kBulkChunk;
    if (cudaFuncSetAttribute(hbm_bulk_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRing) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    const size_t chunks = (bytes + kBulkChunk - 1) / kBulkChunk;
    const unsigned g = (unsigned)(chunks < (size_t)sms ? chunks : (size_t)sms);  // one CTA (its ring) per SM
    hbm_bulk_read_kernel<<<g, 32, kRing, st>>>(static_cast<const uint8_t *>(src), bytes, err_flag);
    return launch_status(cudaGetLastError());
  }
  if (mode == 3) {
    const int ctas = 2 * sms;
    const size_t runs = (size_t)1 << lg;
    const int per_warp = (int)(runs / ((size_t)ctas * 4) > 0 ? runs / ((size_t)ctas * 4) : 1);
    constexpr int kRingBytes = 4 * kGatherSlots * 2 * kGatherRun + 1024;
    if (cudaFuncSetAttribute(hbm_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    hbm_gather_kernel<<<ctas, 128, kRingBytes, st>>>(static_cast<const uint8_t *>(src), lg, per_warp, err_flag);
    return launch_status(cudaGetLastError());
  }
  if (mode == 0)
    hbm_read_kernel<<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4 *>(src), n, static_cast<uint4 *>(sink),
                                                    0x9e3779b9u);
  else
    hbm_copy_kernel<<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n);
  return launch_status(cudaGetLastError());
}

extern "C" int pa_selftest_bounded_wait(long long limit_cycles, int32_t *err_flag, int32_t *done, void *stream) {
  using namespace pa;
  if (limit_cycles < 1 || limit_cycles > kWaitLimitCycles || !done) return PA_ERR_INVALID;
  pa::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, err_flag, done);
  return launch_status(cudaGetLastError());
}
