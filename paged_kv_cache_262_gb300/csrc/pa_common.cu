// Common host code of libpagedattn: version, status strings, device-attribute
// cache, tensor-map encoding through the driver entry point, and the decode
// split-K plan.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace pa {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < kMaxDevices) {
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool encode_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_kv_halves_3d(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, 2};
  cuuint64_t strides[2] = {256, 128};  // a row, a 64-column half (bytes)
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int validate_decode_desc(const pa_decode_desc *d) {
  if (!d) return PA_ERR_INVALID;
  if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_blocks <= 0 ||
      d->max_blocks_per_seq <= 0 || d->max_context_len < 0)
    return PA_ERR_INVALID;
  if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_INVALID;
  if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (d->block_size != 16 && d->block_size != 32) return PA_ERR_UNSUPPORTED;
  if (d->num_q_heads / d->num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  // TMA row coordinates are int32: every (block, head, token) row must fit.
  if ((int64_t)d->num_blocks * d->num_kv_heads * d->block_size >= ((int64_t)1 << 31))
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)d->max_blocks_per_seq * d->block_size >= ((int64_t)1 << 31)) return PA_ERR_INVALID;
  // Longest supported context: kMaxParts parts of kMaxPartPages pages.
  if (((int64_t)d->max_context_len + d->block_size - 1) / d->block_size >
      (int64_t)kMaxParts * kMaxPartPages)
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// A new nonzero tag for the split-K arrival counters of one decode launch.
unsigned int next_decode_epoch() {
  static std::atomic<unsigned int> counter{0};
  unsigned int e;
  do {
    e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  } while (e == 0);
  return e;
}

// Split policy.  Each CTA streams one part (part_pages pages of one
// (sequence, kv head)); two CTAs (16-token pages) or three (32-token pages)
// are resident per SM.  The host knows only the longest-context bound, so it
// plans for every unit at that length.  A context longer than kMaxPartPages
// pages is always cut.  When the units leave room, each is cut into as many
// equal parts as fit one wave of the resident slots: the CTAs all start at
// once, stream equal shares and end together (8 x 32768 tokens, GQA 8:
// four 512-page parts, 256 CTAs, 166.0 us, against 168.3-169.7 us for
// eight parts in 1.7 waves; a thin last wave leaves HBM idle: 320 CTAs on
// 304 slots 218 us, 384 CTAs 190 us).  With more units than that, parts are
// sized for about 1.5 CTAs per resident slot (ragged batches then start
// longest context first).  Parts never go below kMinPartPages pages unless
// the context is shorter.  PA_PARTITION_PAGES in the environment overrides
// the part length (tuning).
DecodePlan make_decode_plan(const pa_decode_desc *d, int sm_count) {
  const int kCtasPerSm = d->block_size == 16 ? 2 : 3;  // resident decode CTAs per SM (shared memory)
  constexpr int kMinPartPages = 32;
  DecodePlan p;
  const int B = d->block_size;
  const int64_t max_pages = std::max<int64_t>(1, ((int64_t)d->max_context_len + B - 1) / B);
  const int64_t units = std::max<int64_t>(1, (int64_t)d->num_seqs * d->num_kv_heads);
  int64_t pp;
  const char *env = getenv("PA_PARTITION_PAGES");
  if (env && atoi(env) > 0) {
    pp = atoi(env);
  } else {
    const int64_t slots = (int64_t)std::max(sm_count, 1) * kCtasPerSm;
    const int64_t least = (max_pages + kMaxPartPages - 1) / kMaxPartPages;  // parts of <= kMaxPartPages pages
    const int64_t most = std::min<int64_t>(kMaxParts, std::max<int64_t>(1, max_pages / kMinPartPages));
    if (units * least <= slots) {
      const int64_t np = std::max(least, std::min(slots / units, most));
      pp = (max_pages + np - 1) / np;
    } else {
      pp = (units * max_pages * 2 + slots * 3 - 1) / (slots * 3);
      pp = std::max<int64_t>(pp, kMinPartPages);
    }
  }
  pp = std::max<int64_t>(pp, (max_pages + kMaxParts - 1) / kMaxParts);
  pp = std::min<int64_t>(pp, kMaxPartPages);
  pp = std::min<int64_t>(pp, max_pages);
  pp = std::max<int64_t>(pp, 1);
  p.part_pages = (int)pp;
  p.max_parts = (int)((max_pages + pp - 1) / pp);
  if (p.max_parts > 1 && d->num_seqs > 0) {
    const size_t G = d->num_q_heads / d->num_kv_heads;
    const size_t n = (size_t)d->num_seqs * d->num_kv_heads * p.max_parts * G;
    auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
    p.ws_o_bytes = up(n * d->head_dim * sizeof(float));
    p.ws_ml_bytes = up(n * 2 * sizeof(float));
    p.ws_cnt_bytes = up((size_t)d->num_seqs * d->num_kv_heads * sizeof(unsigned long long));
  }
  return p;
}

}  // namespace pa

extern "C" {

const char *pa_version(void) { return "libpagedattn 0.1.0 (sm_103a)"; }

const char *pa_status_string(int s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_OOM: return "out of blocks or host memory";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_STATE: return "bad block-manager state";
    default: return "unknown status";
  }
}

size_t pa_decode_workspace_bytes(const pa_decode_desc *desc) {
  if (pa::validate_decode_desc(desc) != PA_OK) return 0;
  return pa::make_decode_plan(desc, pa::current_sm_count()).total();
}

}  // extern "C"
