// Decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin inside a host
// framework that owns every device byte, a real-time path where cudaMalloc's
// implicit synchronisation is not allowed, or an embedded set-up whose memory
// is fixed at start-up.  For them this file keeps the split-K scratch of the
// decode kernel in a fixed, file-scope device array instead of a caller
// buffer.  The array lives on every GPU that loads this library until the
// process exits.
//
// The call allocates nothing: it resolves the array's device address once per
// device and hands it to the ordinary decode launcher as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

// Scratch of the allocation-free decode (PA_NOALLOC_SCRATCH_BYTES).  Device
// code could name it directly; host code must use the address returned by
// cudaGetSymbolAddress -- the host-side symbol is only a stand-in.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, resolved once
// per device (with that device current) and cached.
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_paged_attention_decode_noalloc(const pa_decode_desc *desc, const void *q,
                                                 const void *k_pool, const void *v_pool,
                                                 const int32_t *block_tables,
                                                 const int32_t *context_lens, void *out,
                                                 int32_t *err_flag, void *stream) {
  int st = pa::validate_decode_desc(desc);
  if (st != PA_OK) return st;
  if (desc->num_seqs == 0) return PA_OK;
  const int sms = pa::current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  if (pa::make_decode_plan(desc, sms).total() > (size_t)PA_NOALLOC_SCRATCH_BYTES)
    return PA_ERR_WORKSPACE;  // this shape needs more split-K scratch than the fixed array
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  return pa_paged_attention_decode(desc, q, k_pool, v_pool, block_tables, context_lens, out, scratch,
                                   (size_t)PA_NOALLOC_SCRATCH_BYTES, err_flag, stream);
}
