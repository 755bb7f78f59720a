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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

// Scratch of the allocation-free decode (PA_NOALLOC_SCRATCH_BYTES).  Device
// code could name it directly; host code must use the address returned by
// cudaGetSymbolAddress -- the host-side symbol is only a stand-in.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct Cached {
  unsigned long long ctx_id;  // the context the address belongs to (0: none yet)
  void *ptr;
};
Cached g_scratch[kMaxDevices];

// Id of the calling thread's current context, unique over the process's
// lifetime (a context created after cudaDeviceReset gets a new one); 0 when
// there is no current context.  The driver calls come through the runtime's
// entry-point query, so the library links no driver library.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array on the current device.  It is looked
// up (with that device current) on the first call and again whenever the
// device's context has changed since -- after cudaDeviceReset the module is
// loaded anew and the array may sit elsewhere.
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  const unsigned long long id = current_ctx_id();
  if (id == 0 || g_scratch[dev].ctx_id != id || !g_scratch[dev].ptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    g_scratch[dev] = Cached{current_ctx_id(), p};  // the lookup made the context current if it was not
  }
  *out = g_scratch[dev].ptr;
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
