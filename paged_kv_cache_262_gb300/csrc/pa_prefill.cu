// Causal chunked-prefill attention (tcgen05) -- not yet built: the entry point
// validates nothing and reports PA_ERR_UNSUPPORTED.
#include "pagedattn.h"

extern "C" int pa_paged_attention_prefill_chunk(const pa_decode_desc *, const void *, const int32_t *,
                                                int, const void *, const void *, const int32_t *,
                                                const int32_t *, void *, int32_t *, void *) {
  return PA_ERR_UNSUPPORTED;
}
