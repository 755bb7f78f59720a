"""libpagedattn: paged KV-cache attention for GB300 (sm_103a).

The product is the C-ABI shared library declared in ``include/pagedattn.h``;
this package holds its CUDA/C++ sources (``csrc/``), the in-tree build
(``build.py``) and a thin ctypes binding with the same call names.
"""
from ._binding import (  # noqa: F401
    DEVERR_CTX, DEVERR_PAGE, DEVERR_PAIR, DEVERR_SLOT, DEVERR_TIMEOUT, EXPORTS, PA_ERR_CUDA,
    PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_STATE, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_OK,
    NOALLOC_SCRATCH_BYTES, BlockManager, DecodeDesc, PaError, copy_blocks, decode_workspace, decode_workspace_bytes,
    hbm_probe, load, selftest_bounded_wait,
    make_desc, paged_attention_decode, paged_attention_decode_append, paged_attention_decode_noalloc, paged_attention_decode_shared_prefix, paged_attention_mixed, paged_attention_prefill_chunk, reshape_and_cache,
    status_string, swap_blocks, version)
