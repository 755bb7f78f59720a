"""The allocation-free decode entry point, for callers that cannot allocate
device memory (their framework owns all of it, or cudaMalloc's implicit
synchronisation is not allowed where they run).  It keeps the split-K scratch
in a fixed device array instead of a caller workspace.

Called through the C ABI and compared with the ordinary entry point (which
takes a workspace) on the same inputs, twice in a row: the fixed array keeps
the previous call's contents, and the second call must not be disturbed by
them.  This file is collected last so that a failure here comes after every
other test has run."""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_host, need_gpu, upload_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def test_noalloc_matches_workspace_entry_point_twice(torch):
    case = wl.make_decode_case("noalloc", [6000, 9000, 3000, 12000], 32, 8, 128, 16, seed=12,
                               with_new_tokens=False)
    d = upload_case(case, torch)
    lib = pa.load()
    desc = pa.make_desc(d["q"], d["k_pool"], d["bt"], scale=case.scale, max_context_len=case.max_context_len)
    need = pa.decode_workspace_bytes(desc)
    assert 0 < need <= pa.NOALLOC_SCRATCH_BYTES  # this shape splits, so the scratch is used
    ref = bf16_host(pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"],
                                              scale=case.scale, max_context_len=case.max_context_len))
    stream = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(d["q"], float("nan"))
        st = lib.pa_paged_attention_decode_noalloc(ctypes.byref(desc), d["q"].data_ptr(), d["k_pool"].data_ptr(),
                                                   d["v_pool"].data_ptr(), d["bt"].data_ptr(), d["ctx"].data_ptr(),
                                                   out.data_ptr(), err.data_ptr(), stream)
        assert st == pa.PA_OK, pa.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(bf16_host(out), np.asarray((ref.astype(np.uint32) << 16).view(np.float32), np.float64),
                     f"noalloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch(torch):
    lib = pa.load()
    desc = pa.DecodeDesc(num_seqs=512, num_q_heads=128, num_kv_heads=8, head_dim=128, block_size=16,
                         num_blocks=1000, max_blocks_per_seq=4096, max_context_len=65536, scale=0.1)
    assert pa.decode_workspace_bytes(desc) > pa.NOALLOC_SCRATCH_BYTES
    st = lib.pa_paged_attention_decode_noalloc(ctypes.byref(desc), 16, 16, 16, 16, 16, 16, None, None)
    assert st == pa.PA_ERR_WORKSPACE
