"""The allocation-free decode entry point, for callers that cannot allocate
device memory (their framework owns all of it, or cudaMalloc's implicit
synchronisation is not allowed where they run).  It keeps the split-K scratch
in a fixed device array instead of a caller workspace.

Called through the C ABI.  It runs the same kernel with the same split plan as
the ordinary entry point (which takes a workspace), so its output must be
bit-identical to that entry point's; it is also checked once against the fp64
oracle.  The fixed array keeps each call's contents, so the calls come in a
row: the first shape, then a shape cut into many short parts (its partial
results land where the first shape's arrival counters were), then the first
shape again.  This file is collected last so that a failure here comes after
every other test has run."""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_host, need_gpu, oracle_rows, upload_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _noalloc(torch, lib, case, d):
    desc = pa.make_desc(d["q"], d["k_pool"], d["bt"], scale=case.scale, max_context_len=case.max_context_len)
    stream = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    st = lib.pa_paged_attention_decode_noalloc(ctypes.byref(desc), d["q"].data_ptr(), d["k_pool"].data_ptr(),
                                               d["v_pool"].data_ptr(), d["bt"].data_ptr(), d["ctx"].data_ptr(),
                                               out.data_ptr(), err.data_ptr(), stream)
    assert st == pa.PA_OK, pa.status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return bf16_host(out)


def _with_workspace(torch, case, d):
    out = pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"], scale=case.scale,
                                    max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    return bf16_host(out)


def test_noalloc_bit_identical_to_workspace_entry_point(torch, ora, monkeypatch):
    lib = pa.load()
    monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    first = wl.make_decode_case("noalloc", [6000, 9000, 3000, 12000], 32, 8, 128, 16, seed=12,
                                with_new_tokens=False)
    d1 = upload_case(first, torch)
    need1 = pa.decode_workspace_bytes(pa.make_desc(d1["q"], d1["k_pool"], d1["bt"],
                                                   max_context_len=first.max_context_len))
    assert 0 < need1 <= pa.NOALLOC_SCRATCH_BYTES  # this shape splits, so the scratch is used
    want1 = _with_workspace(torch, first, d1)

    got = _noalloc(torch, lib, first, d1)
    assert np.array_equal(got, want1), "noalloc call 1 differs from the workspace entry point"
    assert_close(got, oracle_rows(ora, first).reshape(got.shape), "noalloc call 1 against the oracle")

    # another shape cut into 3-page parts: more parts, a larger layout over the array
    monkeypatch.setenv("PA_PARTITION_PAGES", "3")
    second = wl.make_decode_case("noalloc2", [5000, 1, 2999], 16, 4, 128, 16, seed=13, with_new_tokens=False)
    d2 = upload_case(second, torch)
    need2 = pa.decode_workspace_bytes(pa.make_desc(d2["q"], d2["k_pool"], d2["bt"],
                                                   max_context_len=second.max_context_len))
    assert 2 * need1 < need2 <= pa.NOALLOC_SCRATCH_BYTES  # its partial results cover the first layout
    want2 = _with_workspace(torch, second, d2)
    got = _noalloc(torch, lib, second, d2)
    assert np.array_equal(got, want2), "noalloc call 2 differs from the workspace entry point"

    # the first shape again, over the second call's leftovers
    monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    got = _noalloc(torch, lib, first, d1)
    assert np.array_equal(got, want1), "noalloc call 3 differs from the workspace entry point"


def test_noalloc_rejects_shapes_beyond_its_scratch(torch):
    lib = pa.load()
    desc = pa.DecodeDesc(num_seqs=512, num_q_heads=128, num_kv_heads=8, head_dim=128, block_size=16,
                         num_blocks=1000, max_blocks_per_seq=4096, max_context_len=65536, scale=0.1)
    assert pa.decode_workspace_bytes(desc) > pa.NOALLOC_SCRATCH_BYTES
    st = lib.pa_paged_attention_decode_noalloc(ctypes.byref(desc), 16, 16, 16, 16, 16, 16, None, None)
    assert st == pa.PA_ERR_WORKSPACE
