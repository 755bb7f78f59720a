"""The bounded on-chip wait.  Every kernel of the library waits on
shared-memory mbarriers with a bound, after which it reports
PA_DEVERR_TIMEOUT and returns instead of hanging the GPU.  Here one warp waits,
through the same routine, on an mbarrier that nothing arrives on, with a short
bound: the launch must end by itself with the status set, and the context must
stay usable (a decode afterwards still matches the oracle)."""
import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_host, need_gpu, upload_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("limit", [1, 2_000_000])
def test_wait_gives_up_and_reports_timeout(torch, ora, limit):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pa.selftest_bounded_wait(limit, err, done)
    e1.record()
    torch.cuda.synchronize()
    assert int(done.item()) == 1, "the waiting kernel did not run to its end"
    assert int(err.item()) == pa.DEVERR_TIMEOUT
    ms = e0.elapsed_time(e1)
    assert ms < 1000.0
    if limit > 1:  # it waited about the bound (SM clock at most ~2.1 GHz) before giving up
        assert ms >= 0.5 * limit / 2.1e9 * 1e3, ms

    # the context is still usable: a decode step against the oracle
    case = wl.tiny_decode()
    d = upload_case(case, torch)
    err.zero_()
    pa.reshape_and_cache(d["new_k"], d["new_v"], d["k_pool"], d["v_pool"], d["slots"], err_flag=err)
    out = pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"], scale=case.scale,
                                    max_context_len=case.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    assert ora.reshape_and_cache(case.new_k, case.new_v, kp, vp, case.slot_mapping) == 0
    ref, st = ora.decode(case.q, kp, vp, case.block_tables, case.context_lens, case.scale)
    assert np.all(st == 0)
    assert_close(bf16_host(out), ref, "decode after a timed-out wait")


def test_wait_bound_is_checked_on_the_host(torch):
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, -5, 4_000_000_001):
        with pytest.raises(pa.PaError):
            pa.selftest_bounded_wait(bad, None, done)
