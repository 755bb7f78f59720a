"""Decode with append (pa_paged_attention_decode_append): the decode step's
cache write and attention in one launch must give the same bits, in the
output and in both pools, as reshape_and_cache followed by decode -- over
every kernel instance (head dim, block size, GQA group, split-K, CTA order),
plus the fp64 oracle on a full layer, the refused slots and graph replay."""
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


def two_launches(torch, case, d, slots=None):
    kp, vp = d["k_pool"].clone(), d["v_pool"].clone()
    pa.reshape_and_cache(d["new_k"], d["new_v"], kp, vp, d["slots"] if slots is None else slots)
    out = pa.paged_attention_decode(d["q"], kp, vp, d["bt"], d["ctx"], scale=case.scale,
                                    max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    return bf16_host(out), bf16_host(kp), bf16_host(vp)


def one_launch(torch, case, d, slots=None, err=None):
    kp, vp = d["k_pool"].clone(), d["v_pool"].clone()
    out = pa.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slots"] if slots is None else slots,
                                           kp, vp, d["bt"], d["ctx"], scale=case.scale,
                                           max_context_len=case.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    return bf16_host(out), bf16_host(kp), bf16_host(vp)


CASES = [
    # name, context lengths, Hq, Hkv, D, B, split-K part length (pages) or None
    ("b16_g4", [1, 2, 15, 16, 17, 31, 32, 33, 300, 900, 2048], 32, 8, 128, 16, None),
    ("b16_g4_split", [1, 16, 17, 129, 700, 2001], 32, 8, 128, 16, 3),
    ("b32_g8", [1, 31, 32, 33, 64, 65, 1000, 3000], 64, 8, 128, 32, None),
    ("b32_g8_split", [1, 33, 1000, 3000], 64, 8, 128, 32, 4),
    ("b16_g16", [1, 17, 250, 513], 32, 2, 128, 16, None),
    ("d64_b16_g1", [1, 5, 16, 17, 100, 400], 4, 4, 64, 16, None),
    ("d64_b32_g2", [1, 32, 33, 100, 777], 8, 4, 64, 32, 2),
]


@pytest.mark.parametrize("lpt", [None, "1", "0"])
@pytest.mark.parametrize("name,ctx,hq,hkv,D,B,pp", CASES, ids=[c[0] for c in CASES])
def test_append_bits_equal_two_launches(torch, monkeypatch, name, ctx, hq, hkv, D, B, pp, lpt):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    if lpt is None:
        monkeypatch.delenv("PA_DECODE_LPT", raising=False)
    else:
        monkeypatch.setenv("PA_DECODE_LPT", lpt)
    case = wl.make_decode_case(f"append_{name}", ctx, hq, hkv, D, B, seed=31, stream=len(ctx) + D + B)
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = two_launches(torch, case, d)
    got = one_launch(torch, case, d, err=err)
    assert int(err.item()) == 0
    for g, w, what in zip(got, want, ("out", "k_pool", "v_pool")):
        assert np.array_equal(g, w), f"{name}: {what} differs from reshape_and_cache + decode"


def test_append_llama8b_against_oracle(torch, ora):
    """A Llama-3-8B-shaped layer: pools bit-exact with the oracle's cache
    write, attention within tolerance of the fp64 oracle."""
    case = wl.llama8b_decode()
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kp, vp = one_launch(torch, case, d, err=err)
    hk, hv = case.k_pool.copy(), case.v_pool.copy()
    assert ora.reshape_and_cache(case.new_k, case.new_v, hk, hv, case.slot_mapping) == 0
    assert np.array_equal(kp, hk) and np.array_equal(vp, hv)
    ref, st = ora.decode(case.q, hk, hv, case.block_tables, case.context_lens, case.scale)
    assert np.all(st == 0) and int(err.item()) == 0
    assert_close(out, ref, "llama8b decode with append")


def test_append_negative_slot_writes_nothing(torch):
    case = wl.make_decode_case("append_skip", [1, 17, 40, 300, 64], 16, 4, 128, 16, seed=32, stream=3)
    d = upload_case(case, torch)
    slots = d["slots"].clone()
    slots[1] = -1
    slots[3] = -7
    want = two_launches(torch, case, d, slots)  # reshape_and_cache skips them too
    got = one_launch(torch, case, d, slots)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_append_refuses_a_slot_that_is_not_the_last_position(torch):
    """A slot elsewhere in the pool, or outside it, sets PA_DEVERR_SLOT and
    writes nothing: the sequence attends to its cache as it was."""
    case = wl.make_decode_case("append_bad_slot", [20, 17, 40, 300], 16, 4, 128, 16, seed=33, stream=4)
    d = upload_case(case, torch)
    slots = d["slots"].clone()
    slots[0] = slots[0] - 1                      # position ctx-2 of the same sequence
    slots[2] = case.num_blocks * case.block_size  # past the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kp, vp = one_launch(torch, case, d, slots, err)
    assert int(err.item()) & pa.DEVERR_SLOT
    # only the good sequences' tokens were written ...
    ok_slots = slots.clone()
    ok_slots[0] = -1
    ok_slots[2] = -1
    w_out, w_kp, w_vp = two_launches(torch, case, d, ok_slots)
    assert np.array_equal(kp, w_kp) and np.array_equal(vp, w_vp)
    # ... and every output equals decode over that cache
    assert np.array_equal(out, w_out)


def test_append_bad_context_writes_nothing(torch):
    case = wl.make_decode_case("append_bad_ctx", [30, 50, 9], 8, 2, 128, 16, seed=34, stream=5)
    d = upload_case(case, torch)
    ctx = d["ctx"].clone()
    ctx[1] = 0
    d2 = dict(d, ctx=ctx)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kp, vp = one_launch(torch, case, d2, err=err)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(out[1])                    # rows of a bad context are zeros
    slots = d["slots"].clone()
    slots[1] = -1
    w_out, w_kp, w_vp = two_launches(torch, case, d2, slots)
    assert np.array_equal(kp, w_kp) and np.array_equal(vp, w_vp)
    assert np.array_equal(out, w_out)


def test_append_graph_replay(torch, monkeypatch):
    """Captured once and replayed: the same bits each replay (the append is
    idempotent on a fixed step's inputs)."""
    monkeypatch.setenv("PA_PARTITION_PAGES", "4")  # split-K counters across replays
    case = wl.make_decode_case("append_graph", [1, 100, 999, 64, 500], 32, 8, 128, 16, seed=35, stream=6)
    d = upload_case(case, torch)
    want = one_launch(torch, case, d)
    kp, vp = d["k_pool"].clone(), d["v_pool"].clone()
    out = torch.empty_like(d["q"])
    desc = pa.make_desc(d["q"], kp, d["bt"], scale=case.scale, max_context_len=case.max_context_len)
    ws = pa.decode_workspace(desc, d["q"].device)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            pa.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slots"], kp, vp, d["bt"], d["ctx"],
                                             out, scale=case.scale, max_context_len=case.max_context_len,
                                             workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(out), want[0])
        assert np.array_equal(bf16_host(kp), want[1]) and np.array_equal(bf16_host(vp), want[2])


def test_append_rejects_bad_arguments(torch):
    case = wl.make_decode_case("append_args", [10, 20], 8, 2, 128, 16, seed=36, stream=7)
    d = upload_case(case, torch)
    with pytest.raises(ValueError):
        pa.paged_attention_decode_append(d["q"], d["new_k"][:1], d["new_v"], d["slots"], d["k_pool"], d["v_pool"],
                                         d["bt"], d["ctx"])
    desc = pa.make_desc(d["q"], d["k_pool"], d["bt"])
    lib = pa.load()
    st = lib.pa_paged_attention_decode_append(
        ctypes.byref(desc), d["q"].data_ptr(), None,
        d["new_v"].data_ptr(), d["slots"].data_ptr(), d["k_pool"].data_ptr(), d["v_pool"].data_ptr(),
        d["bt"].data_ptr(), d["ctx"].data_ptr(), d["q"].data_ptr(), None, 0, None, None)
    assert st == pa.PA_ERR_INVALID


def test_append_long_context_full_size(torch, ora):
    """The 8 x 32768-token, GQA-8 case as the bench launches it (decode with
    append, four 512-page split-K parts): bits equal to the two launches on
    every output and pool byte, every (sequence, query head) row against the
    fp64 oracle."""
    case = wl.long_context_decode()
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = two_launches(torch, case, d)
    got = one_launch(torch, case, d, err=err)
    assert int(err.item()) == 0
    for g, w, what in zip(got, want, ("out", "k_pool", "v_pool")):
        assert np.array_equal(g, w), f"long context: {what} differs from the two launches"
    hk, hv = case.k_pool.copy(), case.v_pool.copy()
    assert ora.reshape_and_cache(case.new_k, case.new_v, hk, hv, case.slot_mapping) == 0
    sub = case.__class__(**{**case.__dict__, "k_pool": hk, "v_pool": hv})
    ref = oracle_rows(ora, sub).reshape(got[0].shape)
    assert_close(got[0], ref, "long context with append")
