"""The mixed-step launch (pa_paged_attention_mixed): a continuous-batching
step's chunked prefill and decode in one grid whose CTAs take one role each.
Its outputs must be the bits of pa_paged_attention_prefill_chunk and
pa_paged_attention_decode called separately with the same arguments -- over
page sizes, GQA groups, split-K decode, the three dispatch orders, empty
parts, bad contexts and graph replay -- and agree with the fp64 oracle."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def upload(torch, m):
    """The mixed case on the device, with the chunks' K/V already cached."""
    dec = m.decode
    d = {"kp": bf16_dev(dec.k_pool, torch), "vp": bf16_dev(dec.v_pool, torch),
         "qc": bf16_dev(m.q_chunk, torch), "cu": torch.from_numpy(m.cu_q).cuda(),
         "cbt": torch.from_numpy(m.chunk_tables).cuda(), "cctx": torch.from_numpy(m.chunk_ctx).cuda(),
         "qd": bf16_dev(dec.q, torch), "dbt": torch.from_numpy(dec.block_tables).cuda(),
         "dctx": torch.from_numpy(dec.context_lens).cuda()}
    if len(m.chunk_slots):
        pa.reshape_and_cache(bf16_dev(m.chunk_new_k, torch), bf16_dev(m.chunk_new_v, torch), d["kp"], d["vp"],
                             torch.from_numpy(m.chunk_slots).cuda())
    torch.cuda.synchronize()
    return d


def oracle_pools(ora, m):
    """The cache as the oracle writes it: the chunks' K/V into host copies of the pools."""
    hk, hv = m.decode.k_pool.copy(), m.decode.v_pool.copy()
    if len(m.chunk_slots):
        assert ora.reshape_and_cache(m.chunk_new_k, m.chunk_new_v, hk, hv, m.chunk_slots) == 0
    return hk, hv


def kw(m):
    return dict(max_q_len=max(1, int(m.chunk_lens.max()) if len(m.chunk_lens) else 1), scale=m.decode.scale)


def separate(torch, m, d, err=None):
    k = kw(m)
    pmax = int(m.chunk_ctx.max()) if len(m.chunk_ctx) else 1
    dmax = int(m.decode.context_lens.max()) if m.decode.num_seqs else 1
    po = pa.paged_attention_prefill_chunk(d["qc"], d["cu"], d["kp"], d["vp"], d["cbt"], d["cctx"],
                                          max_q_len=k["max_q_len"], scale=k["scale"], max_context_len=pmax,
                                          err_flag=err)
    do = pa.paged_attention_decode(d["qd"], d["kp"], d["vp"], d["dbt"], d["dctx"], scale=k["scale"],
                                   max_context_len=dmax, err_flag=err)
    torch.cuda.synchronize()
    return bf16_host(po), bf16_host(do)


def fused(torch, m, d, err=None, pout=None, dout=None):
    k = kw(m)
    pmax = int(m.chunk_ctx.max()) if len(m.chunk_ctx) else 1
    dmax = int(m.decode.context_lens.max()) if m.decode.num_seqs else 1
    po, do = pa.paged_attention_mixed(d["qc"], d["cu"], d["cbt"], d["cctx"], d["qd"], d["dbt"], d["dctx"], d["kp"],
                                      d["vp"], pout, dout, max_q_len=k["max_q_len"], scale=k["scale"],
                                      prefill_max_context_len=pmax, decode_max_context_len=dmax, err_flag=err)
    torch.cuda.synchronize()
    return bf16_host(po), bf16_host(do)


CASES = [
    # name, chunk lengths, chunk contexts, decode contexts, Hq, Hkv, B, split-K part length or None
    ("b32_g4", [70, 129, 200, 512], [300, 129, 700, 2000], [1, 31, 64, 65, 900, 2000, 3000, 17], 32, 8, 32, None),
    ("b16_g4", [70, 129, 200], [300, 129, 700], [1, 16, 17, 300, 1200, 63], 32, 8, 16, None),
    ("b16_g16_split", [100, 33], [400, 2100], [1, 500, 3000, 2048, 20], 32, 2, 16, 8),
    ("b32_g1_split", [256, 5], [256, 900], [2, 33, 1500, 4000], 8, 8, 32, 5),
    ("b32_g8", [130], [1000], list(range(1, 200, 13)), 64, 8, 32, None),
]


@pytest.mark.parametrize("order", [None, "decode-first", "prefill-first"])
@pytest.mark.parametrize("name,cl,cc,dc,hq,hkv,B,pp", CASES, ids=[c[0] for c in CASES])
def test_mixed_bits_equal_separate_launches(torch, monkeypatch, name, cl, cc, dc, hq, hkv, B, pp, order):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    if order is None:
        monkeypatch.delenv("PA_MIXED_ORDER", raising=False)
    else:
        monkeypatch.setenv("PA_MIXED_ORDER", order)
    m = wl.make_mixed_step(f"mixed_{name}", cl, cc, dc, hq, hkv, 128, B, seed=41, stream=len(dc) + B)
    d = upload(torch, m)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = separate(torch, m, d)
    got = fused(torch, m, d, err)
    assert int(err.item()) == 0
    assert np.array_equal(got[0], want[0]), f"{name}: prefill rows differ from the prefill kernel"
    assert np.array_equal(got[1], want[1]), f"{name}: decode rows differ from the decode kernel"


def test_mixed_against_oracle(torch, ora):
    m = wl.make_mixed_step("mixed_oracle", [64, 200], [500, 1300], [1, 77, 640, 1500, 33], 32, 8, 128, 32,
                           seed=42, stream=9)
    d = upload(torch, m)
    po, do = fused(torch, m, d)
    hk, hv = oracle_pools(ora, m)
    ref, st = ora.decode(m.decode.q, hk, hv, m.decode.block_tables, m.decode.context_lens, m.decode.scale)
    assert np.all(st == 0)
    assert_close(do, ref, "mixed launch, decode rows")
    rows = [(0, 0), (0, 63), (1, 0), (1, 101), (1, 199)]
    got = np.stack([po[m.cu_q[r] + i] for r, i in rows])
    want = np.stack([np.stack([ora.prefill_row(m.q_chunk, m.cu_q, hk, hv, m.chunk_tables, m.chunk_ctx, m.decode.scale,
                                               r, i, h)[0] for h in range(32)]) for r, i in rows])
    assert_close(got, want, "mixed launch, prefill rows")


def test_mixed_with_one_part_empty(torch):
    only_p = wl.make_mixed_step("mixed_only_prefill", [90, 40], [90, 600], [], 16, 4, 128, 16, seed=43, stream=1)
    d = upload(torch, only_p)
    got, want = fused(torch, only_p, d), separate(torch, only_p, d)
    assert np.array_equal(got[0], want[0])
    only_d = wl.make_mixed_step("mixed_only_decode", [], [], [5, 700, 64], 16, 4, 128, 16, seed=43, stream=2)
    d = upload(torch, only_d)
    d["qc"] = torch.zeros((0, 16, 128), dtype=torch.bfloat16, device="cuda")
    d["cu"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    d["cbt"] = torch.zeros((0, d["dbt"].shape[1]), dtype=torch.int32, device="cuda")
    d["cctx"] = torch.zeros(0, dtype=torch.int32, device="cuda")
    got = fused(torch, only_d, d)
    want = pa.paged_attention_decode(d["qd"], d["kp"], d["vp"], d["dbt"], d["dctx"], scale=only_d.decode.scale,
                                     max_context_len=700)
    torch.cuda.synchronize()
    assert np.array_equal(got[1], bf16_host(want))


def test_mixed_bad_contexts_flagged_like_separate_calls(torch):
    m = wl.make_mixed_step("mixed_bad", [50, 60], [200, 300], [40, 70, 90], 16, 4, 128, 32, seed=44, stream=3)
    d = upload(torch, m)
    d["dctx"][1] = 0        # a decode sequence with no context
    d["cctx"][0] = 10       # a chunk longer than its context
    e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    po_f, do_f = fused(torch, m, d, e1, torch.zeros_like(d["qc"]), torch.zeros_like(d["qd"]))
    pa.paged_attention_prefill_chunk(d["qc"], d["cu"], d["kp"], d["vp"], d["cbt"], d["cctx"], max_q_len=60,
                                     scale=m.decode.scale, max_context_len=300, err_flag=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) & pa.DEVERR_CTX and int(e2.item()) & pa.DEVERR_CTX
    assert not np.any(do_f[1]) and not np.any(po_f[:50])
    want = separate(torch, m, d)
    assert np.array_equal(do_f, want[1]) and np.array_equal(po_f[50:], want[0][50:])


def test_mixed_rejects_different_pools(torch):
    m = wl.make_mixed_step("mixed_args", [20], [40], [10], 16, 4, 128, 16, seed=45, stream=4)
    d = upload(torch, m)
    other = torch.zeros((d["kp"].shape[0], 4, 32, 128), dtype=torch.bfloat16, device="cuda")  # 32-token pages
    pdesc = pa.make_desc(d["qc"], d["kp"], d["cbt"], num_seqs=1)
    ddesc = pa.make_desc(d["qd"], other, d["dbt"])
    import ctypes
    st = pa.load().pa_paged_attention_mixed(ctypes.byref(pdesc), d["qc"].data_ptr(), d["cu"].data_ptr(), 20, 20,
                                            d["cbt"].data_ptr(), d["cctx"].data_ptr(), d["qc"].data_ptr(),
                                            ctypes.byref(ddesc), d["qd"].data_ptr(), d["dbt"].data_ptr(),
                                            d["dctx"].data_ptr(), d["qd"].data_ptr(), None, 0, d["kp"].data_ptr(),
                                            d["vp"].data_ptr(), None, None)
    assert st == pa.PA_ERR_INVALID


def test_mixed_graph_replay(torch, monkeypatch):
    monkeypatch.setenv("PA_PARTITION_PAGES", "6")
    m = wl.make_mixed_step("mixed_graph", [100, 300], [500, 1000], [3, 1000, 2500, 77], 32, 8, 128, 32,
                           seed=46, stream=5)
    d = upload(torch, m)
    want = fused(torch, m, d)
    pout, dout = torch.empty_like(d["qc"]), torch.empty_like(d["qd"])
    ddesc = pa.make_desc(d["qd"], d["kp"], d["dbt"], max_context_len=2500)
    ws = pa.decode_workspace(ddesc, d["qd"].device)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            pa.paged_attention_mixed(d["qc"], d["cu"], d["cbt"], d["cctx"], d["qd"], d["dbt"], d["dctx"], d["kp"],
                                     d["vp"], pout, dout, max_q_len=300, scale=m.decode.scale,
                                     prefill_max_context_len=1000, decode_max_context_len=2500, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        pout.zero_()
        dout.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(pout), want[0]) and np.array_equal(bf16_host(dout), want[1])
    assert math.isfinite(float(bf16_host(dout).astype(np.float32).sum()))


def test_mixed_full_size(torch, ora):
    """The benchmark's mixed step (16 chunks x 512 over contexts U[512,8192] +
    240 decodes, 32-token pages) through the mixed-step launch: bits equal to
    the separate prefill and decode calls on every row; every decode row and
    sampled prefill rows against the fp64 oracle."""
    m = wl.mixed_step()
    d = upload(torch, m)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = separate(torch, m, d)
    got = fused(torch, m, d, err)
    assert int(err.item()) == 0
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    hk, hv = oracle_pools(ora, m)
    dec = m.decode
    sub = dec.__class__(**{**dec.__dict__, "k_pool": hk, "v_pool": hv})
    ref = oracle_rows(ora, sub).reshape(got[1].shape)
    assert_close(got[1], ref, "mixed step, decode rows")
    rows = [(r, i) for r in (0, 7, 15) for i in (0, 255, 511)]
    pre = np.stack([np.stack([ora.prefill_row(m.q_chunk, m.cu_q, hk, hv, m.chunk_tables, m.chunk_ctx,
                                              dec.scale, r, i, h)[0] for h in (0, 13, 31)]) for r, i in rows])
    gotp = np.stack([np.stack([got[0][m.cu_q[r] + i, h] for h in (0, 13, 31)]) for r, i in rows])
    assert_close(gotp, pre, "mixed step, prefill rows")
