"""Every entry point captured into a CUDA graph and replayed gives the same
bits as the same calls launched eagerly.  A serving loop replays its decode
step from a graph, so the launch-time state each call bakes in (tensor maps,
the split plan, the arrival-counter epoch of split-K decode) has to stay valid
for every replay; replays also run back to back on one workspace."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import bf16_dev, bf16_host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


@pytest.mark.parametrize("pp", [None, 3])
def test_decode_graph_replays(torch, monkeypatch, pp):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))  # several parts per sequence: split-K merge
    st = wl.Stream(7, 1)
    case = wl.make_decode_case("graph", st.integers(1, 900, 19), 32, 8, 128, 16, seed=7, stream=11)
    q, kp, vp = bf16_dev(case.q, torch), bf16_dev(case.k_pool, torch), bf16_dev(case.v_pool, torch)
    bt = torch.from_numpy(case.block_tables).cuda()
    ctx = torch.from_numpy(case.context_lens).cuda()
    desc = pa.make_desc(q, kp, bt, max_context_len=case.max_context_len)
    ws = pa.decode_workspace(desc, q.device)
    eager = pa.paged_attention_decode(q, kp, vp, bt, ctx, max_context_len=case.max_context_len, workspace=ws)
    torch.cuda.synchronize()
    want = bf16_host(eager)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def body():
        for _ in range(3):  # back-to-back launches on one workspace inside the graph
            pa.paged_attention_decode(q, kp, vp, bt, ctx, out, max_context_len=case.max_context_len, workspace=ws,
                                      err_flag=err)

    g = capture(torch, body)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(out), want)
    assert int(err.item()) == 0


def test_prefill_graph_replays(torch):
    Hq, Hkv, D, B = 16, 4, 128, 32
    st = wl.Stream(8, 1)
    chunk_ctx = np.array([300, 129, 700], np.int32)
    chunk_len = np.array([70, 129, 200], np.int32)
    case = wl.make_decode_case("graph_prefill", chunk_ctx, Hq, Hkv, D, B, seed=8, stream=12, with_new_tokens=False)
    cu = np.concatenate([[0], np.cumsum(chunk_len)]).astype(np.int32)
    qc = wl.normal_bf16(st, (int(cu[-1]), Hq, D))
    kp, vp = bf16_dev(case.k_pool, torch), bf16_dev(case.v_pool, torch)
    q = bf16_dev(qc, torch)
    bt = torch.from_numpy(case.block_tables).cuda()
    ctx = torch.from_numpy(chunk_ctx).cuda()
    cu_d = torch.from_numpy(cu).cuda()
    kw = dict(max_q_len=int(chunk_len.max()), scale=1 / math.sqrt(D), max_context_len=int(chunk_ctx.max()))
    eager = pa.paged_attention_prefill_chunk(q, cu_d, kp, vp, bt, ctx, **kw)
    torch.cuda.synchronize()
    want = bf16_host(eager)
    out = torch.empty_like(q)
    g = capture(torch, lambda: pa.paged_attention_prefill_chunk(q, cu_d, kp, vp, bt, ctx, out, **kw))
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(out), want)


def test_cache_writes_graph_replay(torch):
    case = wl.make_decode_case("graph_cache", [5, 40, 17, 64], 8, 4, 128, 16, seed=9, stream=13)
    pairs = np.array([[case.block_tables[0, 0], case.num_blocks - 1], [case.block_tables[1, 1], case.num_blocks - 2]],
                     np.int64)
    kp0, vp0 = bf16_dev(case.k_pool, torch), bf16_dev(case.v_pool, torch)
    nk, nv = bf16_dev(case.new_k, torch), bf16_dev(case.new_v, torch)
    slots = torch.from_numpy(case.slot_mapping).cuda()
    pr = torch.from_numpy(pairs).cuda()

    def step(kp, vp):
        pa.copy_blocks([kp], [vp], pr)
        pa.reshape_and_cache(nk, nv, kp, vp, slots)

    ke, ve = kp0.clone(), vp0.clone()
    step(ke, ve)
    kg, vg = kp0.clone(), vp0.clone()
    g = capture(torch, lambda: step(kg, vg))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(kg, ke) and torch.equal(vg, ve)
