"""GPU parity of causal chunked-prefill attention (tcgen05) with the fp64
oracle, through the C-ABI library; plus the full mixed continuous-batching
step (prefill chunks and decode sequences sharing one page pool)."""
import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def upload_chunks(m, torch):
    d = {
        "q": bf16_dev(m.q_chunk, torch),
        "k_pool": bf16_dev(m.decode.k_pool, torch),
        "v_pool": bf16_dev(m.decode.v_pool, torch),
        "bt": torch.from_numpy(np.ascontiguousarray(m.chunk_tables)).cuda(),
        "ctx": torch.from_numpy(np.ascontiguousarray(m.chunk_ctx)).cuda(),
        "cu": torch.from_numpy(np.ascontiguousarray(m.cu_q)).cuda(),
        "nk": bf16_dev(m.chunk_new_k, torch),
        "nv": bf16_dev(m.chunk_new_v, torch),
        "slots": torch.from_numpy(np.ascontiguousarray(m.chunk_slots)).cuda(),
    }
    return d


def run_prefill(torch, m, d, err=None):
    pa.reshape_and_cache(d["nk"], d["nv"], d["k_pool"], d["v_pool"], d["slots"], err_flag=err)
    out = pa.paged_attention_prefill_chunk(d["q"], d["cu"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"],
                                           max_q_len=int(m.chunk_lens.max()), scale=m.decode.scale,
                                           max_context_len=int(m.chunk_ctx.max()), err_flag=err)
    torch.cuda.synchronize()
    return out


def oracle_pools(ora, m):
    kp, vp = m.decode.k_pool.copy(), m.decode.v_pool.copy()
    assert ora.reshape_and_cache(m.chunk_new_k, m.chunk_new_v, kp, vp, m.chunk_slots) == 0
    return kp, vp


CASES = [  # (chunk_lens, chunk_ctx, Hq, Hkv, B)
    ([1, 37, 128, 200], [1, 100, 128, 700], 8, 2, 16),
    ([64, 300, 33], [64, 300, 1000], 32, 8, 32),
    ([129, 5], [400, 5], 8, 8, 16),
    ([100, 257], [613, 257], 16, 2, 32),
    ([40, 77], [2000, 77], 16, 1, 16),
    ([300], [1300], 4, 2, 32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"C{c[0]}ctx{c[1]}q{c[2]}kv{c[3]}b{c[4]}")
def test_prefill_chunks_full(torch, ora, case):
    lens, ctxs, Hq, Hkv, B = case
    m = wl.make_mixed_step("pf", lens, ctxs, [], Hq, Hkv, 128, B, seed=21, stream=sum(lens) % 997)
    d = upload_chunks(m, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_prefill(torch, m, d, err)
    assert int(err.item()) == 0
    kp, vp = oracle_pools(ora, m)
    got = bf16_host(out)
    ref = np.zeros((int(m.cu_q[-1]), Hq, 128))
    for r in range(len(lens)):
        for i in range(lens[r]):
            for h in range(Hq):
                o, st = ora.prefill_row(m.q_chunk, m.cu_q, kp, vp, m.chunk_tables, m.chunk_ctx, m.decode.scale,
                                        r, i, h)
                assert st == 0
                ref[m.cu_q[r] + i, h] = o
    assert_close(got, ref, f"prefill {case}")


def test_prefill_first_row_of_whole_prompt_is_v0(torch):
    """C = ctx: row 0 sees only key 0, so its output is v0 exactly."""
    m = wl.make_mixed_step("v0", [200], [200], [], 8, 2, 128, 16, seed=22, stream=5)
    d = upload_chunks(m, torch)
    got = bf16_host(run_prefill(torch, m, d))
    for h in range(8):
        assert np.array_equal(got[0, h], m.chunk_new_v[0, h // 4])


def test_prefill_bad_chunk_flagged(torch):
    m = wl.make_mixed_step("bad", [10, 20], [50, 20], [], 8, 2, 128, 16, seed=23, stream=6)
    d = upload_chunks(m, torch)
    d["ctx"][1] = 5  # 20 query tokens over a 5-token context
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_prefill(torch, m, d, err)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(bf16_host(out)[10:30])


def test_mixed_step_full_size(torch, ora):
    """16 prefill chunks x 512 tokens (ctx ~U[512,8192]) plus 240 decodes
    (ctx ~U[64,4096]) on one B=32 pool: one reshape_and_cache for all new
    tokens, the prefill call and the decode call; sampled outputs of both."""
    m = wl.mixed_step()
    dec = m.decode
    d = upload_chunks(m, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_all = np.concatenate([m.chunk_new_k, dec.new_k])
    v_all = np.concatenate([m.chunk_new_v, dec.new_v])
    s_all = np.concatenate([m.chunk_slots, dec.slot_mapping])
    pa.reshape_and_cache(bf16_dev(k_all, torch), bf16_dev(v_all, torch), d["k_pool"], d["v_pool"],
                         torch.from_numpy(s_all).cuda(), err_flag=err)
    pout = pa.paged_attention_prefill_chunk(d["q"], d["cu"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"],
                                            max_q_len=512, scale=dec.scale, max_context_len=int(m.chunk_ctx.max()),
                                            err_flag=err)
    dq = bf16_dev(dec.q, torch)
    dout = pa.paged_attention_decode(dq, d["k_pool"], d["v_pool"], torch.from_numpy(dec.block_tables).cuda(),
                                     torch.from_numpy(dec.context_lens).cuda(), scale=dec.scale,
                                     max_context_len=dec.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp, vp = dec.k_pool.copy(), dec.v_pool.copy()
    assert ora.reshape_and_cache(k_all, v_all, kp, vp, s_all) == 0
    assert np.array_equal(bf16_host(d["k_pool"]), kp) and np.array_equal(bf16_host(d["v_pool"]), vp)
    gp = bf16_host(pout)
    rows, refs = [], []
    for r in range(len(m.chunk_lens)):
        for i in (0, 1, 127, 128, 255, 300, 511):
            for h in (0, 5, 31):
                o, st = ora.prefill_row(m.q_chunk, m.cu_q, kp, vp, m.chunk_tables, m.chunk_ctx, dec.scale, r, i, h)
                assert st == 0
                rows.append(gp[m.cu_q[r] + i, h])
                refs.append(o)
    assert_close(np.stack(rows), np.stack(refs), "mixed step prefill")
    gd = bf16_host(dout)
    heads = [(s, h) for s in range(0, dec.num_seqs, 7) for h in (0, 17)]
    ref = np.stack([ora.decode_head(dec.q, kp, vp, dec.block_tables, dec.context_lens, dec.scale, s, h)[0]
                    for s, h in heads])
    assert_close(np.stack([gd[s, h] for s, h in heads]), ref, "mixed step decode")
