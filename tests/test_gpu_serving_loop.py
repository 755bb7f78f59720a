"""A serving loop driven the way a caller drives the library: the host block
manager admits prompts (reusing cached prefix blocks), their remaining tokens
are written with reshape_and_cache and attended with chunked prefill; a
sample is forked; then several decode steps append one token per sequence
(copy_blocks for copy-on-write pairs, reshape_and_cache for the new K/V) and
decode every resident sequence, with one sequence swapped out to pinned host
memory and back in the middle.  A host mirror of the pools follows the same
operations through the fp64 oracle: attention outputs match it within
tolerance and the pools match it bit for bit at the end."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu

pytestmark = pytest.mark.gpu

B, HQ, HKV, D = 16, 8, 2, 128
N_DEV, N_HOST = 96, 32
SCALE = 1 / math.sqrt(D)


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("batch", [False, True])
def test_serving_loop_matches_the_oracle(torch, ora, batch):
    """batch: each decode step's appends are one append_batch call and the
    attention call's table matrix and context lengths come from block_tables."""
    st = wl.Stream(91, 4)
    bm = pa.BlockManager(N_DEV, B, num_host_blocks=N_HOST)
    kp = wl.normal_bf16(st, (N_DEV, HKV, B, D))   # never-used slots hold noise
    vp = wl.normal_bf16(st, (N_DEV, HKV, B, D))
    hk, hv = np.zeros((N_HOST, HKV, B, D), np.uint16), np.zeros((N_HOST, HKV, B, D), np.uint16)
    dk, dv = bf16_dev(kp, torch), bf16_dev(vp, torch)
    gk = torch.zeros((N_HOST, HKV, B, D), dtype=torch.bfloat16).pin_memory()
    gv = torch.zeros_like(gk).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv_of = {}  # K/V of a position is a function of the tokens up to it (as a model's would be)

    def kv(tokens, j):
        key = tuple(tokens[: j + 1])
        if key not in kv_of:
            kv_of[key] = (wl.normal_bf16(st, (HKV, D)), wl.normal_bf16(st, (HKV, D)))
        return kv_of[key]

    def write(seq_tokens, table, first):  # reshape_and_cache of positions first.. on both sides
        n = len(seq_tokens)
        if n <= first:
            return
        k = np.stack([kv(seq_tokens, j)[0] for j in range(first, n)])
        v = np.stack([kv(seq_tokens, j)[1] for j in range(first, n)])
        slots = np.array([table[j // B] * B + j % B for j in range(first, n)], np.int64)
        pa.reshape_and_cache(bf16_dev(k, torch), bf16_dev(v, torch), dk, dv, torch.from_numpy(slots).cuda(),
                             err_flag=err)
        assert ora.reshape_and_cache(k, v, kp, vp, slots) == 0

    def tables(seqs):
        ts = [bm.block_table(s) for s in seqs]
        bt = np.full((len(seqs), max(len(t) for t in ts)), -1, np.int32)
        for i, t in enumerate(ts):
            bt[i, : len(t)] = t
        return bt

    # ---- admission: prompts, the second repeating three blocks of the first
    p0 = [int(x) for x in st.integers(0, 30000, 70)]
    prompts = {0: p0, 1: p0[:48] + [int(x) for x in st.integers(0, 30000, 20)],
               2: [int(x) for x in st.integers(0, 30000, 33)]}
    toks = {}
    for s, p in prompts.items():
        cached = bm.add_seq_tokens(s, p)
        assert cached == (48 if s == 1 else 0)
        toks[s] = list(p)
        table = bm.block_table(s)
        write(p, table, cached)
        C, n = len(p) - cached, len(p)
        q = wl.normal_bf16(st, (C, HQ, D))
        out = pa.paged_attention_prefill_chunk(bf16_dev(q, torch), torch.tensor([0, C], dtype=torch.int32,
                                                                                device="cuda"),
                                               dk, dv, torch.from_numpy(tables([s])).cuda(),
                                               torch.tensor([n], dtype=torch.int32, device="cuda"), max_q_len=C,
                                               scale=SCALE, max_context_len=n, err_flag=err)
        torch.cuda.synchronize()
        rows = sorted({0, C // 2, C - 1})
        ref = np.stack([np.stack([ora.prefill_row(q, np.array([0, C], np.int32), kp, vp, tables([s]),
                                                  np.array([n], np.int32), SCALE, 0, i, h)[0]
                                  for h in range(HQ)]) for i in rows])
        assert_close(bf16_host(out)[rows], ref, f"prefill of prompt {s}")
    bm.fork(0, 3)  # a second sample of prompt 0
    toks[3] = list(toks[0])

    # ---- decode steps, with sequence 2 preempted for steps 2 and 3
    swapped = set()
    for step in range(6):
        if step == 2:
            pairs = np.array(bm.swap_out(2), np.int64)
            pa.swap_blocks([dk], [dv], [gk], [gv], torch.from_numpy(pairs).cuda(), err_flag=err)
            for d, h in pairs:
                hk[h], hv[h] = kp[d], vp[d]
            swapped.add(2)
        if step == 4:
            pairs = np.array(bm.swap_in(2), np.int64)
            pa.swap_blocks([gk], [gv], [dk], [dv], torch.from_numpy(pairs).cuda(), err_flag=err)
            for h, d in pairs:
                kp[d], vp[d] = hk[h], hv[h]
            swapped.discard(2)
        live = [s for s in sorted(toks) if s not in swapped]
        cow = []
        if batch:
            for s in live:
                toks[s].append(int(st.integers(0, 30000, 1)[0]))
            sl, cw = bm.append_batch(live)
            for i, s in enumerate(live):
                assert sl[i] == bm.block_table(s)[(len(toks[s]) - 1) // B] * B + (len(toks[s]) - 1) % B
                if cw[i, 0] >= 0:
                    cow.append((int(cw[i, 0]), int(cw[i, 1])))
        for s in live if not batch else ():
            toks[s].append(int(st.integers(0, 30000, 1)[0]))
            slot, pair = bm.append(s)
            assert slot == bm.block_table(s)[(len(toks[s]) - 1) // B] * B + (len(toks[s]) - 1) % B
            if pair is not None:
                cow.append(pair)
        if cow:
            cp = np.array(cow, np.int64)
            pa.copy_blocks([dk], [dv], torch.from_numpy(cp).cuda(), err_flag=err)
            assert ora.copy_blocks([kp], [vp], cp) == 0
        for s in live:
            write(toks[s], bm.block_table(s), len(toks[s]) - 1)
        bt = tables(live)
        ctx = np.array([len(toks[s]) for s in live], np.int32)
        if batch:
            bt2, lens = bm.block_tables(live, bt.shape[1], pad=-1)
            assert np.array_equal(bt2, bt) and np.array_equal(lens, ctx)
            bt = bt2
        q = wl.normal_bf16(st, (len(live), HQ, D))
        out = pa.paged_attention_decode(bf16_dev(q, torch), dk, dv, torch.from_numpy(bt).cuda(),
                                        torch.from_numpy(ctx).cuda(), scale=SCALE, max_context_len=int(ctx.max()),
                                        err_flag=err)
        torch.cuda.synchronize()
        ref, status = ora.decode(q, kp, vp, bt, ctx, SCALE)
        assert np.all(status == 0)
        assert_close(bf16_host(out), ref, f"decode step {step}")
    assert int(err.item()) == 0
    assert np.array_equal(bf16_host(dk), kp) and np.array_equal(bf16_host(dv), vp)
    assert np.array_equal(gk.view(torch.int16).numpy().view(np.uint16), hk)
    assert np.array_equal(gv.view(torch.int16).numpy().view(np.uint16), hv)
