"""Conversation turns through the host block manager, with the fp64 oracle
doing the cache writes and the attention (host only, no GPU).

Each position's K/V is a function of the tokens up to it, as a model's are.
Two conversations run three turns each; every turn's answer is sampled twice
(a fork, the first sample kept), its tokens appended with their ids, their
K/V written into the slots the manager gives (copy-on-write pairs applied
first).  Each turn's prompt -- the history so far plus a new message -- must
find exactly the history's full blocks in the cache (earlier prompts, the
answers' blocks, the block where an answer continued its prompt), and the
oracle's attention for the new tokens over that cache must equal, bit for
bit, its attention over a cache where the same prompt was written from
scratch."""
import numpy as np

import paged_kv_cache_262_gb300 as pa
import workloads as wl

B, HQ, HKV, D = 16, 4, 2, 64
N = 256
SCALE = 0.125


def test_next_turn_over_the_cache_equals_from_scratch(ora):
    st = wl.Stream(71, 2)
    bm = pa.BlockManager(N, B)
    kp, vp = np.zeros((N, HKV, B, D), np.uint16), np.zeros((N, HKV, B, D), np.uint16)
    kv_of = {}

    def kv(toks, j):
        key = tuple(toks[: j + 1])
        if key not in kv_of:
            kv_of[key] = (wl.normal_bf16(st, (HKV, D)), wl.normal_bf16(st, (HKV, D)))
        return kv_of[key]

    def write(toks, table, first, k_pool, v_pool):
        js = range(first, len(toks))
        k = np.stack([kv(toks, j)[0] for j in js])
        v = np.stack([kv(toks, j)[1] for j in js])
        slots = np.array([table[j // B] * B + j % B for j in js], np.int64)
        assert ora.reshape_and_cache(k, v, k_pool, v_pool, slots) == 0

    def attend(q, toks, table, k_pool, v_pool):
        C = q.shape[0]
        cu, bt, ctx = np.array([0, C], np.int32), np.array([table], np.int32), np.array([len(toks)], np.int32)
        out = []
        for i in sorted({0, C // 2, C - 1}):
            for h in range(HQ):
                o, status = ora.prefill_row(q, cu, k_pool, v_pool, bt, ctx, SCALE, 0, i, h)
                assert status == 0
                out.append(o)
        return np.stack(out)

    hist = {0: [], 1: []}
    sid = 0
    for turn in range(3):
        for c in hist:
            toks = hist[c] + [int(x) for x in st.integers(0, 30000, 20 + 7 * turn)]
            cached = bm.add_seq_tokens(sid, toks)
            assert cached == len(hist[c]) // B * B, (turn, c)
            table = bm.block_table(sid)
            write(toks, table, cached, kp, vp)
            fresh = pa.BlockManager(N, B)  # the same prompt written into an empty cache
            fresh.add_seq_tokens(0, toks)
            fk, fv = np.zeros_like(kp), np.zeros_like(vp)
            write(toks, fresh.block_table(0), 0, fk, fv)
            q = wl.normal_bf16(st, (len(toks) - cached, HQ, D))
            assert np.array_equal(attend(q, toks, table, kp, vp), attend(q, toks, fresh.block_table(0), fk, fv))
            # the answer, sampled twice
            bm.fork(sid, sid + 1)
            seqs = {s: list(toks) for s in (sid, sid + 1)}
            n = 5 + 9 * turn
            answers = {s: [int(x) for x in st.integers(0, 30000, n)] for s in seqs}
            for step in range(n):
                for s in seqs:
                    tok = answers[s][step]
                    slot, cow = bm.append(s, tok)
                    if cow is not None:
                        assert ora.copy_blocks([kp], [vp], np.array([cow], np.int64)) == 0
                    seqs[s].append(tok)
                    k, v = kv(seqs[s], len(seqs[s]) - 1)
                    assert ora.reshape_and_cache(k[None], v[None], kp, vp, np.array([slot], np.int64)) == 0
            hist[c] = seqs[sid]
            bm.free_seq(sid)
            bm.free_seq(sid + 1)
            sid += 2
    assert bm.num_free() == N
