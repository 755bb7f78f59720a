"""Host block manager (plain C++, no GPU): on-demand allocation, sharing,
copy-on-write, free on <eos>, fragmentation bound, error states."""
import json
import os

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from paged_kv_cache_262_gb300 import build as pbuild

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    pbuild.build()


def test_block_table_example_1024_tokens():
    """'PagedAttention Architecture Deep Dive' example: 1024 tokens at 16 per
    page occupy 64 pages; a shared page has ref_count 2."""
    fx = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    bm = pa.BlockManager(200, fx["block_size"])
    bm.add_seq(0, fx["tokens"])
    t = bm.block_table(0)
    assert len(t) == fx["pages"]
    assert bm.num_free() == 200 - fx["pages"]
    bm.fork(0, 1)
    assert bm.ref_count(t[2]) == 2
    assert bm.wasted_slots() == 0


def test_on_demand_allocation_and_waste_bound():
    """ceil(n/B) blocks per sequence; at most B-1 unused slots per sequence,
    so waste stays under 4 % once sequences are long compared with B."""
    B = 16
    st = wl.Stream(3, 3)
    lens = st.integers(128, 2048, 64)
    bm = pa.BlockManager(int(sum((l + B - 1) // B for l in lens)), B)
    for i, n in enumerate(lens):
        bm.add_seq(i, int(n))
        assert len(bm.block_table(i)) == (n + B - 1) // B
    assert bm.num_free() == 0
    w = bm.wasted_slots()
    assert w == sum((-int(n)) % B for n in lens)
    assert w <= (B - 1) * len(lens)
    assert w / (w + lens.sum()) < 0.04
    tables = [bm.block_table(i) for i in range(len(lens))]
    flat = [b for t in tables for b in t]
    assert len(flat) == len(set(flat))  # no block given twice


def test_free_returns_all_blocks_and_reuses_them():
    bm = pa.BlockManager(10, 16)
    bm.add_seq(1, 40)
    bm.add_seq(2, 33)
    assert bm.num_free() == 10 - 3 - 3
    t1 = bm.block_table(1)
    bm.free_seq(1)
    assert bm.num_free() == 7
    assert all(bm.ref_count(b) == 0 for b in t1)
    bm.add_seq(3, 16)
    assert bm.block_table(3)[0] in t1  # freed pages are reused next
    bm.free_seq(2)
    bm.free_seq(3)
    assert bm.num_free() == 10


def test_fork_append_copy_on_write():
    B = 16
    bm = pa.BlockManager(32, B)
    bm.add_seq(0, 20)  # 2 blocks, last one holds 4 tokens
    for c in (1, 2, 3):
        bm.fork(0, c)
    t0 = bm.block_table(0)
    assert [bm.ref_count(b) for b in t0] == [4, 4]
    pairs = []
    for s in (0, 1, 2, 3):
        slot, pair = bm.append(s)
        t = bm.block_table(s)
        assert slot == t[1] * B + 4
        pairs.append(pair)
    # three sharers copy the partial block, the last one writes in place
    assert all(p is not None and p[0] == t0[1] for p in pairs[:3])
    assert pairs[3] is None
    assert len({p[1] for p in pairs[:3]}) == 3
    assert bm.ref_count(t0[1]) == 1 and bm.ref_count(t0[0]) == 4
    assert bm.seq_len(2) == 21
    # a full shared block needs no copy: the token opens a new block
    bm.add_seq(10, 32)
    bm.fork(10, 11)
    slot, pair = bm.append(11)
    assert pair is None and slot % B == 0 and bm.block_table(11)[:2] == bm.block_table(10)


def test_prefix_sharing_structure():
    """64 prompts x 4 samples over a 2048-token prefix: the prefix blocks end up
    with ref_count 256 and each partial last block is copied 3 times."""
    plan = wl.prefix_sharing_plan()
    B = plan.B
    bm = pa.BlockManager(plan.num_blocks, B)
    bm.add_seq(100000, plan.prefix_len)
    prefix = bm.block_table(100000)
    for p in range(plan.num_prompts):
        bm.fork(100000, p * 4)
        for _ in range(int(plan.suffix_lens[p])):
            slot, pair = bm.append(p * 4)
            assert pair is None
    bm.free_seq(100000)
    for p in range(plan.num_prompts):
        for i in (1, 2, 3):
            bm.fork(p * 4, p * 4 + i)
    assert all(bm.ref_count(b) == 256 for b in prefix)
    ncow = 0
    for s in range(plan.num_prompts * 4):
        _, pair = bm.append(s)
        ncow += pair is not None
    partial = sum(1 for x in plan.suffix_lens if (plan.prefix_len + int(x)) % B)
    assert ncow == 3 * partial


def test_errors_and_oom_leave_no_trace():
    bm = pa.BlockManager(4, 16)
    with pytest.raises(pa.PaError) as e:
        bm.add_seq(0, 80)
    assert e.value.status == pa.PA_ERR_OOM and bm.num_free() == 4
    bm.add_seq(0, 64)
    with pytest.raises(pa.PaError) as e:
        bm.append(0)
    assert e.value.status == pa.PA_ERR_OOM and bm.seq_len(0) == 64
    with pytest.raises(pa.PaError) as e:
        bm.add_seq(0, 1)
    assert e.value.status == pa.PA_ERR_STATE
    with pytest.raises(pa.PaError):
        bm.free_seq(7)
    with pytest.raises(pa.PaError):
        bm.fork(7, 8)
    bm.free_seq(0)
    with pytest.raises(pa.PaError):
        bm.free_seq(0)
    assert bm.ref_count(-1) == -1 and bm.ref_count(4) == -1
    with pytest.raises(pa.PaError):
        pa.BlockManager(0, 16)


def test_random_operations_keep_invariants():
    """Random add/fork/append/free: reference counts equal the number of tables
    that hold each block, free + referenced = pool, lengths match tables."""
    st = wl.Stream(21, 21)
    B, N = 16, 300
    bm = pa.BlockManager(N, B)
    live = {}
    nxt = 0
    u = st.uniform(4000)
    for k in range(4000):
        op = u[k]
        try:
            if op < 0.25 or not live:
                bm.add_seq(nxt, int(u[k] * 1e6) % 100)
                live[nxt] = True
                nxt += 1
            elif op < 0.4:
                p = list(live)[int(u[k] * 1e7) % len(live)]
                bm.fork(p, nxt)
                live[nxt] = True
                nxt += 1
            elif op < 0.85:
                s = list(live)[int(u[k] * 1e7) % len(live)]
                bm.append(s)
            else:
                s = list(live)[int(u[k] * 1e7) % len(live)]
                bm.free_seq(s)
                del live[s]
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
        if k % 97 == 0:
            refs = np.zeros(N, int)
            for s in live:
                t = bm.block_table(s)
                assert len(t) == (bm.seq_len(s) + B - 1) // B
                for b in t:
                    refs[b] += 1
            assert all(bm.ref_count(b) == refs[b] for b in range(N))
            assert bm.num_free() == int((refs == 0).sum())
    for s in list(live):
        bm.free_seq(s)
    assert bm.num_free() == N


def test_swap_out_and_in_move_blocks_between_pools():
    bm = pa.BlockManager(8, 16, num_host_blocks=6)
    bm.add_seq(1, 40)   # 3 blocks
    bm.add_seq(2, 20)   # 2 blocks
    t1 = bm.block_table(1)
    out = bm.swap_out(1)
    assert [d for d, _ in out] == t1 and len({h for _, h in out}) == 3
    assert bm.num_free() == 8 - 2 and bm.num_free_host() == 3
    assert all(bm.ref_count(b) == 0 for b in t1)
    with pytest.raises(pa.PaError) as e:
        bm.append(1)
    assert e.value.status == pa.PA_ERR_STATE
    with pytest.raises(pa.PaError):
        bm.block_table(1)
    back = bm.swap_in(1)
    assert [h for h, _ in back] == [h for _, h in out]
    assert bm.block_table(1) == [d for _, d in back] and bm.seq_len(1) == 40
    assert bm.num_free_host() == 6 and bm.num_free() == 8 - 5
    slot, _ = bm.append(1)  # usable again
    assert slot == bm.block_table(1)[2] * 16 + 8


def test_swap_refuses_shared_blocks_and_reports_oom_without_trace():
    bm = pa.BlockManager(10, 16, num_host_blocks=2)
    bm.add_seq(0, 32)
    bm.fork(0, 1)
    with pytest.raises(pa.PaError) as e:
        bm.swap_out(1)
    assert e.value.status == pa.PA_ERR_STATE
    bm.add_seq(5, 48)  # 3 blocks > 2 host blocks
    with pytest.raises(pa.PaError) as e:
        bm.swap_out(5)
    assert e.value.status == pa.PA_ERR_OOM
    assert bm.num_free_host() == 2 and len(bm.block_table(5)) == 3
    bm.add_seq(6, 20)
    bm.swap_out(6)
    bm.free_seq(6)  # freeing a swapped sequence returns its host blocks
    assert bm.num_free_host() == 2


def test_prefix_cache_reuses_full_blocks_of_identical_prefixes():
    """Automatic prefix caching: a prompt that repeats another prompt's leading
    full blocks points at the same physical blocks."""
    B = 16
    bm = pa.BlockManager(64, B)
    st = wl.Stream(40, 1)
    a = [int(x) for x in st.integers(0, 50000, 100)]       # 6 full blocks + 4 tokens
    assert bm.add_seq_tokens(0, a) == 0
    assert bm.num_cached_blocks() == 6
    assert bm.add_seq_tokens(1, a) == 96                    # every full block found
    ta, tb = bm.block_table(0), bm.block_table(1)
    assert ta[:6] == tb[:6] and ta[6] != tb[6]              # the partial block is private
    assert all(bm.ref_count(b) == 2 for b in ta[:6])
    c = a[:40] + [a[40] + 1] + a[41:]                       # differs inside block 2
    assert bm.add_seq_tokens(2, c) == 32
    assert bm.block_table(2)[:2] == ta[:2] and bm.block_table(2)[2] != ta[2]
    d = a[:5] + [a[5] + 1] + a[6:]                          # differs in block 0: no reuse at all
    assert bm.add_seq_tokens(3, d) == 0


def test_prefix_cache_survives_free_until_reallocated():
    B = 16
    bm = pa.BlockManager(10, B)
    p = list(range(64))                                     # 4 full blocks
    assert bm.add_seq_tokens(0, p) == 0
    t0 = bm.block_table(0)
    bm.free_seq(0)
    assert bm.num_free() == 10
    assert bm.add_seq_tokens(1, p) == 64                    # content still there
    assert bm.block_table(1) == t0 and bm.num_free() == 6
    bm.free_seq(1)
    bm.add_seq(2, 10 * B)                                   # takes every block: the cache is evicted
    assert bm.num_cached_blocks() == 0
    bm.free_seq(2)
    assert bm.add_seq_tokens(3, p) == 0


def test_prefix_cache_never_hands_out_a_block_twice():
    """Blocks freed, revived by a cache hit and freed again keep one free-list
    entry each."""
    B = 4
    bm = pa.BlockManager(6, B)
    p = list(range(8))
    for rnd in range(5):
        bm.add_seq_tokens(10 + rnd, p)
        bm.free_seq(10 + rnd)
    bm.add_seq(1, 6 * B)
    t = bm.block_table(1)
    assert sorted(t) == list(range(6))
    with pytest.raises(pa.PaError):
        bm.add_seq(2, 1)


def test_prefix_cache_never_serves_a_continuation_of_other_content():
    """A cached block's K/V were computed after its whole prefix.  Once the
    block before it holds other content, a prompt that matches the new
    content must not be given the old continuation."""
    bm = pa.BlockManager(2, 1)
    A, C, X = 100, 200, 300
    assert bm.add_seq_tokens(0, [A, C]) == 0               # A, then C after A
    bm.free_seq(0)                                          # both free, both still cached
    assert bm.num_cached_blocks() == 2
    assert bm.add_seq_tokens(1, [X]) == 0                   # evicts C-after-A, freed first
    assert bm.num_cached_blocks() == 2                      # A and X
    assert bm.add_seq_tokens(2, [X, C]) == 1                # only X is found
    assert bm.num_cached_blocks() == 2                      # X and C-after-X (A evicted for it)


def test_prefix_cache_eviction_order():
    """Free blocks holding no cached content are handed out before any cached
    one; cached free blocks go least recently freed first, which puts a
    prompt's later blocks before its earlier ones; a chain in use is never
    touched; hits stay exact throughout."""
    B = 2
    bm = pa.BlockManager(12, B)
    a, b, c, d = [1, 2], [3, 4], [5, 6], [7, 8]
    assert bm.add_seq_tokens(0, a + b + c) == 0             # blocks 0, 1, 2
    assert bm.add_seq_tokens(1, a + b + d) == 4             # d after b: block 3
    assert bm.add_seq_tokens(2, a + c) == 2                 # c after a: block 4
    assert bm.add_seq_tokens(3, d + d) == 0                 # blocks 5, 6, kept in use
    for s in (1, 2, 0):                                     # freed in this order: 3, 4, then 2, 1, 0
        bm.free_seq(s)
    assert bm.num_free() == 10 and bm.num_cached_blocks() == 7
    bm.add_seq(4, 5 * B)                                    # the 5 never-used blocks go first
    assert sorted(bm.block_table(4)) == [7, 8, 9, 10, 11] and bm.num_cached_blocks() == 7
    bm.add_seq(5, B)                                        # then the least recently freed: d after b
    assert bm.block_table(5) == [3] and bm.num_cached_blocks() == 6
    assert bm.add_seq_tokens(6, a + b + d) == 4             # d after b is gone; c after a is evicted for it
    assert bm.block_table(6)[2] == 4
    assert bm.add_seq_tokens(7, a + b + c) == 6             # the first prompt's chain is whole
    bm.free_seq(6)
    assert bm.add_seq_tokens(8, a + c) == 2                 # c after a was evicted
    assert bm.add_seq_tokens(9, d + d) == 4                 # the live chain, untouched


def _state(bm, ids, N):
    return ([bm.ref_count(b) for b in range(N)], bm.num_free(), bm.num_cached_blocks(),
            {s: (bm.seq_len(s), bm.block_table(s)) for s in ids})


def test_append_batch_equals_single_appends():
    """A decode step's appends in one call give the same slots, copy-on-write
    pairs, tables and reference counts as one call per sequence, through
    forks whose samples share a partial block (some of the sharers appending,
    or all of them) and sequences that open a new block."""
    B, N = 4, 256
    one, bat = pa.BlockManager(N, B), pa.BlockManager(N, B)
    st = wl.Stream(91, 1)
    u = st.uniform(4000)
    k = 0
    live = []
    for p in range(12):
        toks = [int(x) for x in st.integers(0, 1000, 1 + int(u[k] * 30))]
        k += 1
        for m in (one, bat):
            m.add_seq_tokens(100 * p, toks)
        live.append(100 * p)
        for i in range(1, 1 + p % 4):           # 0..3 samples per prompt
            for m in (one, bat):
                m.fork(100 * p, 100 * p + i)
            live.append(100 * p + i)
    for step in range(12):
        batch = [s for s in live if u[k + live.index(s)] < 0.8]  # most, not all, sequences this step
        k += len(live)
        sl, cw = bat.append_batch(batch)
        for i, s in enumerate(batch):
            slot, pair = one.append(s)
            assert sl[i] == slot, (step, s)
            assert (None if cw[i, 0] < 0 else (cw[i, 0], cw[i, 1])) == pair, (step, s)
        assert _state(one, live, N) == _state(bat, live, N)
    sl, cw = bat.append_batch([])
    assert sl.shape == (0,) and cw.shape == (0, 2)


def test_append_batch_checks_everything_first():
    B = 4
    bm = pa.BlockManager(8, B, num_host_blocks=4)
    bm.add_seq(0, 6)                          # 2 blocks, the last half full
    bm.fork(0, 1)
    bm.fork(0, 2)                             # the partial block: ref_count 3
    bm.add_seq(3, 4)                          # full: its next token opens a block
    bm.add_seq(4, 1)
    bm.swap_out(4)
    before = _state(bm, [0, 1, 2, 3], 8)
    assert bm.num_free() == 5
    for ids, status in (([0, 9], pa.PA_ERR_STATE), ([0, 4], pa.PA_ERR_STATE), ([0, 1, 0], pa.PA_ERR_INVALID)):
        with pytest.raises(pa.PaError) as e:
            bm.append_batch(ids)
        assert e.value.status == status and _state(bm, [0, 1, 2, 3], 8) == before
    # all three sharers append: 2 copies (the last keeps the block) + 1 new block = 3 blocks
    bm.add_seq(5, 2 * B)                      # leaves exactly 3 free
    before = _state(bm, [0, 1, 2, 3, 5], 8)
    bm.add_seq(6, 1)                          # leaves 2: one short
    with pytest.raises(pa.PaError) as e:
        bm.append_batch([0, 1, 2, 3])
    assert e.value.status == pa.PA_ERR_OOM
    bm.free_seq(6)
    assert _state(bm, [0, 1, 2, 3, 5], 8) == before
    sl, cw = bm.append_batch([0, 1, 2, 3])
    assert bm.num_free() == 0
    assert (cw[:, 0] >= 0).tolist() == [True, True, False, False]
    assert len({int(x) // B for x in sl[:3]}) == 3          # three different blocks now


def test_block_tables_matrix():
    B = 16
    bm = pa.BlockManager(64, B, num_host_blocks=8)
    lens = [1, 16, 17, 100, 0]
    for s, n in enumerate(lens):
        bm.add_seq(s, n)
    t, l = bm.block_tables([3, 0, 4, 2], 8, pad=-7)
    assert l.tolist() == [100, 1, 0, 17]
    for row, s in zip(t, [3, 0, 4, 2]):
        bt = bm.block_table(s)
        assert row[: len(bt)].tolist() == bt and (row[len(bt):] == -7).all()
    with pytest.raises(pa.PaError) as e:
        bm.block_tables([3], 6)                  # 100 tokens need 7 blocks
    assert e.value.status == pa.PA_ERR_INVALID
    bm.swap_out(1)
    for ids in ([1], [99]):
        with pytest.raises(pa.PaError) as e:
            bm.block_tables(ids, 8)
        assert e.value.status == pa.PA_ERR_STATE
    t, l = bm.block_tables([], 8)
    assert t.shape == (0, 8) and l.shape == (0,)


def test_batch_calls_reject_bad_arguments_through_the_c_abi():
    import ctypes
    bm = pa.BlockManager(8, 4)
    bm.add_seq(0, 3)
    lib, h = bm._lib, bm._h
    ids = np.array([0], np.int32)
    slots, cows = np.zeros(1, np.int64), np.zeros((1, 2), np.int64)
    out, lens = np.zeros((1, 4), np.int32), np.zeros(1, np.int32)
    P = lambda a: a.ctypes.data  # noqa: E731
    assert lib.pa_bm_append_batch(None, P(ids), None, 1, P(slots), P(cows)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_append_batch(h, P(ids), None, -1, P(slots), P(cows)) == pa.PA_ERR_INVALID
    for args in ((None, P(slots), P(cows)), (P(ids), None, P(cows)), (P(ids), P(slots), None)):
        assert lib.pa_bm_append_batch(h, args[0], None, 1, args[1], args[2]) == pa.PA_ERR_INVALID
    assert lib.pa_bm_append_batch(h, None, None, 0, None, None) == pa.PA_OK
    assert lib.pa_bm_block_tables(None, P(ids), 1, P(out), 4, 0, P(lens)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_block_tables(h, P(ids), -1, P(out), 4, 0, P(lens)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_block_tables(h, P(ids), 1, P(out), -1, 0, P(lens)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_block_tables(h, None, 1, P(out), 4, 0, P(lens)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_block_tables(h, P(ids), 1, None, 4, 0, P(lens)) == pa.PA_ERR_INVALID
    assert lib.pa_bm_block_tables(h, P(ids), 1, P(out), 4, 9, None) == pa.PA_OK  # lengths optional
    assert out[0].tolist() == [bm.block_table(0)[0], 9, 9, 9]
    assert bm.seq_len(0) == 3 and bm.num_free() == 7                              # nothing appended


def test_swapped_out_prompt_keeps_its_earlier_blocks_longest():
    """A swapped-out sequence's device blocks are freed last to first, as by
    free_seq: reusing one of them evicts the prompt's last cached block, and
    the earlier ones stay findable."""
    B = 4
    bm = pa.BlockManager(4, B, num_host_blocks=4)
    p = list(range(12))                                      # 3 full blocks, all cached
    bm.add_seq_tokens(0, p)
    bm.add_seq(1, B)                                         # the pool's last never-used block
    bm.swap_out(0)
    assert bm.num_free() == 3 and bm.num_cached_blocks() == 3
    bm.add_seq(2, B)                                         # evicts the third block, a leaf
    assert bm.num_cached_blocks() == 2
    assert bm.add_seq_tokens(3, p[:8]) == 8


def test_generated_blocks_serve_the_next_turn():
    """A conversation's second turn repeats the first turn's prompt and the
    answer generated for it.  Appends that give the token ids register every
    block they fill, so the second turn finds the answer's full blocks too;
    without the ids only the first prompt's full blocks are found."""
    B = 8
    st = wl.Stream(61, 1)
    p1 = [int(x) for x in st.integers(0, 1000, 37)]          # 4 full blocks + 5 tokens
    ans = [int(x) for x in st.integers(0, 1000, 20)]         # fills blocks 4, 5, 6; 1 token into block 7
    msg = [int(x) for x in st.integers(0, 1000, 10)]
    for with_ids, want in ((True, 56), (False, 32)):
        bm = pa.BlockManager(64, B)
        assert bm.add_seq_tokens(0, p1) == 0
        for t in ans:
            bm.append(0, t if with_ids else None)
        t0 = bm.block_table(0)
        assert bm.num_cached_blocks() == (7 if with_ids else 4)
        bm.free_seq(0)
        assert bm.add_seq_tokens(1, p1 + ans + msg) == want
        assert bm.block_table(1)[: want // B] == t0[: want // B]
    # an append without its id ends the registering: block 4, filled by the
    # third append, is registered; blocks 5 and 6 are not
    bm = pa.BlockManager(64, B)
    bm.add_seq_tokens(0, p1)
    for i, t in enumerate(ans):
        bm.append(0, None if i == 5 else t)
    assert bm.num_cached_blocks() == 5
    bm.free_seq(0)
    assert bm.add_seq_tokens(1, p1 + ans + msg) == 40


def test_conversations_find_every_full_block_of_their_history():
    """Six conversations over five turns, each turn's answer sampled twice
    (a fork; the first sample is kept) with token ids given to every
    append.  With a pool large enough that nothing is evicted, each turn's
    prompt -- the history so far plus a new message -- finds exactly the
    history's full blocks: the earlier prompts' blocks, the blocks the kept
    answers filled, and the block where an answer continued its prompt."""
    B = 16
    bm = pa.BlockManager(4096, B)
    st = wl.Stream(63, 1)
    ints = lambda n: [int(x) for x in st.integers(0, 30000, n)]  # noqa: E731
    hist = {c: [] for c in range(6)}
    sid = 0
    for turn in range(5):
        for c in hist:
            toks = hist[c] + ints(5 + int(st.integers(0, 36, 1)[0]))
            assert bm.add_seq_tokens(sid, toks) == len(hist[c]) // B * B, (turn, c)
            bm.fork(sid, sid + 1)
            n = 1 + int(st.integers(0, 50, 1)[0])
            kept, other = ints(n), ints(n)
            bm.append_batch([sid, sid + 1], [kept[0], other[0]])
            for x, y in zip(kept[1:], other[1:]):
                bm.append(sid, x)
                bm.append(sid + 1, y)
            hist[c] = toks + kept
            bm.free_seq(sid)
            bm.free_seq(sid + 1)
            sid += 2
    assert bm.num_free() == 4096


def test_forked_samples_register_their_own_continuations():
    B = 4
    bm = pa.BlockManager(64, B)
    prompt = list(range(100, 110))                             # 2 full blocks + 2 tokens
    bm.add_seq_tokens(0, prompt)
    bm.fork(0, 1)
    a, b = [1, 2, 3, 4, 5, 6], [7, 8, 9, 10, 11, 12]
    for x, y in zip(a, b):
        bm.append(0, x)                                        # the first copies the shared partial block
        bm.append(1, y)
    assert bm.num_cached_blocks() == 2 + 2 * 2                 # each sample filled blocks 2 and 3
    bm.free_seq(0)
    bm.free_seq(1)
    assert bm.add_seq_tokens(2, prompt + a + [0]) == 16
    assert bm.add_seq_tokens(3, prompt + b + [0]) == 16
    assert bm.add_seq_tokens(4, prompt + a[:2] + b[2:] + [0]) == 12  # the samples' blocks 2 differ


def test_append_batch_with_ids_equals_single_appends_with_ids():
    B, N = 4, 128
    one, bat = pa.BlockManager(N, B), pa.BlockManager(N, B)
    st = wl.Stream(62, 1)
    for m in (one, bat):
        m.add_seq_tokens(0, list(range(9)))
        m.fork(0, 1)
        m.add_seq_tokens(2, list(range(50, 53)))
        m.add_seq(3, 5)                                        # ids unknown: never registered
    ids = [0, 1, 2, 3]
    for step in range(11):
        tok = [int(x) for x in st.integers(0, 1000, 4)]
        sl, cw = bat.append_batch(ids, tok)
        for i, s in enumerate(ids):
            slot, pair = one.append(s, tok[i])
            assert sl[i] == slot and (None if cw[i, 0] < 0 else (cw[i, 0], cw[i, 1])) == pair
        assert _state(one, ids, N) == _state(bat, ids, N)
    assert bat.num_cached_blocks() == 2 + 3 + 3 + 3            # prompt 0; 3 more each for 0, 1 and 2
    with pytest.raises(ValueError):
        bat.append_batch(ids, tok[:3])


def test_failed_allocations_leave_no_trace(tmp_path):
    """Every host allocation inside every block-manager call made to fail in
    turn (a replaced operator new, in a C++ driver built with the block
    manager's source): each failure comes back as an error status, never as a
    C++ exception through the C ABI, and leaves the manager as it was."""
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    exe = str(tmp_path / "bm_alloc_fail")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "bm_alloc_fail.cpp"),
                    os.path.join(root, "paged_kv_cache_262_gb300", "csrc", "pa_block_manager.cpp"),
                    "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok ") and int(r.stdout.split()[1]) >= 20, r.stdout


@pytest.mark.parametrize("N,batch,ids", [(24, False, False), (64, False, False), (24, True, False), (64, True, False),
                                         (24, False, True), (64, False, True), (24, True, True), (64, True, True)])
def test_model_based_contents_through_cow_swap_and_prefix_cache(N, batch, ids):
    """Random prompts (some repeating earlier prompts' leading blocks), forks,
    appends, frees, swap-outs and swap-ins against simulated device and host
    page pools.  The test plays the caller: it writes each new token into the
    slot the manager gives, applies every copy-on-write pair and every swap
    pair to the simulated pools, and after each operation reads every resident
    sequence back through its block table: the tokens must be exactly the
    sequence's own, and each block's reference count must equal the number of
    resident tables holding it.  A slot holds what a key or value depends on:
    the token and every token before it (a fingerprint of the prefix), so a
    prefix-cache hit on a block whose content was computed after another
    prefix fails the read-back.  With `batch`, appends go to a random subset
    of the resident sequences in one append_batch call, and the step's copies
    and writes are applied in the batch's order.  With `ids`, most appends
    give their token id (so the blocks they fill enter the prefix cache) and
    some prompts continue a live or freed sequence's whole history, as a
    conversation's next turn does."""
    B, H = 8, 24
    bm = pa.BlockManager(N, B, num_host_blocks=H)
    dev = np.full((N, B), -1, np.int64)
    host = np.full((H, B), -1, np.int64)
    model, swapped = {}, set()
    st = wl.Stream(77, 3)
    u = st.uniform(3000)
    fresh = iter(range(10 ** 6, 10 ** 7))
    chunks = [[next(fresh) for _ in range(B)] for _ in range(4)]
    history = []  # the token lists of freed sequences
    prompts = []
    nxt = 0

    def fp(toks):  # per position: a fingerprint of toks[:j + 1]
        out, h = [], 0
        for x in toks:
            h = (h * 1000003 + x + 1) % (1 << 61)
            out.append(h)
        return out

    def write(s, start):
        t = bm.block_table(s)
        f = fp(model[s])
        for j in range(start, len(model[s])):
            dev[t[j // B], j % B] = f[j]

    def check_all():
        refs = np.zeros(N, int)
        for s, toks in model.items():
            if s in swapped:
                continue
            t = bm.block_table(s)
            assert len(t) == (len(toks) + B - 1) // B and bm.seq_len(s) == len(toks)
            assert [int(dev[t[j // B], j % B]) for j in range(len(toks))] == fp(toks), f"seq {s}"
            for b in t:
                refs[b] += 1
        assert all(bm.ref_count(b) == refs[b] for b in range(N))

    def pick(pred=lambda s: True):
        c = [s for s in model if pred(s)]
        return c[int(u[k] * 1e7) % len(c)] if c else None

    for k in range(3000):
        op = u[(k * 7919) % 3000]
        try:
            if op < 0.2 or not model:
                if prompts and op < 0.08:  # repeat some full blocks of an earlier prompt
                    base = prompts[int(u[k] * 1e6) % len(prompts)]
                    keep = (int(u[k] * 1e8) % (len(base) // B + 1)) * B
                    toks = base[:keep] + [next(fresh) for _ in range(int(u[k] * 1e5) % 20)]
                elif ids and 0.16 <= op < 0.19:  # the next turn of a conversation
                    cands = history + [model[x] for x in sorted(model)]
                    base = cands[int(u[k] * 1e6) % len(cands)]
                    keep = int(u[k] * 1e8) % (len(base) + 1)
                    toks = base[:keep] + [next(fresh) for _ in range(int(u[k] * 1e5) % 12)]
                elif op < 0.16:  # blocks from a small set in any order: equal blocks after other prefixes
                    n = 1 + int(u[k] * 1e3) % 5
                    toks = [x for i in range(n) for x in chunks[int(u[k] * 10 ** (4 + i)) % len(chunks)]]
                    toks += [next(fresh) for _ in range(int(u[k] * 1e5) % 4 == 3)]
                else:
                    toks = [next(fresh) for _ in range(1 + int(u[k] * 1e5) % 40)]
                if not toks:
                    toks = [next(fresh)]
                c = bm.add_seq_tokens(nxt, toks)
                assert c % B == 0 and 0 <= c <= len(toks)
                model[nxt] = list(toks)
                t = bm.block_table(nxt)
                assert [int(dev[t[j // B], j % B]) for j in range(c)] == fp(toks)[:c]  # cached blocks hold the prompt
                write(nxt, c)
                prompts.append(list(toks))
                nxt += 1
            elif op < 0.27:
                p = pick(lambda s: s not in swapped)
                if p is not None:
                    bm.fork(p, nxt)
                    model[nxt] = list(model[p])
                    nxt += 1
            elif op < 0.6 and batch:
                res = [s for s in model if s not in swapped]
                sub = [s for i, s in enumerate(res) if u[(k * 31 + i) % 3000] < 0.5]
                if sub:
                    new = [next(fresh) for _ in sub]
                    sl, cw = bm.append_batch(sub, new if ids else None)
                    for i, s in enumerate(sub):
                        if cw[i, 0] >= 0:
                            dev[cw[i, 1]] = dev[cw[i, 0]]
                        model[s].append(new[i])
                        dev[sl[i] // B, sl[i] % B] = fp(model[s])[-1]
            elif op < 0.6:
                s = pick(lambda s: s not in swapped)
                if s is not None:
                    tok = next(fresh)
                    slot, cow = bm.append(s, tok if ids and u[(k * 17) % 3000] < 0.95 else None)
                    if cow is not None:
                        dev[cow[1]] = dev[cow[0]]
                    model[s].append(tok)
                    dev[slot // B, slot % B] = fp(model[s])[-1]
            elif op < 0.78:
                s = pick()
                if s is not None:
                    bm.free_seq(s)
                    history.append(model[s])
                    del model[s]
                    swapped.discard(s)
            elif op < 0.89:
                s = pick(lambda s: s not in swapped)
                if s is not None:
                    before = bm.block_table(s)
                    try:
                        pairs = bm.swap_out(s)
                    except pa.PaError as e:
                        assert e.status in (pa.PA_ERR_STATE, pa.PA_ERR_OOM)
                        assert bm.block_table(s) == before
                    else:
                        assert [d for d, _ in pairs] == before
                        for d, h in pairs:
                            host[h] = dev[d]
                        swapped.add(s)
            else:
                s = pick(lambda s: s in swapped)
                if s is not None:
                    pairs = bm.swap_in(s)
                    for h, d in pairs:
                        dev[d] = host[h]
                    swapped.discard(s)
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
        check_all()
    for s in list(model):
        bm.free_seq(s)
    assert bm.num_free() == N and bm.num_free_host() == H


def test_block_manager_benchmark_runs():
    """bench.py --workload block_manager (host only): one pass of admission with
    prefix-cache hits, forks, copy-on-write appends, swaps and frees."""
    import types

    import bench
    res = bench.run_block_manager(types.SimpleNamespace(steps=1, warmup=0))
    assert res["value"] > 0 and res["gpu_launches"] == 0
    # every prompt after the first finds the 2048-token system prompt cached (whole blocks)
    assert 0.5 < res["cached_fraction"] < 1.0
    assert 0.0 < res["ops_per_s"]["copy_on_write_share"] <= 1.0
    # the next turn finds its history, including blocks the decode steps filled (their ids given)
    assert res["next_turn"]["cached_fraction"] > res["cached_fraction"]
    assert res["next_turn"]["tokens_found_in_blocks_decode_filled_per_prompt"] > 0
    assert res["decode_step_host_us"]["steady"] > 0
