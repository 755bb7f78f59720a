"""Block manager under hypothesis' stateful testing (host only).

Random programs of prompts (built from a tiny set of chunks, from an earlier
sequence's whole history, or from the appends' vocabulary, so that equal
blocks follow different
prefixes and cache hits are frequent), forks, appends with and without token
ids (drawn from a two-token vocabulary, so that generated blocks repeat
after other prefixes too), batch appends, frees and swaps run against
simulated device and host pools.  Each slot of the simulated pools holds a
fingerprint of its token and every token before it, as a key or value depends
on its whole prefix.  After every step every resident sequence must read back
its own fingerprints through its block table, every block's reference count
must equal the number of resident tables holding it, and the free counts must
add up.  Failures shrink to a minimal program."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import settings, strategies as st  # noqa: E402
from hypothesis.stateful import RuleBasedStateMachine, invariant, precondition, rule  # noqa: E402

import paged_kv_cache_262_gb300 as pa  # noqa: E402
from paged_kv_cache_262_gb300 import build as pbuild  # noqa: E402

B, N, H = 4, 20, 12
CHUNKS = [[10, 11, 12, 13], [20, 21, 22, 23], [30, 31, 32, 33]]


def fp(toks):
    out, h = [], 0
    for x in toks:
        h = (h * 1000003 + x + 1) % (1 << 61)
        out.append(h)
    return out


class BlockManagerMachine(RuleBasedStateMachine):
    def __init__(self):
        super().__init__()
        pbuild.build()
        self.bm = pa.BlockManager(N, B, num_host_blocks=H)
        self.dev = np.full((N, B), -1, np.int64)
        self.host = np.full((H, B), -1, np.int64)
        self.model, self.swapped, self.history = {}, set(), []
        self.next_id, self.next_tok = 0, 1000

    def fresh(self):
        self.next_tok += 1
        return self.next_tok

    def resident(self):
        return sorted(s for s in self.model if s not in self.swapped)

    def write(self, s, start):
        t, f = self.bm.block_table(s), fp(self.model[s])
        for j in range(start, len(self.model[s])):
            self.dev[t[j // B], j % B] = f[j]

    @rule(parts=st.lists(st.integers(0, 2), max_size=4), tail=st.integers(0, 3), mode=st.integers(0, 2),
          keep=st.integers(0, 40), small=st.lists(st.integers(0, 1), max_size=12))
    def admit(self, parts, tail, mode, keep, small):
        if mode == 1 and self.history:  # the next turn of an earlier sequence
            base = self.history[keep % len(self.history)]
            toks = base[: keep % (len(base) + 1)]
        elif mode == 2:  # the appends' vocabulary: may equal a generated block anywhere
            toks = list(small)
        else:
            toks = [x for p in parts for x in CHUNKS[p]]
        toks = toks + [self.fresh() for _ in range(tail)]
        if not toks:
            return
        try:
            c = self.bm.add_seq_tokens(self.next_id, toks)
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
            return
        assert c % B == 0 and 0 <= c <= len(toks)
        t = self.bm.block_table(self.next_id)
        f = fp(toks)
        assert [int(self.dev[t[j // B], j % B]) for j in range(c)] == f[:c]  # hits hold this prompt's prefix
        self.model[self.next_id] = list(toks)
        self.write(self.next_id, c)
        self.next_id += 1

    @precondition(lambda self: self.resident())
    @rule(i=st.integers(0, 1000))
    def fork(self, i):
        r = self.resident()
        p = r[i % len(r)]
        self.bm.fork(p, self.next_id)
        self.model[self.next_id] = list(self.model[p])
        self.next_id += 1

    def apply(self, s, slot, cow, tok):
        if cow is not None:
            self.dev[cow[1]] = self.dev[cow[0]]
        self.model[s].append(tok)
        self.dev[slot // B, slot % B] = fp(self.model[s])[-1]

    @precondition(lambda self: self.resident())
    @rule(i=st.integers(0, 1000), no_id=st.integers(0, 7), tok=st.integers(0, 1))
    def append(self, i, no_id, tok):
        r = self.resident()
        s = r[i % len(r)]
        try:
            slot, cow = self.bm.append(s, None if no_id == 0 else tok)  # the id given 7 times in 8
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
            return
        self.apply(s, slot, cow, tok)

    @precondition(lambda self: self.resident())
    @rule(mask=st.integers(1, 255), no_ids=st.integers(0, 7),
          vocab=st.lists(st.integers(0, 1), min_size=8, max_size=8))
    def append_batch(self, mask, no_ids, vocab):
        with_ids = no_ids != 0
        r = self.resident()
        sub = [s for k, s in enumerate(r) if mask >> (k % 8) & 1] or r[:1]
        toks = [vocab[k % 8] for k in range(len(sub))]
        try:
            sl, cw = self.bm.append_batch(sub, toks if with_ids else None)
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
            return
        for k, s in enumerate(sub):
            self.apply(s, int(sl[k]), None if cw[k, 0] < 0 else (int(cw[k, 0]), int(cw[k, 1])), toks[k])

    @precondition(lambda self: self.model)
    @rule(i=st.integers(0, 1000))
    def free(self, i):
        ids = sorted(self.model)
        s = ids[i % len(ids)]
        self.bm.free_seq(s)
        self.history.append(self.model.pop(s))
        self.swapped.discard(s)

    @precondition(lambda self: self.resident())
    @rule(i=st.integers(0, 1000))
    def swap_out(self, i):
        r = self.resident()
        s = r[i % len(r)]
        before = self.bm.block_table(s)
        try:
            pairs = self.bm.swap_out(s)
        except pa.PaError as e:
            assert e.status in (pa.PA_ERR_STATE, pa.PA_ERR_OOM) and self.bm.block_table(s) == before
            return
        assert [d for d, _ in pairs] == before
        for d, h in pairs:
            self.host[h] = self.dev[d]
        self.swapped.add(s)

    @precondition(lambda self: self.swapped)
    @rule(i=st.integers(0, 1000))
    def swap_in(self, i):
        sw = sorted(self.swapped)
        s = sw[i % len(sw)]
        try:
            pairs = self.bm.swap_in(s)
        except pa.PaError as e:
            assert e.status == pa.PA_ERR_OOM
            return
        for h, d in pairs:
            self.dev[d] = self.host[h]
        self.swapped.discard(s)

    @invariant()
    def contents_and_counts(self):
        refs = np.zeros(N, int)
        used_host = 0
        for s, toks in self.model.items():
            if s in self.swapped:
                used_host += (len(toks) + B - 1) // B
                continue
            t = self.bm.block_table(s)
            assert len(t) == (len(toks) + B - 1) // B and self.bm.seq_len(s) == len(toks)
            assert [int(self.dev[t[j // B], j % B]) for j in range(len(toks))] == fp(toks), s
            for b in t:
                refs[b] += 1
        assert [self.bm.ref_count(b) for b in range(N)] == refs.tolist()
        assert self.bm.num_free() == int((refs == 0).sum())
        assert self.bm.num_free_host() == H - used_host
        assert 0 <= self.bm.num_cached_blocks() <= N

    def teardown(self):
        self.bm.close()


TestBlockManagerStateful = BlockManagerMachine.TestCase
TestBlockManagerStateful.settings = settings(max_examples=150, stateful_step_count=40, deadline=None,
                                             derandomize=True)
