"""The seeded input generator: determinism, the C fast path against its numpy
definition, and the workload recipes' structure."""
import numpy as np

import workloads as wl


def test_splitmix_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += GAMMA; mix) are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    z = []
    state = 0
    for _ in range(2):
        state = (state + wl.GAMMA) & ((1 << 64) - 1)
        z.append(wl._mix64_int(state))
    assert z == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_c_fast_path_matches_numpy_definition():
    for seed, stream, n in ((0, 0, 1), (3, 7, 1001), (11, 2, 200_000)):
        a = wl.normal_bf16(wl.Stream(seed, stream), (n,))
        b = wl.normal_bf16_numpy(wl.Stream(seed, stream), (n,))
        assert np.array_equal(a, b)


def test_stream_continuation():
    s1 = wl.Stream(5, 5)
    a = wl.normal_bf16(s1, (10,))
    b = wl.normal_bf16(s1, (6,))
    s2 = wl.Stream(5, 5)
    c = wl.normal_bf16(s2, (16,))
    assert np.array_equal(np.concatenate([a, b]), c)


def test_normal_moments_and_bf16_rounding():
    x = wl.bf16_bits_to_f32(wl.normal_bf16(wl.Stream(1, 1), (400_000,))).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    # round-to-nearest-even on ties: 1 + 2^-8 (exactly between two bf16) -> 1.0
    assert wl.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert wl.f64_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82


def test_permutation_is_permutation():
    p = wl.Stream(2, 2).permutation(1000)
    assert np.array_equal(np.sort(p), np.arange(1000))


def test_tiny_decode_shape():
    c = wl.tiny_decode()
    assert list(c.context_lens) == [1, 17, 33, 100]
    assert c.num_blocks == 64 and c.head_dim == 64 and c.block_size == 16
    used = c.block_tables[c.block_tables >= 0]
    assert len(used) == 13 and len(set(used.tolist())) == 13
    # the new token of every sequence lands at position ctx-1
    for s, ctx in enumerate(c.context_lens):
        j = ctx - 1
        assert c.slot_mapping[s] == c.block_tables[s, j // 16] * 16 + j % 16


def test_llama8b_decode_shape():
    c = wl.llama8b_decode()
    assert c.num_seqs == 64 and c.num_q_heads == 32 and c.num_kv_heads == 8
    assert c.context_lens.min() >= 128 and c.context_lens.max() <= 2048
    used = c.block_tables[c.block_tables >= 0]
    assert len(set(used.tolist())) == len(used)
    assert c.num_blocks == int(np.ceil(1.25 * len(used)))


def test_mixed_step_shape():
    m = wl.make_mixed_step("t", [5, 7], [9, 30], [3, 40, 65], 4, 2, 16, 32)
    assert list(m.cu_q) == [0, 5, 12]
    # chunk rows are the last C tokens of each context
    for r in range(2):
        c0 = m.chunk_ctx[r] - m.chunk_lens[r]
        for i in range(m.chunk_lens[r]):
            j = c0 + i
            assert m.chunk_slots[m.cu_q[r] + i] == m.chunk_tables[r, j // 32] * 32 + j % 32


def test_sharing_workloads_subgroups():
    """The sub-group partition the bench forms for the two sharing workloads
    (from the host block manager's tables): consecutive, covering every
    sequence; members agree on their shared blocks; the shared length is whole
    blocks, at least the common prefix and at most every member's context; one
    block of each member's own at most (the copy made on its append)."""
    import bench
    import paged_kv_cache_262_gb300 as pa
    for plan in (None, wl.parallel_sampling_plan()):
        plan, bt, ctx, slots, pairs = bench.prefix_sharing_setup(pa, plan)
        ss, sh = bench.prefix_sharing_subgroups(plan, bt, ctx)
        B = plan.B
        assert ss[0] == 0 and ss[-1] == len(ctx) and np.all(np.diff(ss) >= 1)
        assert len(sh) == len(ss) - 1
        for k in range(len(sh)):
            a, b = ss[k], ss[k + 1]
            assert sh[k] % B == 0 and plan.prefix_len <= sh[k] <= ctx[a:b].min()
            assert np.all(bt[a:b, : sh[k] // B] == bt[a, : sh[k] // B])
            assert np.all(ctx[a:b] - sh[k] <= B)
        # the appended token of every sample went to a slot of its own last block
        for s in range(len(ctx)):
            assert slots[s] // B == bt[s, (ctx[s] - 1) // B]
