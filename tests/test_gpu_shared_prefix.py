"""GPU parity of shared-prefix-aware decode: groups of sequences that share
their leading blocks have the prefix attended once on the tensor cores and
merged with each sequence's own keys.  Checked against the fp64 oracle and
against plain paged decode on the same inputs."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def grouped_case(Hq, Hkv, D, B, groups, ungrouped, seed):
    """groups: list of (members, prefix_len); each member gets a random suffix
    (0 .. 300 tokens); ungrouped: number of extra sequences without a shared
    prefix.  Returns a DecodeCase whose tables share the prefix blocks, plus
    the group arrays."""
    st = wl.Stream(seed, 31)
    rows, ctx, gstart, gpref, ptabs = [], [], [0], [], []
    nblk = 0
    for members, plen in groups:
        assert plen % B == 0
        prefix = list(range(nblk, nblk + plen // B))
        nblk += plen // B
        suf = st.integers(0, 300, members)
        suf[0] = 0  # one member ends exactly at the prefix
        for sfx in suf:
            n = plen + int(sfx)
            own = (n + B - 1) // B - len(prefix)
            rows.append(prefix + list(range(nblk, nblk + own)))
            nblk += own
            ctx.append(n)
        gstart.append(gstart[-1] + members)
        gpref.append(plen)
        ptabs.append(prefix)
    for n in st.integers(1, 400, ungrouped):
        k = (int(n) + B - 1) // B
        rows.append(list(range(nblk, nblk + k)))
        nblk += k
        ctx.append(int(n))
    nblk += 5
    perm = st.permutation(nblk).astype(np.int32)  # scatter the pages
    mb = max(len(r) for r in rows)
    bt = np.full((len(rows), mb), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, : len(r)] = perm[r]
    pmb = max(len(p) for p in ptabs)
    pt = np.full((len(ptabs), pmb), -1, np.int32)
    for i, p in enumerate(ptabs):
        pt[i, : len(p)] = perm[p]
    S = len(rows)
    case = wl.DecodeCase("grouped", S, Hq, Hkv, D, B, nblk, mb, 1.0 / math.sqrt(D), np.array(ctx, np.int32), bt,
                         wl.normal_bf16(st, (S, Hq, D)), wl.normal_bf16(st, (nblk, Hkv, B, D)),
                         wl.normal_bf16(st, (nblk, Hkv, B, D)))
    return case, np.array(gstart, np.int32), np.array(gpref, np.int32), pt


def run_both(torch, case, gs, gp, pt, err):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    q, kp, vp = bf16_dev(case.q, torch), bf16_dev(case.k_pool, torch), bf16_dev(case.v_pool, torch)
    bt, ctx = dev(case.block_tables), dev(case.context_lens)
    shared = pa.paged_attention_decode_shared_prefix(
        q, kp, vp, bt, ctx, dev(gs), dev(gp), dev(pt), max_group_size=int(np.diff(gs).max()),
        max_prefix_len=int(gp.max()), scale=case.scale, max_context_len=case.max_context_len, err_flag=err)
    plain = pa.paged_attention_decode(q, kp, vp, bt, ctx, scale=case.scale, max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    return bf16_host(shared), bf16_host(plain)


SHAPES = [(32, 8, 128, 16), (64, 8, 128, 32), (16, 16, 128, 16), (32, 2, 128, 16)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "q%dkv%dd%db%d" % s)
@pytest.mark.parametrize("pp", [None, 2])
def test_shared_prefix_small(torch, ora, monkeypatch, shape, pp):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    Hq, Hkv, D, B = shape
    case, gs, gp, pt = grouped_case(Hq, Hkv, D, B, [(5, 4 * B), (3, 10 * B), (1, B)], 3, seed=hash(shape) % 997)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shared, plain = run_both(torch, case, gs, gp, pt, err)
    assert int(err.item()) == 0
    ref, st = ora.decode_case(case)
    assert np.all(st == 0)
    assert_close(shared, ref, f"shared {shape} pp={pp}")
    assert_close(plain, ref, f"plain {shape} pp={pp}")


def test_shared_prefix_workload(torch, ora):
    """The prefix-sharing workload (256 sequences over one 2048-token prefix,
    copy-on-write suffixes): one group with the block manager's tables."""
    import bench
    plan, bt, ctx, slots, pairs = bench.prefix_sharing_setup(pa)
    kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
    if len(pairs):
        assert ora.copy_blocks([kp], [vp], pairs) == 0
    assert ora.reshape_and_cache(nk, nv, kp, vp, slots) == 0
    S, B = len(ctx), plan.B
    npre = plan.prefix_len // B
    assert np.all(bt[:, :npre] == bt[0, :npre])
    case = wl.DecodeCase("prefix", S, plan.Hq, plan.Hkv, plan.D, B, plan.num_blocks, bt.shape[1],
                         1 / math.sqrt(plan.D), ctx, bt, q, kp, vp)
    gs = np.array([0, S], np.int32)
    gp = np.array([plan.prefix_len], np.int32)
    pt = bt[:1, :npre].copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shared, plain = run_both(torch, case, gs, gp, pt, err)
    assert int(err.item()) == 0
    heads = [(s, h) for s in range(0, S, 5) for h in (0, 9, 31)]
    ref = ora.decode_case(case, heads=heads)
    assert_close(np.stack([shared[s, h] for s, h in heads]), ref, "shared prefix workload")
    # against plain decode on every output (both sides within tolerance of fp64)
    assert_close(shared, (plain.astype(np.uint32) << 16).view(np.float32).astype(np.float64), "shared vs plain")


def test_prefix_not_block_multiple_flagged(torch):
    case, gs, gp, pt = grouped_case(32, 8, 128, 16, [(3, 64)], 2, seed=5)
    gp = gp + 3  # not a whole number of blocks
    pt = np.concatenate([pt, pt[:, :1]], axis=1)  # room for the extra tokens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shared, plain = run_both(torch, case, gs, gp, pt, err)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(shared[:3])                  # the group's rows: zeros, as for any bad context
    assert np.array_equal(shared[3:], plain[3:])   # sequences outside the group: plain decode


@pytest.mark.parametrize("pp", [None, 2])
def test_shared_prefix_graph_replay(torch, monkeypatch, pp):
    """Captured once and replayed: the merge counters are reset by each merge,
    so every replay (same epoch) merges again and gives the same bits."""
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    case, gs, gp, pt = grouped_case(32, 8, 128, 16, [(6, 128), (2, 64)], 2, seed=11)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    q, kp, vp = bf16_dev(case.q, torch), bf16_dev(case.k_pool, torch), bf16_dev(case.v_pool, torch)
    bt, ctx, gsd, gpd, ptd = dev(case.block_tables), dev(case.context_lens), dev(gs), dev(gp), dev(pt)
    kw = dict(max_group_size=int(np.diff(gs).max()), max_prefix_len=int(gp.max()), scale=case.scale,
              max_context_len=case.max_context_len)
    want = bf16_host(pa.paged_attention_decode_shared_prefix(q, kp, vp, bt, ctx, gsd, gpd, ptd, **kw))
    out = torch.empty_like(q)
    desc = pa.make_desc(q, kp, bt, scale=case.scale, max_context_len=case.max_context_len)
    import ctypes
    need = int(pa.load().pa_shared_prefix_workspace_bytes(ctypes.byref(desc)))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            pa.paged_attention_decode_shared_prefix(q, kp, vp, bt, ctx, gsd, gpd, ptd, out, workspace=ws, **kw)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(out), want)
