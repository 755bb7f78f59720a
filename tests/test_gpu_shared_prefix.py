"""GPU parity of shared-prefix-aware decode: groups of sequences that share
their leading blocks have the prefix attended once on the tensor cores and
merged with each sequence's own keys.  Checked against the fp64 oracle and
against plain paged decode on the same inputs."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu, oracle_rows, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.fixture(params=["auto", "tasks", "units", "wide"])
def decode_kernel(request, monkeypatch):
    """The second launch of the shared-prefix decode: the library's choice,
    the task-queue kernel, one CTA per unit, or the tensor-core (wide-group)
    kernel, forced."""
    monkeypatch.delenv("PA_DECODE_TASKS", raising=False)
    monkeypatch.delenv("PA_DECODE_WIDE", raising=False)
    if request.param == "tasks":
        monkeypatch.setenv("PA_DECODE_TASKS", "1")
    elif request.param == "units":
        monkeypatch.setenv("PA_DECODE_TASKS", "0")
        monkeypatch.setenv("PA_DECODE_WIDE", "0")
    elif request.param == "wide":
        monkeypatch.setenv("PA_DECODE_WIDE", "1")
    return request.param


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
def test_shared_prefix_small(torch, ora, monkeypatch, shape, pp, decode_kernel):
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
    ref = oracle_rows(ora, case).reshape(shared.shape)
    assert_close(shared, ref, "shared prefix workload")
    # against plain decode on every output (both sides within tolerance of fp64)
    assert_close(shared, (plain.astype(np.uint32) << 16).view(np.float32).astype(np.float64), "shared vs plain")


def test_prefix_not_block_multiple_flagged(torch, decode_kernel):
    case, gs, gp, pt = grouped_case(32, 8, 128, 16, [(3, 64)], 2, seed=5)
    gp = gp + 3  # not a whole number of blocks
    pt = np.concatenate([pt, pt[:, :1]], axis=1)  # room for the extra tokens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shared, plain = run_both(torch, case, gs, gp, pt, err)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(shared[:3])                  # the group's rows: zeros, as for any bad context
    # sequences outside the group: decoded as usual (plain decode's result, within rounding)
    assert_close(shared[3:], to_f64(plain[3:]), "sequences outside the bad group")


@pytest.mark.parametrize("pp", [None, 2])
def test_shared_prefix_graph_replay(torch, monkeypatch, pp, decode_kernel):
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


def nested_case(Hq, Hkv, D, B, spec, seed):
    """Two levels of sharing.  spec: list of (prefix_blocks or None, subgroups)
    where subgroups is a list of (extra_shared_blocks, [own tokens per
    member]); prefix None = sub-groups outside every group.  Members of a
    sub-group share the group prefix plus its extra blocks, then have their own
    blocks.  Returns the case, the group arrays and the sub-group arrays."""
    st = wl.Stream(seed, 41)
    rows, ctx, gstart, gpref, ptabs, sstart, sshared = [], [], [], [], [], [0], []
    nblk, gend = 0, 0
    for pblocks, subs in spec:
        prefix = list(range(nblk, nblk + (pblocks or 0)))
        nblk += len(prefix)
        first = len(rows)
        for extra, owns in subs:
            shared = prefix + list(range(nblk, nblk + extra))
            nblk += extra
            for own in owns:
                n = len(shared) * B + own
                k = (n + B - 1) // B - len(shared)
                rows.append(shared + list(range(nblk, nblk + k)))
                nblk += k
                ctx.append(n)
            sstart.append(len(rows))
            sshared.append(len(shared) * B)
        if pblocks:
            gstart.append(first)
            gpref.append(pblocks * B)
            ptabs.append(prefix)
            gend = len(rows)
    if gpref:  # grouped entries come first, consecutive
        gstart.append(gend)
    nblk += 5
    perm = st.permutation(nblk).astype(np.int32)
    mb = max(len(r) for r in rows)
    bt = np.full((len(rows), mb), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, : len(r)] = perm[r]
    S = len(rows)
    case = wl.DecodeCase("nested", S, Hq, Hkv, D, B, nblk, mb, 1.0 / math.sqrt(D), np.array(ctx, np.int32), bt,
                         wl.normal_bf16(st, (S, Hq, D)), wl.normal_bf16(st, (nblk, Hkv, B, D)),
                         wl.normal_bf16(st, (nblk, Hkv, B, D)))
    if gpref:
        pmb = max(len(p) for p in ptabs)
        pt = np.full((len(ptabs), pmb), -1, np.int32)
        for i, p in enumerate(ptabs):
            pt[i, : len(p)] = perm[p]
    else:
        pt = np.zeros((1, 1), np.int32)
    return (case, np.array(gstart, np.int32), np.array(gpref, np.int32), pt, np.array(sstart, np.int32),
            np.array(sshared, np.int32))


def nested_inputs(torch, case, gs, gp, pt, ss, sh):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    ng = len(gp)
    return dict(q=bf16_dev(case.q, torch), kp=bf16_dev(case.k_pool, torch), vp=bf16_dev(case.v_pool, torch),
                bt=dev(case.block_tables), ctx=dev(case.context_lens), gs=dev(gs if ng else np.zeros(1, np.int32)),
                gp=dev(gp if ng else np.zeros(0, np.int32)), pt=dev(pt), ss=dev(ss), sh=dev(sh),
                kw=dict(max_group_size=int(np.diff(gs).max()) if ng else 0,
                        max_prefix_len=int(gp.max()) if ng else 0, scale=case.scale,
                        max_context_len=case.max_context_len, max_subgroup_size=int(np.diff(ss).max())))


def launch_nested(x, err=None, out=None, workspace=None):
    return pa.paged_attention_decode_shared_prefix(
        x["q"], x["kp"], x["vp"], x["bt"], x["ctx"], x["gs"], x["gp"], x["pt"], out, err_flag=err,
        subgroup_starts=x["ss"], subgroup_shared_lens=x["sh"], workspace=workspace, **x["kw"])


def run_nested(torch, case, gs, gp, pt, ss, sh, err):
    res = launch_nested(nested_inputs(torch, case, gs, gp, pt, ss, sh), err)
    torch.cuda.synchronize()
    return bf16_host(res)


NESTED = {
    # G = 4: sub-groups of up to 4 members (16 query rows); one member ends where its sub-group's sharing ends
    (32, 8, 128, 16): [(4, [(3, [1, 9, 16, 0]), (0, [5, 30]), (2, [17])]), (10, [(1, [3, 3, 40])]),
                       (None, [(2, [4, 7]), (0, [100])])],
    (64, 8, 128, 32): [(3, [(2, [5, 40]), (1, [1])]), (None, [(0, [70]), (1, [2, 33])])],
    # G = 1: sixteen members in one sub-group
    (16, 16, 128, 16): [(2, [(1, list(range(1, 17))), (0, [20])])],
    # G = 16: one member per sub-group
    (32, 2, 128, 16): [(5, [(2, [9]), (0, [1]), (3, [0])])],
}


@pytest.mark.parametrize("shape", list(NESTED), ids=lambda s: "q%dkv%dd%db%d" % s)
@pytest.mark.parametrize("pp", [None, 2])
def test_subgroups_against_oracle(torch, ora, monkeypatch, shape, pp, decode_kernel):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))  # the group prefix pass splits; sub-groups do not
    Hq, Hkv, D, B = shape
    case, gs, gp, pt, ss, sh = nested_case(Hq, Hkv, D, B, NESTED[shape], seed=sum(shape))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_nested(torch, case, gs, gp, pt, ss, sh, err)
    assert int(err.item()) == 0
    ref, st = ora.decode_case(case)
    assert np.all(st == 0)
    assert_close(got, ref, f"sub-groups {shape} pp={pp}")


def test_subgroup_bad_shared_length_flagged(torch, decode_kernel):
    spec = [(4, [(2, [3, 5]), (1, [8, 9])])]
    case, gs, gp, pt, ss, sh = nested_case(32, 8, 128, 16, spec, seed=3)
    sh = sh.copy()
    sh[0] += 5  # not a whole number of blocks
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_nested(torch, case, gs, gp, pt, ss, sh, err)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(got[:2])  # the bad sub-group's members: zeros
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    plain = pa.paged_attention_decode(bf16_dev(case.q, torch), bf16_dev(case.k_pool, torch),
                                      bf16_dev(case.v_pool, torch), dev(case.block_tables), dev(case.context_lens),
                                      scale=case.scale, max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    assert_close(got[2:], to_f64(bf16_host(plain)[2:]), "the other sub-group")


def test_subgroups_graph_replay(torch, decode_kernel):
    case, gs, gp, pt, ss, sh = nested_case(32, 8, 128, 16, NESTED[(32, 8, 128, 16)], seed=7)
    x = nested_inputs(torch, case, gs, gp, pt, ss, sh)
    want = bf16_host(launch_nested(x))
    torch.cuda.synchronize()
    out = torch.empty_like(x["q"])
    desc = pa.make_desc(x["q"], x["kp"], x["bt"], scale=case.scale, max_context_len=case.max_context_len)
    import ctypes
    ws = torch.empty(int(pa.load().pa_shared_prefix_workspace_bytes(ctypes.byref(desc))), dtype=torch.uint8,
                     device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            launch_nested(x, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(out), want)


@pytest.mark.parametrize("which", ["prefix_sharing", "parallel_sampling"])
def test_subgroups_prefix_sharing_workload(torch, ora, which, decode_kernel):
    """The prefix-sharing workload with its second level (the 4 samples of each
    prompt share the prompt's full suffix blocks), and the parallel-sampling
    workload (no common prefix, sub-groups only) -- bench --workload ..."""
    import bench
    plan, bt, ctx, slots, pairs = bench.prefix_sharing_setup(
        pa, wl.parallel_sampling_plan() if which == "parallel_sampling" else None)
    kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
    if len(pairs):
        assert ora.copy_blocks([kp], [vp], pairs) == 0
    assert ora.reshape_and_cache(nk, nv, kp, vp, slots) == 0
    S, B = len(ctx), plan.B
    ss, sh = bench.prefix_sharing_subgroups(plan, bt, ctx)
    for k in range(len(sh)):  # members agree on their shared blocks
        a, b = ss[k], ss[k + 1]
        assert np.all(bt[a:b, : sh[k] // B] == bt[a, : sh[k] // B])
    case = wl.DecodeCase("prefix", S, plan.Hq, plan.Hkv, plan.D, B, plan.num_blocks, bt.shape[1],
                         1 / math.sqrt(plan.D), ctx, bt, q, kp, vp)
    npre = plan.prefix_len // B
    if npre:
        gs, gp, pt = np.array([0, S], np.int32), np.array([plan.prefix_len], np.int32), bt[:1, :npre].copy()
    else:
        gs, gp, pt = np.zeros(1, np.int32), np.zeros(0, np.int32), np.zeros((1, 1), np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_nested(torch, case, gs, gp, pt, ss, sh, err)
    assert int(err.item()) == 0
    ref = oracle_rows(ora, case).reshape(got.shape)
    assert_close(got, ref, f"{which}, sub-groups")


@pytest.mark.parametrize("kernel", ["tasks", "units"])
def test_out_of_pool_page_in_late_task_flagged(torch, monkeypatch, kernel):
    """A table entry outside the pool in the last prompt's suffix of the full
    prefix-sharing workload.  Its tasks have the highest numbers, so the task
    kernel hands them out after every warp's first one (their entries are
    checked when first used, not when described).  The page is flagged
    (PA_DEVERR_PAGE) and read by nothing; every row outside that prompt's
    sub-group is bit-identical to the call without the bad entry."""
    import bench
    monkeypatch.setenv("PA_DECODE_TASKS", "1" if kernel == "tasks" else "0")
    plan, bt, ctx, slots, pairs = bench.prefix_sharing_setup(pa, None)
    kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    k_d, v_d = bf16_dev(kp, torch), bf16_dev(vp, torch)
    if len(pairs):
        pa.copy_blocks([k_d], [v_d], dev(np.asarray(pairs, np.int64).reshape(-1, 2)))
    pa.reshape_and_cache(bf16_dev(nk, torch), bf16_dev(nv, torch), k_d, v_d, dev(slots))
    S, B = len(ctx), plan.B
    ss, sh = bench.prefix_sharing_subgroups(plan, bt, ctx)
    npre = plan.prefix_len // B
    gs, gp, pt = np.array([0, S], np.int32), np.array([plan.prefix_len], np.int32), bt[:1, :npre].copy()
    # the last sub-group with at least two shared blocks past the prefix:
    # members a .. b-1, its shared block j
    k = max(i for i in range(len(sh)) if int(sh[i]) // B - npre >= 2)
    assert k >= len(sh) - 8
    a, b = int(ss[k]), int(ss[k + 1])
    j = (npre + int(sh[k]) // B) // 2
    assert npre <= j < int(sh[k]) // B
    bad = bt.copy()
    bad[a:b, j] = plan.num_blocks + 7
    outs = []
    for table in (bt, bad):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        res = pa.paged_attention_decode_shared_prefix(
            bf16_dev(q, torch), k_d, v_d, dev(table), dev(ctx), dev(gs), dev(gp), dev(pt), None, err_flag=err,
            subgroup_starts=dev(ss), subgroup_shared_lens=dev(sh), max_group_size=S,
            max_prefix_len=plan.prefix_len, scale=1 / math.sqrt(plan.D), max_context_len=int(ctx.max()),
            max_subgroup_size=int(np.diff(ss).max()))
        torch.cuda.synchronize()
        outs.append((bf16_host(res), int(err.item())))
    (clean, e0), (got, e1) = outs
    assert e0 == 0
    assert e1 & pa.DEVERR_PAGE
    keep = np.ones(S, bool)
    keep[a:b] = False
    assert np.array_equal(got[keep], clean[keep])
    assert np.all(np.isfinite(to_f64(got[a:b])))


def test_subgroup_guards(torch, decode_kernel):
    """A sub-group wider than max_subgroup_size promised (more query rows than
    the launch's MMA width) and sub-group starts outside the batch are refused
    in the kernel: PA_DEVERR_CTX, nothing read or written for them, the other
    sub-groups as plain decode."""
    spec = [(None, [(2, [3, 5]), (1, [8, 9, 4]), (0, [30])])]
    case, gs, gp, pt, ss, sh = nested_case(32, 8, 128, 16, spec, seed=9)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    x = nested_inputs(torch, case, gs, gp, pt, ss, sh)
    plain = bf16_host(pa.paged_attention_decode(x["q"], x["kp"], x["vp"], x["bt"], x["ctx"], scale=case.scale,
                                                max_context_len=case.max_context_len))
    # max_subgroup_size 2 promises 8 rows (one MMA n-tile); the 3-member sub-group has 12
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x["kw"] = dict(x["kw"], max_subgroup_size=2)
    out = torch.zeros_like(x["q"])
    launch_nested(x, err, out)
    torch.cuda.synchronize()
    got = bf16_host(out)
    assert int(err.item()) & pa.DEVERR_CTX
    assert not np.any(got[2:5])
    assert_close(np.concatenate([got[:2], got[5:]]), to_f64(np.concatenate([plain[:2], plain[5:]])), "other sub-groups")
    # the last sub-group reaching past the batch: refused before any read
    bad = ss.copy()
    bad[-1] = case.num_seqs + 3
    x = nested_inputs(torch, case, gs, gp, pt, bad, sh)
    err.zero_()
    out = torch.zeros_like(x["q"])
    launch_nested(x, err, out)
    torch.cuda.synchronize()
    got = bf16_host(out)
    assert int(err.item()) & pa.DEVERR_CTX
    assert_close(got[:5], to_f64(plain[:5]), "in-range sub-groups")
    assert not np.any(got[5:])  # the refused sub-group's rows are left alone (zeros from the caller)


@pytest.mark.parametrize("kernel", ["tasks", "wide"])
def test_unit_kernel_edges(torch, ora, monkeypatch, kernel):
    """The task-queue and wide-group kernels on their edge cases, against the
    oracle: a long unit (four long members behind a shared stretch: the most
    parts of a task unit, many key tiles of a wide one), units with no keys
    past the group prefix (every member ends at the prefix: the rows are the
    prefix's states alone), one-member units, and a sub-group outside every
    group beside them."""
    monkeypatch.setenv("PA_DECODE_TASKS" if kernel == "tasks" else "PA_DECODE_WIDE", "1")
    spec = [(3, [(20, [600, 601, 590, 615]), (0, [0, 0]), (0, [0]), (1, [7])]),
            (None, [(2, [1, 300])])]
    case, gs, gp, pt, ss, sh = nested_case(32, 8, 128, 16, spec, seed=23)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_nested(torch, case, gs, gp, pt, ss, sh, err)
    assert int(err.item()) == 0
    ref, st = ora.decode_case(case)
    assert np.all(st == 0)
    assert_close(got, ref, f"{kernel} decode edges")
