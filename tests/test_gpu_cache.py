"""GPU parity of reshape_and_cache and copy_blocks (bit-exact against the
oracle's host application of the same writes), and the copy-on-write flow of
the prefix-sharing workload end to end."""
import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("T,Hkv,D,B", [(1, 1, 64, 16), (64, 8, 128, 16), (8432, 8, 128, 32), (37, 3, 64, 32)])
def test_reshape_and_cache_bit_exact(torch, ora, T, Hkv, D, B):
    st = wl.Stream(T, D)
    nblk = (T + B - 1) // B + 7
    kp = wl.normal_bf16(st, (nblk, Hkv, B, D))
    vp = wl.normal_bf16(st, (nblk, Hkv, B, D))
    k = wl.normal_bf16(st, (T, Hkv, D))
    v = wl.normal_bf16(st, (T, Hkv, D))
    slots = st.permutation(nblk * B)[:T].astype(np.int64)
    if T > 4:
        slots[3] = -1  # padding token: no write
    dk, dv = bf16_dev(kp, torch), bf16_dev(vp, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(bf16_dev(k, torch), bf16_dev(v, torch), dk, dv,
                         torch.from_numpy(slots).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert ora.reshape_and_cache(k, v, kp, vp, slots) == 0
    assert int(err.item()) == 0
    assert np.array_equal(bf16_host(dk), kp) and np.array_equal(bf16_host(dv), vp)


def test_reshape_and_cache_out_of_range_slot_flagged(torch, ora):
    st = wl.Stream(2, 2)
    kp = wl.normal_bf16(st, (4, 2, 16, 64))
    vp = wl.normal_bf16(st, (4, 2, 16, 64))
    k = wl.normal_bf16(st, (3, 2, 64))
    v = wl.normal_bf16(st, (3, 2, 64))
    slots = np.array([5, 4 * 16, 17], np.int64)
    dk, dv = bf16_dev(kp, torch), bf16_dev(vp, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(bf16_dev(k, torch), bf16_dev(v, torch), dk, dv, torch.from_numpy(slots).cuda(),
                         err_flag=err)
    torch.cuda.synchronize()
    assert ora.reshape_and_cache(k, v, kp, vp, slots) & 4
    assert int(err.item()) & pa.DEVERR_SLOT
    assert np.array_equal(bf16_host(dk), kp) and np.array_equal(bf16_host(dv), vp)


@pytest.mark.parametrize("L,pairs", [(1, 1), (3, 17), (130, 5)])
def test_copy_blocks_bit_exact(torch, ora, L, pairs):
    st = wl.Stream(L, pairs)
    nblk, Hkv, B, D = 2 * pairs + 3, 8, 16, 128 if L < 100 else 64
    kps = [wl.normal_bf16(st, (nblk, Hkv, B, D)) for _ in range(L)]
    vps = [wl.normal_bf16(st, (nblk, Hkv, B, D)) for _ in range(L)]
    perm = st.permutation(nblk)
    pr = np.stack([perm[:pairs], perm[pairs: 2 * pairs]], axis=1).astype(np.int64)
    dks = [bf16_dev(a, torch) for a in kps]
    dvs = [bf16_dev(a, torch) for a in vps]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.copy_blocks(dks, dvs, torch.from_numpy(pr).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert ora.copy_blocks(kps, vps, pr) == 0
    assert int(err.item()) == 0
    for l in range(L):
        assert np.array_equal(bf16_host(dks[l]), kps[l]) and np.array_equal(bf16_host(dvs[l]), vps[l])


def test_copy_blocks_bad_pair_flagged(torch):
    kp = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.copy_blocks([kp], [vp], torch.tensor([[0, 9]], dtype=torch.int64, device="cuda"), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_PAIR


def build_prefix_sharing(plan):
    """Drives the block manager through the prefix-sharing workload: returns the
    decode tables, the CoW pairs and the new tokens' slots."""
    B = plan.B
    bm = pa.BlockManager(plan.num_blocks, B)
    R = plan.samples_per_prompt
    S = plan.num_prompts * R
    root = 10 ** 6
    bm.add_seq(root, plan.prefix_len)
    for p in range(plan.num_prompts):
        if plan.independent_suffixes:
            for i in range(R):
                bm.fork(root, p * R + i)
                for _ in range(int(plan.suffix_lens[p * R + i])):
                    bm.append(p * R + i)
        else:
            bm.fork(root, p * R)
            for _ in range(int(plan.suffix_lens[p])):
                bm.append(p * R)
            for i in range(1, R):
                bm.fork(p * R, p * R + i)
    bm.free_seq(root)
    slots, pairs = [], []
    for s in range(S):
        slot, pair = bm.append(s)
        slots.append(slot)
        if pair is not None:
            pairs.append(pair)
    ctx = np.array([bm.seq_len(s) for s in range(S)], np.int32)
    tables = [bm.block_table(s) for s in range(S)]
    mb = max(len(t) for t in tables)
    bt = np.full((S, mb), -1, np.int32)
    for s, t in enumerate(tables):
        bt[s, : len(t)] = t
    return bm, bt, ctx, np.array(slots, np.int64), np.array(pairs, np.int64).reshape(-1, 2)


@pytest.mark.parametrize("independent", [False, True])
def test_prefix_sharing_cow_flow(torch, ora, independent):
    """fork -> copy-on-write (copy_blocks) -> reshape_and_cache -> decode over
    shared tables, against the oracle applying the same steps on the host."""
    plan = wl.prefix_sharing_plan(independent_suffixes=independent)
    bm, bt, ctx, slots, pairs = build_prefix_sharing(plan)
    kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
    S = len(ctx)
    dk, dv = bf16_dev(kp, torch), bf16_dev(vp, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if len(pairs):
        pa.copy_blocks([dk], [dv], torch.from_numpy(pairs).cuda(), err_flag=err)
    pa.reshape_and_cache(bf16_dev(nk, torch), bf16_dev(nv, torch), dk, dv, torch.from_numpy(slots).cuda(),
                         err_flag=err)
    dq = bf16_dev(q, torch)
    out = pa.paged_attention_decode(dq, dk, dv, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(),
                                    max_context_len=int(ctx.max()), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if len(pairs):
        assert ora.copy_blocks([kp], [vp], pairs) == 0
    assert ora.reshape_and_cache(nk, nv, kp, vp, slots) == 0
    assert np.array_equal(bf16_host(dk), kp) and np.array_equal(bf16_host(dv), vp)
    got = bf16_host(out)
    heads = [(s, h) for s in range(0, S, 9) for h in (0, 13, 31)]
    ref = np.stack([ora.decode_head(q, kp, vp, bt, ctx, 1 / np.sqrt(128), s, h)[0] for s, h in heads])
    assert_close(np.stack([got[s, h] for s, h in heads]), ref, "prefix sharing")


def test_swap_out_and_back_in_is_bit_exact(torch, ora):
    """Preemption round trip: a sequence's pages go to a pinned host pool,
    the device blocks are reused, and the pages come back to new device
    blocks bit for bit; decode over the new table is bit-identical."""
    case = wl.make_decode_case("swap", [300, 77, 500], 16, 4, 128, 16, seed=14, pool_blocks=120,
                               with_new_tokens=False)
    L = 2
    st = wl.Stream(14, 2)
    kps = [case.k_pool] + [wl.normal_bf16(st, case.k_pool.shape) for _ in range(L - 1)]
    vps = [case.v_pool] + [wl.normal_bf16(st, case.v_pool.shape) for _ in range(L - 1)]
    dk = [bf16_dev(a, torch) for a in kps]
    dv = [bf16_dev(a, torch) for a in vps]
    nhost = 64
    hk = [torch.zeros((nhost,) + tuple(case.k_pool.shape[1:]), dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    hv = [torch.zeros_like(h).pin_memory() for h in hk]
    # sequence 2 is preempted
    table2 = [int(b) for b in case.block_tables[2] if b >= 0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = bf16_host(pa.paged_attention_decode(bf16_dev(case.q, torch), dk[0], dv[0],
                                              torch.from_numpy(case.block_tables).cuda(),
                                              torch.from_numpy(case.context_lens).cuda(), scale=case.scale,
                                              max_context_len=case.max_context_len))
    out_pairs = np.array([(d, h) for h, d in enumerate(table2)], np.int64)  # device block -> host block
    pa.swap_blocks(dk, dv, hk, hv, torch.from_numpy(out_pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    # the oracle applies the same moves to host copies of every pool
    ok_ = [a.copy() for a in kps]
    ov_ = [a.copy() for a in vps]
    ohk = [np.zeros((nhost,) + case.k_pool.shape[1:], np.uint16) for _ in range(L)]
    ohv = [np.zeros_like(a) for a in ohk]
    assert ora.swap_blocks(ok_, ov_, ohk, ohv, out_pairs) == 0
    for l in range(L):
        assert np.array_equal(hk[l].view(torch.int16).numpy().view(np.uint16), ohk[l])
        assert np.array_equal(hv[l].view(torch.int16).numpy().view(np.uint16), ohv[l])
    # the device blocks get reused by someone else
    for l in range(L):
        dk[l][table2] = 0
        dv[l][table2] = 0
        ok_[l][table2] = 0
        ov_[l][table2] = 0
    # bring the pages back into other (free) device blocks
    used = set(int(b) for b in case.block_tables.flatten() if b >= 0)
    free = [b for b in range(case.num_blocks) if b not in used][: len(table2)]
    in_pairs = np.array([(h, free[h]) for h in range(len(table2))], np.int64)
    pa.swap_blocks(hk, hv, dk, dv, torch.from_numpy(in_pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert ora.swap_blocks(ohk, ohv, ok_, ov_, in_pairs) == 0
    for l in range(L):
        assert np.array_equal(bf16_host(dk[l]), ok_[l]) and np.array_equal(bf16_host(dv[l]), ov_[l])
    bt = case.block_tables.copy()
    bt[2, : len(table2)] = free
    again = bf16_host(pa.paged_attention_decode(bf16_dev(case.q, torch), dk[0], dv[0], torch.from_numpy(bt).cuda(),
                                                torch.from_numpy(case.context_lens).cuda(), scale=case.scale,
                                                max_context_len=case.max_context_len))
    assert np.array_equal(again, ref)
