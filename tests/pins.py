"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with what the pages or mathematics fix:

* brute force: attention over the *contiguous* token sequence computed with
  scipy's softmax and numpy matrix products (no paging, no shared code);
* invariants: physical page permutation, block size 1/16/32, shared pages vs
  private copies, GQA head grouping, split-K recombination;
* closed forms: ctx = 1 gives v0, identical keys / scale 0 give mean(V), a
  dominant key gives its value;
* printed examples from the pages (``tests/golden``): the logical->physical
  block figure and the KV sizing formula.

``ALL_PINS`` is rerun against deliberately broken oracle builds by
``test_oracle_mutants.py``; every planted mistake must trip at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf(st, shape, mul=1.0):
    return wl.f64_to_bf16_bits(st.normal(int(np.prod(shape))) * mul).reshape(shape)


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def brute_attention(q, K, V, scale):
    """Contiguous attention with scipy's softmax: q [D], K,V [n][D] (fp64)."""
    p = softmax(scale * (K @ q))
    return p @ V


def brute_causal(Q, K, V, scale, first_pos):
    """Causal attention of rows Q[i] at positions first_pos + i over K/V[0..pos]."""
    n = K.shape[0]
    S = scale * (Q @ K.T)
    pos = first_pos + np.arange(Q.shape[0])[:, None]
    S = np.where(np.arange(n)[None, :] <= pos, S, -np.inf)
    return softmax(S, axis=1) @ V


def paginate(Kc, Vc, B, perm, nblk, D_fill_stream=None):
    """Lay contiguous per-head K/V [Hkv][n][D] into a pool [nblk][Hkv][B][D] at
    the pages ``perm`` (logical block i -> perm[i]); other pages get noise."""
    Hkv, n, D = Kc.shape
    nb = (n + B - 1) // B
    st = D_fill_stream or wl.Stream(99, 99)
    kp = _bf(st, (nblk, Hkv, B, D))
    vp = _bf(st, (nblk, Hkv, B, D))
    for t in range(n):
        kp[perm[t // B], :, t % B, :] = Kc[:, t, :]
        vp[perm[t // B], :, t % B, :] = Vc[:, t, :]
    table = np.full(max(nb, 1), -1, dtype=np.int32)
    table[:nb] = perm[:nb]
    return kp, vp, table


def _tables(rows, mb):
    bt = np.full((len(rows), mb), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        bt[i, : len(r)] = r
    return bt


# --------------------------------------------------------------------------
def pin_bruteforce(ora):
    """Paged oracle == contiguous scipy attention, tiny inputs, B in {1,2,16}."""
    st = wl.Stream(1, 1)
    for B in (1, 2, 16):
        for (ctxs, Hq, Hkv, D) in (([1, 7, 40], 4, 2, 8), ([33, 16, 5], 2, 2, 16), ([17], 6, 3, 4)):
            S = len(ctxs)
            Kc = [_bf(st, (Hkv, n, D)) for n in ctxs]
            Vc = [_bf(st, (Hkv, n, D)) for n in ctxs]
            q = _bf(st, (S, Hq, D))
            nblk = sum((n + B - 1) // B for n in ctxs) + 5
            perm = st.permutation(nblk)
            kp = _bf(st, (nblk, Hkv, B, D))
            vp = _bf(st, (nblk, Hkv, B, D))
            rows, used = [], 0
            for s, n in enumerate(ctxs):
                nb = (n + B - 1) // B
                pages = perm[used: used + nb]
                used += nb
                for t in range(n):
                    kp[pages[t // B], :, t % B] = Kc[s][:, t]
                    vp[pages[t // B], :, t % B] = Vc[s][:, t]
                rows.append(pages)
            bt = _tables(rows, max(len(r) for r in rows))
            scale = 1.0 / math.sqrt(D)
            out, stt = ora.decode(q, kp, vp, bt, np.array(ctxs), scale)
            assert np.all(stt == 0)
            G = Hq // Hkv
            for s, n in enumerate(ctxs):
                for h in range(Hq):
                    ref = brute_attention(_f64(q[s, h]), _f64(Kc[s][h // G]), _f64(Vc[s][h // G]), scale)
                    assert np.max(np.abs(out[s, h] - ref)) <= 1e-12, (B, s, h)


def _logical_case(st, n, Hq, Hkv, D):
    return _bf(st, (Hkv, n, D)), _bf(st, (Hkv, n, D)), _bf(st, (1, Hq, D))


def pin_permutation(ora):
    """Same logical K/V under two different physical assignments: identical output."""
    st = wl.Stream(2, 2)
    n, Hq, Hkv, D, B = 77, 4, 2, 16, 16
    Kc, Vc, q = _logical_case(st, n, Hq, Hkv, D)
    nblk = 12
    outs = []
    for _ in range(3):
        perm = st.permutation(nblk)
        kp, vp, table = paginate(Kc, Vc, B, perm, nblk)
        out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.25)
        assert s[0] == 0
        outs.append(out)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_block_size(ora):
    """Paging granularity does not change the result: B = 1, 16, 32 agree exactly."""
    st = wl.Stream(3, 3)
    n, Hq, Hkv, D = 70, 2, 1, 8
    Kc, Vc, q = _logical_case(st, n, Hq, Hkv, D)
    outs = []
    for B in (1, 16, 32):
        nblk = (n + B - 1) // B + 3
        perm = st.permutation(nblk)
        kp, vp, table = paginate(Kc, Vc, B, perm, nblk)
        out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.3)
        assert s[0] == 0
        outs.append(out)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_sharing(ora):
    """Two sequences sharing prefix pages == the same sequences with private copies."""
    st = wl.Stream(4, 4)
    Hq, Hkv, D, B = 4, 2, 8, 16
    nblk = 16
    kp = _bf(st, (nblk, Hkv, B, D))
    vp = _bf(st, (nblk, Hkv, B, D))
    q = _bf(st, (2, Hq, D))
    shared = _tables([[3, 5, 9], [3, 5, 11]], 3)
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[12], vp2[12] = kp[3], vp[3]
    kp2[13], vp2[13] = kp[5], vp[5]
    private = _tables([[3, 5, 9], [12, 13, 11]], 3)
    ctx = np.array([40, 45])
    a, sa = ora.decode(q, kp, vp, shared, ctx, 0.35)
    b, sb = ora.decode(q, kp2, vp2, private, ctx, 0.35)
    assert np.all(sa == 0) and np.all(sb == 0)
    assert np.array_equal(a, b)


def pin_ctx1(ora):
    """ctx = 1: the only weight is 1, so the output is v0 exactly."""
    st = wl.Stream(5, 5)
    Hq, Hkv, D, B = 4, 4, 16, 16
    kp = _bf(st, (6, Hkv, B, D))
    vp = _bf(st, (6, Hkv, B, D))
    q = _bf(st, (1, Hq, D))
    out, s = ora.decode(q, kp, vp, np.array([[4]], np.int32), np.array([1]), 0.25)
    assert s[0] == 0
    assert np.array_equal(out[0], _f64(vp[4, :, 0, :]))


def pin_identical_keys(ora):
    """All keys equal: uniform weights, output = mean of the values."""
    st = wl.Stream(6, 6)
    n, Hq, Hkv, D, B = 37, 2, 1, 8, 16
    k1 = _bf(st, (D,))
    Kc = np.broadcast_to(k1, (Hkv, n, D)).copy()
    Vc = _bf(st, (Hkv, n, D))
    q = _bf(st, (1, Hq, D))
    kp, vp, table = paginate(Kc, Vc, B, st.permutation(5), 5)
    out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.4)
    assert s[0] == 0
    ref = _f64(Vc[0]).mean(axis=0)
    for h in range(Hq):
        assert np.max(np.abs(out[0, h] - ref)) <= 1e-13


def pin_scale_zero(ora):
    """scale = 0: every score is 0, output = mean of the values."""
    st = wl.Stream(7, 7)
    n, Hq, Hkv, D, B = 50, 2, 2, 8, 16
    Kc, Vc, q = _logical_case(st, n, Hq, Hkv, D)
    kp, vp, table = paginate(Kc, Vc, B, st.permutation(6), 6)
    out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.0)
    for h in range(Hq):
        assert np.max(np.abs(out[0, h] - _f64(Vc[h]).mean(axis=0))) <= 1e-13


def pin_dominant_key(ora):
    """One key scores 40 above all others: output = that key's value (to e^-40 n)."""
    st = wl.Stream(8, 8)
    n, Hq, Hkv, D, B = 30, 1, 1, 8, 16
    Vc = _bf(st, (Hkv, n, D))
    Kc = np.zeros((Hkv, n, D), dtype=np.uint16)
    one = wl.f64_to_bf16_bits(np.array([1.0]))[0]
    forty = wl.f64_to_bf16_bits(np.array([40.0]))[0]
    Kc[0, 13, 0] = forty
    q = np.zeros((1, Hq, D), dtype=np.uint16)
    q[0, 0, 0] = one
    kp, vp, table = paginate(Kc, Vc, B, st.permutation(4), 4)
    out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 1.0)
    assert np.max(np.abs(out[0, 0] - _f64(Vc[0, 13]))) <= 30 * math.exp(-40) * 8 + 1e-15
    # ... and the dominant key moved to another position follows the move
    Kc2 = np.zeros_like(Kc)
    Kc2[0, 2, 0] = forty
    kp, vp, table = paginate(Kc2, Vc, B, st.permutation(4), 4)
    out2, _ = ora.decode(q, kp, vp, table[None, :], np.array([n]), 1.0)
    assert np.max(np.abs(out2[0, 0] - _f64(Vc[0, 2]))) <= 1e-14


def pin_gqa_grouping(ora):
    """Perturbing kv head g changes exactly the query heads of group g."""
    st = wl.Stream(9, 9)
    n, Hq, Hkv, D, B = 40, 8, 2, 8, 16
    Kc, Vc, q = _logical_case(st, n, Hq, Hkv, D)
    perm = st.permutation(5)
    kp, vp, table = paginate(Kc, Vc, B, perm, 5)
    a, _ = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.3)
    Kc2, Vc2 = Kc.copy(), Vc.copy()
    Kc2[1] = _bf(st, (n, D))
    Vc2[1] = _bf(st, (n, D))
    kp2, vp2, _ = paginate(Kc2, Vc2, B, perm, 5)
    b, _ = ora.decode(q, kp2, vp2, table[None, :], np.array([n]), 0.3)
    G = Hq // Hkv
    for h in range(Hq):
        same = np.array_equal(a[0, h], b[0, h])
        assert same == (h // G == 0), h


def pin_split_combine(ora):
    """Split-K: combining partial states of any split equals the unsplit output."""
    st = wl.Stream(10, 10)
    n, Hq, Hkv, D, B = 53, 2, 1, 8, 16
    Kc, Vc, q = _logical_case(st, n, Hq, Hkv, D)
    kp, vp, table = paginate(Kc, Vc, B, st.permutation(6), 6)
    ctx = np.array([n])
    full, _ = ora.decode(q, kp, vp, table[None, :], ctx, 0.3)
    for h in range(Hq):
        for P in (1, 2, 5, 16, 53, 60):
            ms, ls, os_ = [], [], []
            for j0 in range(0, n, P):
                m, l, o, s = ora.partial(q, kp, vp, table[None, :], ctx, 0.3, 0, h, j0, j0 + P)
                assert s == 0
                ms.append(m), ls.append(l), os_.append(o)
            ms.append(-np.inf), ls.append(0.0), os_.append(np.zeros(D))  # an empty part
            comb = ora.combine(np.array(ms), np.array(ls), np.stack(os_))
            assert np.max(np.abs(comb - full[0, h])) <= 1e-13, (h, P)


def pin_prefill(ora):
    """Chunked prefill: C = ctx equals causal attention over the whole prompt; a
    chunk at the end of a longer context equals causal rows at their positions;
    row 0 of a full-prompt chunk is v0; every row equals decode at pos+1."""
    st = wl.Stream(11, 11)
    Hq, Hkv, D, B = 4, 2, 8, 16
    n = 45
    Kc, Vc, _ = _logical_case(st, n, Hq, Hkv, D)
    perm = st.permutation(6)
    kp, vp, table = paginate(Kc, Vc, B, perm, 6)
    for C in (n, 20, 1):
        qc = _bf(st, (C, Hq, D))
        cu = np.array([0, C], np.int32)
        bt = table[None, :]
        ctx = np.array([n], np.int32)
        G = Hq // Hkv
        for h in range(Hq):
            ref = brute_causal(_f64(qc[:, h]), _f64(Kc[h // G]), _f64(Vc[h // G]), 0.3, n - C)
            for i in range(C):
                out, s = ora.prefill_row(qc, cu, kp, vp, bt, ctx, 0.3, 0, i, h)
                assert s == 0
                assert np.max(np.abs(out - ref[i])) <= 1e-12, (C, i, h)
                dec, _ = ora.decode_head(qc[i: i + 1], kp, vp, bt, np.array([n - C + i + 1]), 0.3, 0, h)
                assert np.array_equal(out, dec)
        if C == n:
            out0, _ = ora.prefill_row(qc, cu, kp, vp, bt, ctx, 0.3, 0, 0, 0)
            assert np.array_equal(out0, _f64(Vc[0, 0]))


def pin_block_map_figure(ora):
    """The pages' logical->physical figure: blocks [9, 2, 14], 16 tokens each."""
    fx = json.load(open(os.path.join(GOLDEN, "block_map_example.json")))
    B = fx["block_size"]
    Hkv, D, nblk = 1, 64, 16
    kp = np.zeros((nblk, Hkv, B, D), np.uint16)
    vp = np.zeros((nblk, Hkv, B, D), np.uint16)
    one = wl.f64_to_bf16_bits(np.array([1.0]))[0]
    # reshape_and_cache each token t at its derived slot with K = 50 e_t, V = e_t
    n = 48
    fifty = wl.f64_to_bf16_bits(np.array([50.0]))[0]
    k = np.zeros((n, Hkv, D), np.uint16)
    v = np.zeros((n, Hkv, D), np.uint16)
    slots = np.zeros(n, np.int64)
    for r in fx["ranges"]:
        for t in range(r["first_token"], r["last_token"] + 1):
            k[t, 0, t] = fifty
            v[t, 0, t] = one
            slots[t] = r["physical_block"] * B + (t - r["first_token"])
    for d in fx["derived"]:
        assert slots[d["token"]] == d["slot"] == d["block"] * B + d["offset"]
    assert ora.reshape_and_cache(k, v, kp, vp, slots) == 0
    for d in fx["derived"]:
        assert kp[d["block"], 0, d["offset"], d["token"]] == fifty
    table = np.array([[r["physical_block"] for r in fx["ranges"]]], np.int32)
    for tok in (0, 20, 47):
        q = np.zeros((1, 1, D), np.uint16)
        q[0, 0, tok] = one
        out, s = ora.decode(q, kp, vp, table, np.array([n]), 1.0)
        assert s[0] == 0
        assert int(np.argmax(out[0, 0])) == tok and out[0, 0, tok] > 0.999


def pin_scatter_gather(ora):
    """Writing a sequence's tokens with reshape_and_cache at the slots its table
    gives, then decoding it, equals contiguous attention over those tokens."""
    st = wl.Stream(12, 12)
    n, Hq, Hkv, D, B, nblk = 70, 4, 2, 16, 16, 9
    kp = _bf(st, (nblk, Hkv, B, D))
    vp = _bf(st, (nblk, Hkv, B, D))
    table = st.permutation(nblk)[: (n + B - 1) // B].astype(np.int32)
    k = _bf(st, (n, Hkv, D))
    v = _bf(st, (n, Hkv, D))
    slots = np.array([table[t // B] * B + t % B for t in range(n)], np.int64)
    slots_pad = np.concatenate([slots[:30], [-1, -1], slots[30:]])
    k_pad = np.concatenate([k[:30], _bf(st, (2, Hkv, D)), k[30:]])
    v_pad = np.concatenate([v[:30], _bf(st, (2, Hkv, D)), v[30:]])
    before = kp.copy()
    assert ora.reshape_and_cache(k_pad, v_pad, kp, vp, slots_pad) == 0
    untouched = np.setdiff1d(np.arange(nblk), table)
    assert np.array_equal(kp[untouched], before[untouched])
    q = _bf(st, (1, Hq, D))
    out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 0.25)
    G = Hq // Hkv
    for h in range(Hq):
        ref = brute_attention(_f64(q[0, h]), _f64(k[:, h // G]), _f64(v[:, h // G]), 0.25)
        assert np.max(np.abs(out[0, h] - ref)) <= 1e-12


def pin_copy_blocks(ora):
    """Copy-on-write: after copying shared pages to fresh ones, every layer's
    copies are bitwise equal, other pages unchanged, and a table pointing at the
    copies decodes exactly like the shared one."""
    st = wl.Stream(13, 13)
    L, nblk, Hkv, B, D, Hq = 3, 10, 2, 16, 8, 4
    kps = [_bf(st, (nblk, Hkv, B, D)) for _ in range(L)]
    vps = [_bf(st, (nblk, Hkv, B, D)) for _ in range(L)]
    orig_k = [a.copy() for a in kps]
    orig_v = [a.copy() for a in vps]
    pairs = np.array([[2, 7], [5, 8], [0, 9]], np.int64)
    assert ora.copy_blocks(kps, vps, pairs) == 0
    for l in range(L):
        for src, dst in pairs:
            assert np.array_equal(kps[l][dst], orig_k[l][src]) and np.array_equal(vps[l][dst], orig_v[l][src])
        others = np.setdiff1d(np.arange(nblk), pairs[:, 1])
        assert np.array_equal(kps[l][others], orig_k[l][others])
        assert np.array_equal(vps[l][others], orig_v[l][others])
    q = _bf(st, (1, Hq, D))
    a, _ = ora.decode(q, kps[1], vps[1], np.array([[2, 5, 0]], np.int32), np.array([40]), 0.3)
    b, _ = ora.decode(q, kps[1], vps[1], np.array([[7, 8, 9]], np.int32), np.array([40]), 0.3)
    assert np.array_equal(a, b)


def pin_swap_blocks(ora):
    """Preemptive swapping: a sequence's blocks go to a host pool of another
    size and come back to other device blocks.  Each moved block is bitwise
    its source, nothing else changes, a pair outside either pool is refused,
    and the sequence decodes exactly as before through its new table."""
    st = wl.Stream(13, 14)
    L, nblk, nhost, Hkv, B, D, Hq = 2, 12, 5, 2, 16, 8, 4
    dk = [_bf(st, (nblk, Hkv, B, D)) for _ in range(L)]
    dv = [_bf(st, (nblk, Hkv, B, D)) for _ in range(L)]
    hk = [np.zeros((nhost, Hkv, B, D), np.uint16) for _ in range(L)]
    hv = [np.zeros((nhost, Hkv, B, D), np.uint16) for _ in range(L)]
    table = [6, 1, 10]
    q = _bf(st, (1, Hq, D))
    before, _ = ora.decode(q, dk[1], dv[1], np.array([table], np.int32), np.array([37]), 0.3)
    saved_k = [a.copy() for a in dk]
    out_pairs = np.array([[6, 3], [1, 0], [10, 4]], np.int64)  # device block -> host block
    assert ora.swap_blocks(dk, dv, hk, hv, out_pairs) == 0
    for l in range(L):
        for src, dst in out_pairs:
            assert np.array_equal(hk[l][dst], dk[l][src]) and np.array_equal(hv[l][dst], dv[l][src])
        assert not hk[l][1].any() and not hv[l][2].any()  # untouched host blocks
        assert np.array_equal(dk[l], saved_k[l])  # the source is only read
        for b in table:  # the device blocks are handed to someone else
            dk[l][b] = 0
            dv[l][b] = 0
    in_pairs = np.array([[3, 2], [0, 8], [4, 11]], np.int64)  # host block -> new device block
    assert ora.swap_blocks(hk, hv, dk, dv, in_pairs) == 0
    after, _ = ora.decode(q, dk[1], dv[1], np.array([[2, 8, 11]], np.int32), np.array([37]), 0.3)
    assert np.array_equal(before, after)
    for l in range(L):
        assert np.array_equal(dk[l][[2, 8, 11]], saved_k[l][table])
    snap = [a.copy() for a in hk]
    assert ora.swap_blocks(dk, dv, hk, hv, np.array([[0, nhost]], np.int64)) & 2  # past the host pool
    assert ora.swap_blocks(dk, dv, hk, hv, np.array([[nblk, 0]], np.int64)) & 2  # past the device pool
    assert all(np.array_equal(a, b) for a, b in zip(hk, snap))


def pin_kv_sizing(ora):
    """The pages' KV sizing example: 2 x 80 x 8 x 128 x 2 = 327,680 bytes/token."""
    fx = json.load(open(os.path.join(GOLDEN, "kv_sizing_llama31_70b.json")))
    b = ora.kv_bytes_per_token(fx["layers"], fx["kv_heads"], fx["head_dim"], fx["bytes_per_element"])
    assert b == fx["bytes_per_token"]
    assert b * fx["context_tokens"] == fx["bytes_per_request_exact"]


def pin_large_scores(ora):
    """Scores in the thousands: no overflow, still equals scipy's softmax."""
    st = wl.Stream(14, 14)
    n, Hq, Hkv, D, B = 33, 2, 1, 8, 16
    Kc = _bf(st, (Hkv, n, D), mul=30.0)
    Vc = _bf(st, (Hkv, n, D))
    q = _bf(st, (1, Hq, D), mul=30.0)
    kp, vp, table = paginate(Kc, Vc, B, st.permutation(4), 4)
    out, s = ora.decode(q, kp, vp, table[None, :], np.array([n]), 1.0)
    assert np.all(np.isfinite(out))
    for h in range(Hq):
        ref = brute_attention(_f64(q[0, h]), _f64(Kc[0]), _f64(Vc[0]), 1.0)
        assert np.max(np.abs(out[0, h] - ref)) <= 1e-12


def pin_errors(ora):
    """ctx <= 0, ctx beyond the table, a bad page id and a slot past the pool are
    reported and produce zeros / no write; slot -1 is skipped."""
    st = wl.Stream(15, 15)
    Hq, Hkv, D, B, nblk = 2, 1, 8, 16, 4
    kp = _bf(st, (nblk, Hkv, B, D))
    vp = _bf(st, (nblk, Hkv, B, D))
    q = _bf(st, (3, Hq, D))
    bt = np.array([[1, 2], [0, 7], [3, -1]], np.int32)
    out, s = ora.decode(q, kp, vp, bt, np.array([0, 20, 33]), 0.3)
    assert s[0] & 1 and s[1] & 2 and s[2] & 1
    assert not np.any(out)
    k = _bf(st, (2, Hkv, D))
    v = _bf(st, (2, Hkv, D))
    kp2 = kp.copy()
    vp2 = vp.copy()
    assert ora.reshape_and_cache(k, v, kp2, vp2, np.array([-1, nblk * B], np.int64)) & 4
    assert np.array_equal(kp2, kp) and np.array_equal(vp2, vp)


def pin_bf16_decoding(ora):
    """The oracle widens bf16 inputs exactly: a bf16 value is the float32
    whose upper 16 bits are its bits (sign, 8-bit exponent, 7-bit mantissa)."""
    cases = {0x0000: 0.0, 0x8000: -0.0, 0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x3F81: 1.0078125,
             0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
             0x7F80: math.inf, 0xFF80: -math.inf}
    for bits, want in cases.items():
        got = ora.bf16_to_f64(bits)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (hex(bits), got, want)
    assert math.isnan(ora.bf16_to_f64(0x7FC0))
    st = wl.Stream(5, 5)
    bits = st.integers(0, 0x7F80, 200).astype(np.uint16)  # finite positives
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert all(ora.bf16_to_f64(int(b)) == r for b, r in zip(bits, ref))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
