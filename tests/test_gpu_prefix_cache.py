"""Automatic prefix caching end to end: a prompt that repeats another
prompt's leading full blocks reuses them from the block manager's cache, and
only its remaining tokens are written (reshape_and_cache) and prefilled as a
chunk whose context includes the cached blocks.  Its outputs must equal the
same prompt prefilled from scratch, and the fp64 oracle."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def prefill(torch, bm, seq, tokens, k_tok, v_tok, q_tok, first, kp, vp, Hq, B, nblk):
    """Writes tokens first.. of `seq` into the cache and prefills them as one
    chunk over the whole context; returns the chunk's outputs (bf16 bits)."""
    n = len(tokens)
    table = bm.block_table(seq)
    slots = np.array([table[j // B] * B + j % B for j in range(first, n)], np.int64)
    pa.reshape_and_cache(bf16_dev(k_tok[first:], torch), bf16_dev(v_tok[first:], torch), kp, vp,
                         torch.from_numpy(slots).cuda())
    bt = np.array([table], np.int32)
    out = pa.paged_attention_prefill_chunk(bf16_dev(q_tok[first:], torch), torch.tensor([0, n - first], dtype=torch.int32,
                                                                                       device="cuda"),
                                           kp, vp, torch.from_numpy(bt).cuda(),
                                           torch.tensor([n], dtype=torch.int32, device="cuda"), max_q_len=n - first,
                                           scale=1 / math.sqrt(128), max_context_len=n)
    torch.cuda.synchronize()
    return bf16_host(out), bt, slots


@pytest.mark.parametrize("B", [16, 32])
def test_cached_prefix_prefill_equals_from_scratch(torch, ora, B):
    Hq, Hkv, D = 16, 4, 128
    st = wl.Stream(50 + B, 2)
    na, nb, shared = 300, 420, 200          # B's first 200 tokens repeat A's
    tok_a = [int(t) for t in st.integers(0, 32000, na)]
    tok_b = tok_a[:shared] + [int(t) for t in st.integers(0, 32000, nb - shared)]
    kv_a = wl.normal_bf16(st, (2, na, Hkv, D))
    kv_b = wl.normal_bf16(st, (2, nb, Hkv, D))
    kv_b[:, :shared] = kv_a[:, :shared]     # a model gives identical prefixes identical K/V
    q_a = wl.normal_bf16(st, (na, Hq, D))
    q_b = wl.normal_bf16(st, (nb, Hq, D))
    nblk = 64
    bm = pa.BlockManager(nblk, B)
    kp = torch.zeros((nblk, Hkv, B, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    assert bm.add_seq_tokens(0, tok_a) == 0
    _, _, slots_a = prefill(torch, bm, 0, tok_a, kv_a[0], kv_a[1], q_a, 0, kp, vp, Hq, B, nblk)
    cached = bm.add_seq_tokens(1, tok_b)
    assert cached == (shared // B) * B and cached > 0
    assert bm.block_table(1)[: cached // B] == bm.block_table(0)[: cached // B]
    got, bt_b, slots_b = prefill(torch, bm, 1, tok_b, kv_b[0], kv_b[1], q_b, cached, kp, vp, Hq, B, nblk)
    # the same prompt from scratch in its own pool and manager
    bm2 = pa.BlockManager(nblk, B)
    kp2 = torch.zeros_like(kp)
    vp2 = torch.zeros_like(kp)
    bm2.add_seq(0, nb)
    full, _, _ = prefill(torch, bm2, 0, tok_b, kv_b[0], kv_b[1], q_b, 0, kp2, vp2, Hq, B, nblk)
    assert_close(got, to_f64(full[cached:]), f"cached vs scratch B={B}")
    # and the oracle, on the cache it writes itself: A's tokens, then B's own ones
    hk = np.zeros((nblk, Hkv, B, D), np.uint16)
    hv = np.zeros_like(hk)
    assert ora.reshape_and_cache(kv_a[0], kv_a[1], hk, hv, slots_a) == 0
    assert ora.reshape_and_cache(kv_b[0][cached:], kv_b[1][cached:], hk, hv, slots_b) == 0
    cu = np.array([0, nb - cached], np.int32)
    rows = [0, 1, 57, nb - cached - 1]
    ref = np.stack([np.stack([ora.prefill_row(q_b[cached:], cu, hk, hv, bt_b, np.array([nb], np.int32),
                                              1 / math.sqrt(128), 0, i, h)[0] for h in range(Hq)]) for i in rows])
    assert_close(got[rows], ref, f"cached prefill vs oracle B={B}")
