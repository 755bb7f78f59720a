"""Cache slots that were never written may hold any bit pattern, NaN
included.  Attention must read only the keys 0 .. ctx-1 of each sequence:
here every slot past a sequence's context (the tail of its last page, and
every page no table uses) holds bf16 NaN in K and V, and the outputs must
still be finite and match the fp64 oracle, which reads the valid keys only."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_dev, bf16_host, need_gpu

pytestmark = pytest.mark.gpu

NAN_BF16 = np.uint16(0x7FC0)


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def poison(case):
    """K and V pools with NaN in every slot outside the sequences' contexts."""
    used = np.zeros((case.num_blocks, case.block_size), bool)
    for s in range(case.num_seqs):
        n = int(case.context_lens[s])
        for j in range(n):
            used[case.block_tables[s, j // case.block_size], j % case.block_size] = True
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    mask = ~used[:, None, :, None]  # [blocks, 1, B, 1]
    kp = np.where(mask, NAN_BF16, kp).astype(np.uint16)
    vp = np.where(mask, NAN_BF16, vp).astype(np.uint16)
    return kp, vp


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("pp", [None, 2])
def test_decode_ignores_unwritten_slots(torch, ora, monkeypatch, B, pp):
    if pp is None:
        monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
    else:
        monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    st = wl.Stream(21, B)
    ctx = st.integers(1, 300, 11)
    ctx[0] = B + 1  # a last page holding one key
    case = wl.make_decode_case("nan_tail", ctx, 32, 8, 128, B, seed=21, stream=B, with_new_tokens=False)
    kp, vp = poison(case)
    out = pa.paged_attention_decode(bf16_dev(case.q, torch), bf16_dev(kp, torch), bf16_dev(vp, torch),
                                    torch.from_numpy(case.block_tables).cuda(),
                                    torch.from_numpy(case.context_lens).cuda(), scale=case.scale,
                                    max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    ref, status = ora.decode(case.q, kp, vp, case.block_tables, case.context_lens, case.scale)
    assert np.all(status == 0) and np.all(np.isfinite(ref))
    assert_close(bf16_host(out), ref, f"decode B={B} pp={pp}")


def test_prefill_ignores_unwritten_slots(torch, ora):
    Hq, Hkv, D, B = 16, 4, 128, 32
    chunk_ctx = np.array([300, 129, 77], np.int32)
    chunk_len = np.array([70, 129, 40], np.int32)
    case = wl.make_decode_case("nan_prefill", chunk_ctx, Hq, Hkv, D, B, seed=22, stream=3, with_new_tokens=False)
    kp, vp = poison(case)
    cu = np.concatenate([[0], np.cumsum(chunk_len)]).astype(np.int32)
    qc = wl.normal_bf16(wl.Stream(22, 9), (int(cu[-1]), Hq, D))
    out = pa.paged_attention_prefill_chunk(bf16_dev(qc, torch), torch.from_numpy(cu).cuda(), bf16_dev(kp, torch),
                                           bf16_dev(vp, torch), torch.from_numpy(case.block_tables).cuda(),
                                           torch.from_numpy(chunk_ctx).cuda(), max_q_len=int(chunk_len.max()),
                                           scale=1 / math.sqrt(D), max_context_len=int(chunk_ctx.max()))
    torch.cuda.synchronize()
    got = bf16_host(out)
    rows = [0, 69, 70, 150, 198, 199, int(cu[-1]) - 1]  # first/last rows of each chunk and one inside

    def where(t):  # (chunk, row in chunk) of global row t
        r = int(np.searchsorted(cu, t, side="right")) - 1
        return r, t - int(cu[r])

    ref = np.stack([np.stack([ora.prefill_row(qc, cu, kp, vp, case.block_tables, chunk_ctx, 1 / math.sqrt(D),
                                              *where(t), h)[0] for h in range(Hq)]) for t in rows])
    assert np.all(np.isfinite(ref))
    assert_close(got[rows], ref, "prefill with NaN past the context")
