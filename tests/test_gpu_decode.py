"""GPU parity of paged decode attention (and its cache write) with the fp64
oracle, through the C-ABI library."""
import math

import numpy as np
import pytest

import paged_kv_cache_262_gb300 as pa
import workloads as wl
from gpu_util import assert_close, bf16_host, need_gpu, oracle_rows, upload_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.fixture
def parts(monkeypatch):
    """Forces the decode split-K part length (pages) for one test."""
    def set_(pp):
        if pp is None:
            monkeypatch.delenv("PA_PARTITION_PAGES", raising=False)
        else:
            monkeypatch.setenv("PA_PARTITION_PAGES", str(pp))
    return set_


def run_step(torch, case, d, err=None):
    """reshape_and_cache of the step's new tokens, then decode."""
    if "new_k" in d:
        pa.reshape_and_cache(d["new_k"], d["new_v"], d["k_pool"], d["v_pool"], d["slots"], err_flag=err)
    out = pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"], scale=case.scale,
                                    max_context_len=case.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    return out


def oracle_step(ora, case):
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    if case.new_k is not None:
        assert ora.reshape_and_cache(case.new_k, case.new_v, kp, vp, case.slot_mapping) == 0
    return kp, vp


def test_tiny_decode_with_cache_write(torch, ora):
    case = wl.tiny_decode()
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(torch, case, d, err)
    kp, vp = oracle_step(ora, case)
    assert np.array_equal(bf16_host(d["k_pool"]), kp) and np.array_equal(bf16_host(d["v_pool"]), vp)
    ref, st = ora.decode(case.q, kp, vp, case.block_tables, case.context_lens, case.scale)
    assert np.all(st == 0) and int(err.item()) == 0
    assert_close(bf16_host(out), ref, "tiny_decode")
    # ctx = 1 sequence: the output is its only value vector, exactly
    v0 = vp[case.block_tables[0, 0], :, 0, :]
    assert np.array_equal(bf16_host(out)[0], v0)


@pytest.mark.parametrize("pp", [None, 8])
def test_llama8b_decode_full(torch, ora, parts, pp):
    parts(pp)
    case = wl.llama8b_decode()
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(torch, case, d, err)
    kp, vp = oracle_step(ora, case)
    assert np.array_equal(bf16_host(d["k_pool"]), kp)
    ref, st = ora.decode(case.q, kp, vp, case.block_tables, case.context_lens, case.scale)
    assert int(err.item()) == 0
    assert_close(bf16_host(out), ref, f"llama8b_decode pp={pp}")


def test_long_context_decode_full(torch, ora):
    """8 x 32768 tokens, GQA 8, split-K: every (sequence, query head) row
    against the oracle."""
    case = wl.long_context_decode()
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(torch, case, d, err)
    kp, vp = oracle_step(ora, case)
    got = bf16_host(out)
    sub = case.__class__(**{**case.__dict__, "k_pool": kp, "v_pool": vp})
    ref = oracle_rows(ora, sub).reshape(got.shape)
    assert int(err.item()) == 0
    assert_close(got, ref, "long_context_decode")


SHAPES = [  # (Hq, Hkv, D, B)
    (4, 4, 64, 16), (8, 2, 64, 32), (32, 8, 128, 16), (64, 8, 128, 16), (32, 8, 128, 32),
    (16, 1, 128, 16), (6, 2, 128, 32), (2, 2, 128, 16), (48, 4, 64, 16),
]
CTX = [1, 2, 15, 16, 17, 31, 32, 33, 100, 257, 513, 1000, 1999]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "q%dkv%dd%db%d" % s)
@pytest.mark.parametrize("pp", [None, 1, 3])
@pytest.mark.parametrize("lpt", [None, "1", "0"])
def test_ragged_shapes(torch, ora, parts, monkeypatch, shape, pp, lpt):
    """Every CTA order: the launcher's choice, longest context first, grid order."""
    Hq, Hkv, D, B = shape
    parts(pp)
    if lpt is None:
        monkeypatch.delenv("PA_DECODE_LPT", raising=False)
    else:
        monkeypatch.setenv("PA_DECODE_LPT", lpt)
    case = wl.make_decode_case("ragged", CTX, Hq, Hkv, D, B, seed=7, stream=hash(shape) % 1000,
                               scale=1.0 / math.sqrt(D), with_new_tokens=False)
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(torch, case, d, err)
    ref, st = ora.decode_case(case)
    assert int(err.item()) == 0 and np.all(st == 0)
    assert_close(bf16_host(out), ref, f"{shape} pp={pp} lpt={lpt}")


def _relaid(case, seed):
    """Same logical K/V under another physical page assignment."""
    st = wl.Stream(seed, 1)
    perm = st.permutation(case.num_blocks)
    kp = np.empty_like(case.k_pool)
    vp = np.empty_like(case.v_pool)
    kp[perm] = case.k_pool
    vp[perm] = case.v_pool
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    return case.__class__(**{**case.__dict__, "k_pool": kp, "v_pool": vp, "block_tables": bt})


@pytest.mark.parametrize("pp", [None, 2])
def test_physical_permutation_bit_identical(torch, parts, pp):
    parts(pp)
    case = wl.make_decode_case("perm", [5, 300, 64, 1031], 32, 8, 128, 16, seed=3, with_new_tokens=False)
    outs = []
    for c in (case, _relaid(case, 11), _relaid(case, 12)):
        d = upload_case(c, torch)
        outs.append(bf16_host(run_step(torch, c, d)))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_vs_private_copies_bit_identical(torch):
    case = wl.make_decode_case("share", [200, 200, 200], 16, 4, 128, 16, seed=4, pool_blocks=60,
                               with_new_tokens=False)
    bt = case.block_tables.copy()
    bt[1, :10] = bt[0, :10]  # seqs 0,1,2 share the first 10 pages of seq 0
    bt[2, :10] = bt[0, :10]
    shared = case.__class__(**{**case.__dict__, "block_tables": bt})
    priv_bt = bt.copy()
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    free = [b for b in range(case.num_blocks) if b not in set(bt.flatten().tolist())]
    for s in (1, 2):
        for i in range(10):
            nb = free.pop()
            kp[nb], vp[nb] = kp[bt[0, i]], vp[bt[0, i]]
            priv_bt[s, i] = nb
    private = case.__class__(**{**case.__dict__, "block_tables": priv_bt, "k_pool": kp, "v_pool": vp})
    a = bf16_host(run_step(torch, shared, upload_case(shared, torch)))
    b = bf16_host(run_step(torch, private, upload_case(private, torch)))
    assert np.array_equal(a, b)


def test_device_errors_flagged_not_trapped(torch, ora):
    case = wl.make_decode_case("err", [0, 40, 33, 50], 8, 2, 128, 16, seed=5, pool_blocks=20,
                               with_new_tokens=False)
    bt = case.block_tables.copy()
    bt[2, 1] = 10_000  # page id outside the pool
    case = case.__class__(**{**case.__dict__, "block_tables": bt})
    d = upload_case(case, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"], scale=case.scale,
                                    max_context_len=48, err_flag=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_CTX and e & pa.DEVERR_PAGE
    got = bf16_host(out)
    assert not np.any(got[0]) and not np.any(got[3])  # ctx 0 and ctx 50 > max_context_len
    ref = ora.decode_case(case, heads=[(1, h) for h in range(8)])
    assert_close(got[1], ref, "valid sequence beside bad ones")


def test_workspace_rejected_when_too_small(torch):
    case = wl.make_decode_case("ws", [4000], 8, 2, 128, 16, seed=6, with_new_tokens=False)
    d = upload_case(case, torch)
    desc = pa.make_desc(d["q"], d["k_pool"], d["bt"], max_context_len=4000)
    need = pa.decode_workspace_bytes(desc)
    assert need > 0
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"],
                                  max_context_len=4000, workspace=small)
    assert e.value.status == pa.PA_ERR_WORKSPACE


def test_repeated_calls_reuse_workspace(torch, ora, parts):
    """Split-K counters reset themselves: many calls on one workspace agree."""
    parts(2)
    case = wl.make_decode_case("rep", [700, 33, 1200], 16, 2, 128, 16, seed=8, with_new_tokens=False)
    d = upload_case(case, torch)
    first = bf16_host(run_step(torch, case, d))
    for _ in range(5):
        assert np.array_equal(bf16_host(run_step(torch, case, d)), first)
    ref, _ = ora.decode_case(case)
    assert_close(first, ref, "repeat")


def test_workspace_needs_no_clearing(torch, ora, parts):
    """Garbage in the workspace and calls of different split layouts sharing
    one workspace do not change results (epoch-tagged arrival counters)."""
    parts(3)
    a = wl.make_decode_case("wa", [900, 40, 1300], 16, 2, 128, 16, seed=9, with_new_tokens=False)
    b = wl.make_decode_case("wb", [2000, 2000, 17, 600, 5], 8, 4, 64, 32, seed=10, with_new_tokens=False)
    da, db = upload_case(a, torch), upload_case(b, torch)
    need = max(pa.decode_workspace_bytes(pa.make_desc(d["q"], d["k_pool"], d["bt"], max_context_len=c.max_context_len))
               for d, c in ((da, a), (db, b)))
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    ref_a, _ = ora.decode_case(a)
    ref_b, _ = ora.decode_case(b)
    for _ in range(3):
        for d, c, ref in ((da, a, ref_a), (db, b, ref_b)):
            out = pa.paged_attention_decode(d["q"], d["k_pool"], d["v_pool"], d["bt"], d["ctx"], scale=c.scale,
                                            max_context_len=c.max_context_len, workspace=ws)
            torch.cuda.synchronize()
            assert_close(bf16_host(out), ref, c.name)
        ws[: need // 2].random_(0, 256)  # scribble over partial results and counters
