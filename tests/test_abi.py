"""The C-ABI library loads and exports every call include/pagedattn.h
declares; host-side validation rejects bad arguments before any GPU work.
(No compute call runs here: this file needs no GPU.)"""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_262_gb300 as pa
from paged_kv_cache_262_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pa.load()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(pa_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = declared_functions()
    assert declared, "no declarations found"
    assert declared == set(pa.EXPORTS), declared ^ set(pa.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)", out))
    assert declared <= exported, declared - exported


def test_version_and_status_strings(lib):
    assert "sm_103a" in pa.version()
    assert pa.status_string(pa.PA_ERR_WORKSPACE) == "workspace missing or too small"
    assert pa.status_string(12345) == "unknown status"


def _desc(**kw):
    d = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=10,
             max_blocks_per_seq=4, max_context_len=64, scale=0.1)
    d.update(kw)
    return pa.DecodeDesc(**d)


@pytest.mark.parametrize("kw,expect", [
    (dict(head_dim=96), pa.PA_ERR_UNSUPPORTED),
    (dict(block_size=8), pa.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), pa.PA_ERR_INVALID),
    (dict(num_q_heads=34, num_kv_heads=2), pa.PA_ERR_UNSUPPORTED),
    (dict(num_seqs=-1), pa.PA_ERR_INVALID),
    (dict(num_blocks=0), pa.PA_ERR_INVALID),
])
def test_decode_desc_validation(lib, kw, expect):
    d = _desc(**kw)
    st = lib.pa_paged_attention_decode(ctypes.byref(d), 16, 16, 16, 16, 16, 16, None, 0, None, None)
    assert st == expect
    assert lib.pa_decode_workspace_bytes(ctypes.byref(d)) == 0


def test_decode_null_and_misaligned_pointers(lib):
    d = _desc()
    assert lib.pa_paged_attention_decode(None, 16, 16, 16, 16, 16, 16, None, 0, None, None) == pa.PA_ERR_INVALID
    assert lib.pa_paged_attention_decode(ctypes.byref(d), None, 16, 16, 16, 16, 16, None, 0, None, None) == pa.PA_ERR_INVALID
    assert lib.pa_paged_attention_decode(ctypes.byref(d), 18, 16, 16, 16, 16, 16, None, 0, None, None) == pa.PA_ERR_INVALID
    # zero sequences: nothing to launch, OK without touching the GPU
    d0 = _desc(num_seqs=0)
    assert lib.pa_paged_attention_decode(ctypes.byref(d0), None, None, None, None, None, None, None, 0, None, None) == pa.PA_OK


def test_cache_call_validation(lib):
    f = lib.pa_reshape_and_cache
    assert f(16, 16, 16, 16, 16, 0, 8, 128, 16, 10, None, None) == pa.PA_OK  # nothing to write
    assert f(16, 16, 16, 16, 16, 4, 8, 100, 16, 10, None, None) == pa.PA_ERR_UNSUPPORTED
    assert f(None, 16, 16, 16, 16, 4, 8, 128, 16, 10, None, None) == pa.PA_ERR_INVALID
    assert f(24, 16, 16, 16, 16, 4, 8, 128, 16, 10, None, None) == pa.PA_ERR_INVALID
    P = ctypes.c_void_p * 1
    g = lib.pa_copy_blocks
    assert g(P(16), P(16), 1, 16, 0, 10, 4096, None, None) == pa.PA_OK  # no pairs
    assert g(P(16), P(16), 0, 16, 1, 10, 4096, None, None) == pa.PA_ERR_INVALID
    assert g(P(16), P(16), 1, 16, 1, 10, 4095, None, None) == pa.PA_ERR_INVALID
    assert g(P(None), P(16), 1, 16, 1, 10, 4096, None, None) == pa.PA_ERR_INVALID


def test_new_entry_points_validate_before_any_gpu_work(lib):
    """Decode with append, the mixed-step launch and the sub-group decode reject
    bad arguments on the host, before touching the GPU."""
    d = _desc()
    app = lib.pa_paged_attention_decode_append
    # q, new_k, new_v, slots, k_pool, v_pool, tables, ctx, out, workspace, ws_bytes, err, stream
    assert app(ctypes.byref(d), 16, None, 16, 16, 16, 16, 16, 16, 16, None, 0, None, None) == pa.PA_ERR_INVALID
    assert app(ctypes.byref(d), 16, 18, 16, 16, 16, 16, 16, 16, 16, None, 0, None, None) == pa.PA_ERR_INVALID
    assert app(ctypes.byref(_desc(head_dim=96)), 16, 16, 16, 16, 16, 16, 16, 16, 16, None, 0, None,
               None) == pa.PA_ERR_UNSUPPORTED
    mixed = lib.pa_paged_attention_mixed

    def call_mixed(pd, dd):
        return mixed(pd, 16, 16, 8, 8, 16, 16, 16, dd, 16, 16, 16, 16, None, 0, 16, 16, None, None)
    assert call_mixed(None, ctypes.byref(d)) == pa.PA_ERR_INVALID
    assert call_mixed(ctypes.byref(_desc(block_size=32)), ctypes.byref(d)) == pa.PA_ERR_INVALID  # other pools
    g3 = _desc(num_q_heads=6, num_kv_heads=2)  # a GQA group the tensor-core prefill does not build
    assert call_mixed(ctypes.byref(g3), ctypes.byref(g3)) == pa.PA_ERR_UNSUPPORTED
    sp2 = lib.pa_paged_attention_decode_shared_prefix2

    def call_sp2(desc, nsub, starts, shared, max_size):
        return sp2(ctypes.byref(desc), 16, 16, 16, 16, 16, 0, None, None, None, 0, 0, 0, nsub, starts, shared,
                   max_size, 16, 16, 1 << 20, None, None)
    assert call_sp2(d, -1, 16, 16, 4) == pa.PA_ERR_INVALID
    assert call_sp2(d, 2, None, 16, 4) == pa.PA_ERR_INVALID
    assert call_sp2(d, 2, 16, 16, 5) == pa.PA_ERR_UNSUPPORTED   # 5 members x 4 heads > 16 query rows
    assert call_sp2(_desc(head_dim=64), 2, 16, 16, 2) == pa.PA_ERR_UNSUPPORTED
    assert call_sp2(_desc(num_seqs=0), 2, 16, 16, 4) == pa.PA_OK  # nothing to decode
    for q, out in ((18, 16), (16, 24), (None, 16)):  # q and out: 16-byte aligned device pointers
        assert sp2(ctypes.byref(d), q, 16, 16, 16, 16, 0, None, None, None, 0, 0, 0, 2, 16, 16, 4, out, 16, 1 << 20,
                   None, None) == pa.PA_ERR_INVALID


def test_diagnostics_validate_before_any_gpu_work(lib):
    """The HBM probe and the bounded-wait self-test refuse bad arguments on the
    host: sizes that are not whole 16-byte words, misaligned or missing
    buffers, an unknown mode, a wait bound outside 1 .. the library's own."""
    probe = lib.pa_hbm_probe
    assert probe(16, None, 0, 0, 16, None, None) == pa.PA_ERR_INVALID      # no bytes
    assert probe(16, None, 24, 0, 16, None, None) == pa.PA_ERR_INVALID     # not a multiple of 16
    assert probe(8, None, 32, 0, 16, None, None) == pa.PA_ERR_INVALID      # misaligned source
    assert probe(None, None, 32, 0, 16, None, None) == pa.PA_ERR_INVALID
    assert probe(16, None, 32, 0, None, None, None) == pa.PA_ERR_INVALID   # read mode needs its sink
    assert probe(16, None, 32, 1, 16, None, None) == pa.PA_ERR_INVALID     # copy mode needs dst
    assert probe(16, 16, 32, 4, 16, None, None) == pa.PA_ERR_INVALID       # unknown mode
    assert probe(16, None, 4096, 3, None, None, None) == pa.PA_ERR_INVALID  # gather: not one 4 KB run a half
    wait = lib.pa_selftest_bounded_wait
    assert wait(0, None, 16, None) == pa.PA_ERR_INVALID
    assert wait(4000000001, None, 16, None) == pa.PA_ERR_INVALID
    assert wait(1000, None, None, None) == pa.PA_ERR_INVALID


def test_binding_checks_shapes_and_devices_before_any_call():
    """The plain-pointer C ABI cannot see buffer sizes, so the binding refuses
    arguments that would make a kernel read or write past a tensor: K and V
    pools of different shapes, per-sequence arrays shorter than the batch, a
    head_dim unlike the pools', an output of another shape, tensors on
    different devices."""
    import torch
    from paged_kv_cache_262_gb300 import _binding as b
    kp = torch.zeros(8, 2, 16, 64, dtype=torch.bfloat16)
    q = torch.zeros(3, 4, 64, dtype=torch.bfloat16)
    bt = torch.zeros(3, 5, dtype=torch.int32)
    ctx = torch.zeros(3, dtype=torch.int32)
    b._attn_shapes(q, kp, kp.clone(), bt, ctx, q.clone(), 3)            # consistent: no error
    bad = [
        (q, kp, torch.zeros(7, 2, 16, 64, dtype=torch.bfloat16), bt, ctx, q, 3),   # v_pool smaller
        (q, kp, kp, bt[:2], ctx, q, 3),                                            # a table row short
        (q, kp, kp, bt, ctx[:2], q, 3),                                            # a context length short
        (torch.zeros(3, 4, 128, dtype=torch.bfloat16), kp, kp, bt, ctx,
         torch.zeros(3, 4, 128, dtype=torch.bfloat16), 3),                         # head_dim 128 vs 64
        (q, kp, kp, bt, ctx, q[:2], 3),                                            # out of another shape
        (q, kp, kp, bt.to("meta"), ctx, q, 3),                                     # another device
    ]
    for args in bad:
        with pytest.raises(ValueError):
            b._attn_shapes(*args)
    with pytest.raises(ValueError):
        b._shapes(group_starts=torch.zeros(2, dtype=torch.int32), rows=(("group_starts", 3),))
    with pytest.raises(TypeError):
        b._flag(torch.zeros(1, dtype=torch.int32))                         # a host error word
    with pytest.raises(TypeError):
        b._ws(torch.zeros(16, dtype=torch.uint8))                          # a host workspace
    assert b._flag(None) is None and b._ws(None) is None


def test_default_workspaces_are_per_stream(monkeypatch):
    """Calls that pass no workspace share one per (device, stream): calls on
    one stream reuse it (they run in order), a call on another stream gets
    its own (the two may run at once), and each is allocated on its stream.
    torch.cuda's stream calls are faked, so this runs without a GPU."""
    import contextlib
    import torch
    from paged_kv_cache_262_gb300 import _binding as b

    class S:
        def __init__(self, h):
            self.cuda_stream = h

    cur, active, made = S(7), [], []
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: cur)

    @contextlib.contextmanager
    def on(s):
        active.append(s)
        yield
        active.pop()

    monkeypatch.setattr(torch.cuda, "stream", on)
    real_empty = torch.empty

    def fake_empty(n, dtype=None, device=None):
        made.append((n, active[-1].cuda_stream if active else None, device))
        return real_empty(n, dtype=dtype)

    monkeypatch.setattr(torch, "empty", fake_empty)
    cache = {}
    a = b._cached_ws(cache, 100, "cuda", None)                     # the current stream (7)
    assert b._cached_ws(cache, 80, "cuda", None) is a               # same stream: reused
    other = S(9)
    c = b._cached_ws(cache, 100, "cuda", other)
    assert c is not a                                               # another stream: its own
    d = b._cached_ws(cache, 200, torch.device("cuda", 0), None)     # grown, on stream 7
    assert d is not a and d.numel() == 200
    assert b._cached_ws(cache, 100, "cuda", other) is c
    assert [m[:2] for m in made] == [(100, 7), (100, 9), (200, 7)]
    assert all(m[2] == torch.device("cuda", 0) for m in made)


def test_every_wrapper_marshals_its_call_without_a_gpu(monkeypatch):
    """Each attention and cache wrapper runs end to end on CPU tensors against
    a recording stand-in for the library (the CUDA checks and torch.cuda's
    stream calls faked): every argument check passes on consistent shapes,
    the call reaches the library with the sizes it should, and a default
    workspace is taken from the per-stream cache."""
    import contextlib
    import torch
    import paged_kv_cache_262_gb300 as pa
    from paged_kv_cache_262_gb300 import _binding as b

    calls = []

    class Lib:
        def __getattr__(self, name):
            def f(*args):
                calls.append((name, args))
                return 4096 if name.endswith("workspace_bytes") else 0
            return f

    class S:
        cuda_stream = 7

    def need(t, dtype, name, ndim=None):  # _need without the device check
        assert isinstance(t, torch.Tensor) and t.dtype == dtype and t.is_contiguous(), name
        assert ndim is None or t.dim() == ndim, name

    monkeypatch.setattr(b, "load", lambda path=None: Lib())
    monkeypatch.setattr(b, "_need", need)
    monkeypatch.setattr(b, "_ws", lambda w: None if w is None else w.data_ptr())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: S())
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    real_empty = torch.empty
    monkeypatch.setattr(torch, "empty", lambda *a, **k: real_empty(*a, **{x: y for x, y in k.items() if x != "device"}))
    monkeypatch.setattr(b, "_WS", {})
    monkeypatch.setattr(b, "_WS_SP", {})

    bf, i32, i64 = torch.bfloat16, torch.int32, torch.int64
    S_, HQ, HKV, D, B, NB, MB = 4, 8, 2, 128, 16, 32, 6
    kp, vp = torch.zeros(NB, HKV, B, D, dtype=bf), torch.zeros(NB, HKV, B, D, dtype=bf)
    q = torch.zeros(S_, HQ, D, dtype=bf)
    bt, ctx = torch.zeros(S_, MB, dtype=i32), torch.full((S_,), 40, dtype=i32)
    err = torch.zeros(1, dtype=i32)
    nk, nv, slots = torch.zeros(S_, HKV, D, dtype=bf), torch.zeros(S_, HKV, D, dtype=bf), torch.zeros(S_, dtype=i64)

    pa.paged_attention_decode(q, kp, vp, bt, ctx, err_flag=err)
    pa.paged_attention_decode_append(q, nk, nv, slots, kp, vp, bt, ctx, err_flag=err)
    pa.paged_attention_decode_noalloc(q, kp, vp, bt, ctx, err_flag=err)
    gs, gp, pt = torch.tensor([0, 2], dtype=i32), torch.tensor([32], dtype=i32), torch.zeros(1, 2, dtype=i32)
    pa.paged_attention_decode_shared_prefix(q, kp, vp, bt, ctx, gs, gp, pt, max_group_size=2, max_prefix_len=32,
                                            err_flag=err)
    pa.paged_attention_decode_shared_prefix(q, kp, vp, bt, ctx, gs, gp, pt, max_group_size=2, max_prefix_len=32,
                                            subgroup_starts=torch.tensor([0, 2, 4], dtype=i32),
                                            subgroup_shared_lens=torch.tensor([16, 0], dtype=i32),
                                            max_subgroup_size=2, err_flag=err)
    cu = torch.tensor([0, 5, 9], dtype=i32)
    pq = torch.zeros(9, HQ, D, dtype=bf)
    pa.paged_attention_prefill_chunk(pq, cu, kp, vp, bt[:2], ctx[:2], max_q_len=5, err_flag=err)
    pa.paged_attention_mixed(pq, cu, bt[:2], ctx[:2], q, bt, ctx, kp, vp, max_q_len=5, err_flag=err)
    pa.reshape_and_cache(nk, nv, kp, vp, slots, err_flag=err)
    pa.copy_blocks([kp], [vp], torch.tensor([[1, 2]], dtype=i64), err_flag=err)

    names = [n for n, _ in calls if not n.endswith("workspace_bytes")]
    assert names == ["pa_paged_attention_decode", "pa_paged_attention_decode_append",
                     "pa_paged_attention_decode_noalloc", "pa_paged_attention_decode_shared_prefix",
                     "pa_paged_attention_decode_shared_prefix2", "pa_paged_attention_prefill_chunk",
                     "pa_paged_attention_mixed", "pa_reshape_and_cache", "pa_copy_blocks"]
    args = dict(calls)
    assert args["pa_reshape_and_cache"][5:10] == (S_, HKV, D, B, NB)
    assert args["pa_paged_attention_prefill_chunk"][3:5] == (5, 9)
    assert args["pa_paged_attention_decode_shared_prefix2"][13] == 2            # sub-groups
    assert len(b._WS) == 1 and len(b._WS_SP) == 1                              # one per (device, stream)
    # and a mismatched pool is refused before the library is reached
    n = len(calls)
    with pytest.raises(ValueError):
        pa.paged_attention_decode(q, kp, vp[:-1].contiguous(), bt, ctx)
    assert len(calls) == n
