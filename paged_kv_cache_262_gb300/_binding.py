"""ctypes binding of libpagedattn (``include/pagedattn.h``).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  torch supplies device memory and streams.  If the shared
library is missing the calls raise immediately -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

from . import build as _build

_c = ctypes
_P = _c.c_void_p

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_OOM, PA_ERR_WORKSPACE, PA_ERR_STATE = (
    0, -1, -2, -3, -4, -5, -6)
DEVERR_CTX, DEVERR_PAGE, DEVERR_SLOT, DEVERR_PAIR, DEVERR_TIMEOUT = 1, 2, 4, 8, 16

# Every symbol include/pagedattn.h declares.
EXPORTS = (
    "pa_version", "pa_status_string", "pa_decode_workspace_bytes", "pa_paged_attention_decode",
    "pa_paged_attention_decode_append", "pa_paged_attention_mixed",
    "pa_paged_attention_decode_noalloc", "pa_paged_attention_prefill_chunk",
    "pa_shared_prefix_workspace_bytes", "pa_paged_attention_decode_shared_prefix",
    "pa_paged_attention_decode_shared_prefix2", "pa_swap_blocks",
    "pa_bm_create_with_host", "pa_bm_swap_out", "pa_bm_swap_in", "pa_bm_num_free_host",
    "pa_bm_add_seq_tokens", "pa_bm_num_cached_blocks", "pa_reshape_and_cache", "pa_copy_blocks",
    "pa_bm_create", "pa_bm_destroy", "pa_bm_add_seq", "pa_bm_fork", "pa_bm_append", "pa_bm_free_seq",
    "pa_bm_block_table", "pa_bm_seq_len", "pa_bm_ref_count", "pa_bm_num_free", "pa_bm_wasted_slots",
    "pa_bm_append_batch", "pa_bm_block_tables", "pa_bm_append_token", "pa_hbm_probe",
    "pa_selftest_bounded_wait",
)


class DecodeDesc(_c.Structure):
    _fields_ = [("num_seqs", _c.c_int), ("num_q_heads", _c.c_int), ("num_kv_heads", _c.c_int),
                ("head_dim", _c.c_int), ("block_size", _c.c_int), ("num_blocks", _c.c_int),
                ("max_blocks_per_seq", _c.c_int), ("max_context_len", _c.c_int), ("scale", _c.c_float)]


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_LIB = None
_LOCK = threading.Lock()


def load(path: Optional[str] = None):
    """Loads the shared library (raises if it has not been built)."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"libpagedattn is not built ({p} missing); run "
                               "`python -c \"import __graft_entry__ as g; g.build()\"` at the repository root")
        lib = _c.CDLL(p)
        i, sz, i64 = _c.c_int, _c.c_size_t, _c.c_int64
        lib.pa_version.restype = _c.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_status_string.restype = _c.c_char_p
        lib.pa_status_string.argtypes = [i]
        lib.pa_decode_workspace_bytes.restype = sz
        lib.pa_decode_workspace_bytes.argtypes = [_c.POINTER(DecodeDesc)]
        lib.pa_paged_attention_decode.restype = i
        lib.pa_paged_attention_decode.argtypes = [_c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, _P, _P, sz,
                                                  _P, _P]
        lib.pa_paged_attention_decode_append.restype = i
        lib.pa_paged_attention_decode_append.argtypes = [_c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, _P, _P, _P,
                                                         _P, _P, sz, _P, _P]
        lib.pa_paged_attention_mixed.restype = i
        lib.pa_paged_attention_mixed.argtypes = [_c.POINTER(DecodeDesc), _P, _P, i, i, _P, _P, _P,
                                                 _c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, sz, _P, _P, _P, _P]
        lib.pa_paged_attention_decode_noalloc.restype = i
        lib.pa_paged_attention_decode_noalloc.argtypes = [_c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, _P, _P, _P]
        lib.pa_shared_prefix_workspace_bytes.restype = sz
        lib.pa_shared_prefix_workspace_bytes.argtypes = [_c.POINTER(DecodeDesc)]
        lib.pa_paged_attention_decode_shared_prefix.restype = i
        lib.pa_paged_attention_decode_shared_prefix.argtypes = [_c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, i, _P, _P,
                                                                _P, i, i, i, _P, _P, sz, _P, _P]
        lib.pa_paged_attention_decode_shared_prefix2.restype = i
        lib.pa_paged_attention_decode_shared_prefix2.argtypes = [_c.POINTER(DecodeDesc), _P, _P, _P, _P, _P, i, _P, _P,
                                                                 _P, i, i, i, i, _P, _P, i, _P, _P, sz, _P, _P]
        lib.pa_paged_attention_prefill_chunk.restype = i
        lib.pa_paged_attention_prefill_chunk.argtypes = [_c.POINTER(DecodeDesc), _P, _P, i, i, _P, _P, _P,
                                                         _P, _P, _P, _P]
        lib.pa_reshape_and_cache.restype = i
        lib.pa_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, i, i, i, i, i, _P, _P]
        lib.pa_copy_blocks.restype = i
        lib.pa_copy_blocks.argtypes = [_c.POINTER(_P), _c.POINTER(_P), i, _P, i, i, sz, _P, _P]
        lib.pa_bm_create.restype = _P
        lib.pa_bm_create.argtypes = [i, i]
        lib.pa_bm_create_with_host.restype = _P
        lib.pa_bm_create_with_host.argtypes = [i, i, i]
        lib.pa_bm_swap_out.restype = i
        lib.pa_bm_swap_out.argtypes = [_P, i, _c.POINTER(i64), i, _c.POINTER(i)]
        lib.pa_bm_swap_in.restype = i
        lib.pa_bm_swap_in.argtypes = [_P, i, _c.POINTER(i64), i, _c.POINTER(i)]
        lib.pa_bm_add_seq_tokens.restype = i
        lib.pa_bm_add_seq_tokens.argtypes = [_P, i, _c.POINTER(_c.c_int32), i, _c.POINTER(i)]
        lib.pa_bm_num_cached_blocks.restype = i
        lib.pa_bm_num_cached_blocks.argtypes = [_P]
        lib.pa_bm_num_free_host.restype = i
        lib.pa_bm_num_free_host.argtypes = [_P]
        lib.pa_swap_blocks.restype = i
        lib.pa_swap_blocks.argtypes = [_c.POINTER(_P), _c.POINTER(_P), _c.POINTER(_P), _c.POINTER(_P), i, _P, i, i,
                                       i, sz, _P, _P]
        lib.pa_bm_destroy.restype = None
        lib.pa_bm_destroy.argtypes = [_P]
        lib.pa_bm_add_seq.restype = i
        lib.pa_bm_add_seq.argtypes = [_P, i, i]
        lib.pa_bm_fork.restype = i
        lib.pa_bm_fork.argtypes = [_P, i, i]
        lib.pa_bm_append.restype = i
        lib.pa_bm_append.argtypes = [_P, i, _c.POINTER(i64), _c.POINTER(i64)]
        lib.pa_bm_free_seq.restype = i
        lib.pa_bm_free_seq.argtypes = [_P, i]
        lib.pa_bm_block_table.restype = i
        lib.pa_bm_block_table.argtypes = [_P, i, _c.POINTER(_c.c_int32), i, _c.POINTER(i)]
        lib.pa_bm_append_batch.restype = i
        lib.pa_bm_append_batch.argtypes = [_P, _P, _P, i, _P, _P]
        lib.pa_bm_append_token.restype = i
        lib.pa_bm_append_token.argtypes = [_P, i, _c.c_int32, _c.POINTER(i64), _c.POINTER(i64)]
        lib.pa_bm_block_tables.restype = i
        lib.pa_bm_block_tables.argtypes = [_P, _P, i, _P, i, _c.c_int32, _P]
        lib.pa_bm_seq_len.restype = i
        lib.pa_bm_seq_len.argtypes = [_P, i]
        lib.pa_bm_ref_count.restype = i
        lib.pa_bm_ref_count.argtypes = [_P, i]
        lib.pa_bm_num_free.restype = i
        lib.pa_bm_num_free.argtypes = [_P]
        lib.pa_bm_wasted_slots.restype = i64
        lib.pa_bm_wasted_slots.argtypes = [_P]
        lib.pa_hbm_probe.restype = i
        lib.pa_hbm_probe.argtypes = [_P, _P, sz, i, _P, _P, _P]
        lib.pa_selftest_bounded_wait.restype = i
        lib.pa_selftest_bounded_wait.argtypes = [_c.c_longlong, _P, _P, _P]
        if path is None:
            _LIB = lib
        return lib


def status_string(st: int) -> str:
    try:
        return load().pa_status_string(int(st)).decode()
    except Exception:
        return "unknown"


def version() -> str:
    return load().pa_version().decode()


def _check(st: int, what: str):
    if st != PA_OK:
        raise PaError(st, what)


# --------------------------------------------------------------- tensor helpers
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _flag(err_flag) -> Optional[int]:
    """The device error word the kernels OR their PA_DEVERR_* bits into."""
    if err_flag is None:
        return None
    import torch
    _need(err_flag, torch.int32, "err_flag")
    if err_flag.numel() < 1:
        raise ValueError("err_flag needs one int32")
    return err_flag.data_ptr()


def _ws(workspace) -> Optional[int]:
    if workspace is None:
        return None
    import torch
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t, dtype, name, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _shapes(*, rows=None, **named):
    """Host-side checks a plain-pointer C ABI cannot make: every tensor on one
    device, K and V pools alike, per-sequence arrays with a row for every
    sequence, head_dim as in the pools.  `rows` is (name, count) pairs that
    must have at least count rows."""
    import torch
    ts = [(n, t) for n, t in named.items() if t is not None]
    dev = ts[0][1].device
    if dev.type == "cuda" and dev.index != torch.cuda.current_device():
        raise ValueError(f"{ts[0][0]} is on {dev}, the current device is cuda:{torch.cuda.current_device()}")
    for n, t in ts:
        if t.device != dev:
            raise ValueError(f"{n} is on {t.device}, {ts[0][0]} on {dev}")
    kp, vp = named.get("k_pool"), named.get("v_pool")
    if kp is not None and vp is not None and tuple(kp.shape) != tuple(vp.shape):
        raise ValueError(f"k_pool {tuple(kp.shape)} and v_pool {tuple(vp.shape)} differ")
    for n, need in rows or ():
        if named[n].shape[0] < need:
            raise ValueError(f"{n} has {named[n].shape[0]} rows, needs {need}")


def _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, num_seqs, qname="q", oname="out",
                 tname="block_tables", cname="context_lens"):
    _shapes(**{qname: q, "k_pool": k_pool, "v_pool": v_pool, tname: block_tables, cname: context_lens,
               oname: out}, rows=((tname, num_seqs), (cname, num_seqs)))
    if q.shape[2] != k_pool.shape[3]:
        raise ValueError(f"{qname} head_dim {q.shape[2]} != the pools' {k_pool.shape[3]}")
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"{oname} must have {qname}'s shape {tuple(q.shape)}")


def make_desc(q, k_pool, block_tables, *, num_seqs=None, scale=None, max_context_len=None) -> DecodeDesc:
    import math
    nblk, hkv, bs, d = k_pool.shape
    return DecodeDesc(int(q.shape[0] if num_seqs is None else num_seqs), int(q.shape[1]), int(hkv), int(d),
                      int(bs), int(nblk), int(block_tables.shape[1]),
                      int(max_context_len if max_context_len is not None else block_tables.shape[1] * bs),
                      float(scale if scale is not None else 1.0 / math.sqrt(d)))


def decode_workspace_bytes(desc: DecodeDesc) -> int:
    return int(load().pa_decode_workspace_bytes(_c.byref(desc)))


_WS = {}
_WS_SP = {}


def _cached_ws(cache, need, device, stream):
    """A workspace of at least `need` bytes for launches on `stream` (None:
    the device's current stream), cached per (device, stream) and reused by
    later calls on that stream, which run after the earlier ones; its
    contents need no clearing between calls.  Calls on different streams
    get different workspaces, so they may run at the same time.  It is
    allocated on its stream, so replacing it with a larger one never hands
    its memory to other work while a launch on that stream may still use
    it."""
    import torch
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(idx)
    key = (idx, s.cuda_stream)
    ws = cache.get(key)
    if ws is None or ws.numel() < need:
        with torch.cuda.stream(s):
            ws = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", idx))
        cache[key] = ws
    return ws


def decode_workspace(desc: DecodeDesc, device, stream=None):
    """The workspace a decode call of `desc` needs on `stream` (None: the
    current stream), or None when it needs none; see _cached_ws."""
    need = decode_workspace_bytes(desc)
    if need == 0:
        return None
    return _cached_ws(_WS, need, device, stream)


# --------------------------------------------------------------- the four calls
def paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, out=None, *, scale=None,
                           max_context_len=None, workspace=None, err_flag=None, stream=None):
    """out[s][h] = softmax(scale q k^T) v over the paged context (see pagedattn.h)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, q.shape[0])
    desc = make_desc(q, k_pool, block_tables, scale=scale, max_context_len=max_context_len)
    if workspace is None:
        workspace = decode_workspace(desc, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_paged_attention_decode(_c.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                          _ptr(block_tables), _ptr(context_lens), _ptr(out),
                                          _ws(workspace), ws_bytes, _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_paged_attention_decode")
    return out


def paged_attention_decode_append(q, new_k, new_v, slot_mapping, k_pool, v_pool, block_tables, context_lens,
                                  out=None, *, scale=None, max_context_len=None, workspace=None, err_flag=None,
                                  stream=None):
    """The decode step's cache write and attention in one launch: each
    sequence's new token (new_k/new_v[s], position ctx-1) is stored at
    slot_mapping[s], then decode attention runs over the cache (see
    pagedattn.h)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    nblk, hkv, bs, d = k_pool.shape
    S = q.shape[0]
    if tuple(new_k.shape) != (S, hkv, d) or tuple(new_v.shape) != (S, hkv, d) or slot_mapping.shape[0] != S:
        raise ValueError("new_k/new_v must be [num_seqs][num_kv_heads][head_dim] and slot_mapping [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, S)
    _shapes(q=q, new_k=new_k, new_v=new_v, slot_mapping=slot_mapping)
    desc = make_desc(q, k_pool, block_tables, scale=scale, max_context_len=max_context_len)
    if workspace is None:
        workspace = decode_workspace(desc, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_paged_attention_decode_append(_c.byref(desc), _ptr(q), _ptr(new_k), _ptr(new_v),
                                                 _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool),
                                                 _ptr(block_tables), _ptr(context_lens), _ptr(out),
                                                 _ws(workspace), ws_bytes, _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_paged_attention_decode_append")
    return out


NOALLOC_SCRATCH_BYTES = 8 << 20


def paged_attention_decode_shared_prefix(q, k_pool, v_pool, block_tables, context_lens, group_starts,
                                         group_prefix_lens, prefix_tables, out=None, *, max_group_size,
                                         max_prefix_len, scale=None, max_context_len=None, workspace=None,
                                         err_flag=None, stream=None, subgroup_starts=None,
                                         subgroup_shared_lens=None, max_subgroup_size=0):
    """Decode with each group's shared prefix attended once; with sub-groups
    (subgroup_starts / subgroup_shared_lens), a second level of sharing read
    once per sub-group (see pagedattn.h)."""
    import torch
    for t, n, dt, nd in ((q, "q", torch.bfloat16, 3), (k_pool, "k_pool", torch.bfloat16, 4),
                         (v_pool, "v_pool", torch.bfloat16, 4), (block_tables, "block_tables", torch.int32, 2),
                         (context_lens, "context_lens", torch.int32, 1), (group_starts, "group_starts", torch.int32, 1),
                         (group_prefix_lens, "group_prefix_lens", torch.int32, 1),
                         (prefix_tables, "prefix_tables", torch.int32, 2)):
        _need(t, dt, n, nd)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, q.shape[0])
    ng0 = int(group_prefix_lens.shape[0])
    _shapes(q=q, group_starts=group_starts, group_prefix_lens=group_prefix_lens, prefix_tables=prefix_tables,
            subgroup_starts=subgroup_starts, subgroup_shared_lens=subgroup_shared_lens,
            rows=(("group_starts", ng0 + 1 if ng0 else 0), ("prefix_tables", ng0)))
    if subgroup_shared_lens is not None and subgroup_starts is not None and \
            subgroup_starts.shape[0] < subgroup_shared_lens.shape[0] + 1:
        raise ValueError("subgroup_starts needs num_subgroups + 1 entries")
    desc = make_desc(q, k_pool, block_tables, scale=scale, max_context_len=max_context_len)
    if workspace is None:
        need = int(load().pa_shared_prefix_workspace_bytes(_c.byref(desc)))
        workspace = _cached_ws(_WS_SP, need, q.device, stream)
    ng = int(group_prefix_lens.shape[0])
    if subgroup_starts is None:
        st = load().pa_paged_attention_decode_shared_prefix(
            _c.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens), ng,
            _ptr(group_starts), _ptr(group_prefix_lens), _ptr(prefix_tables), int(prefix_tables.shape[1]),
            int(max_group_size), int(max_prefix_len), _ptr(out), _ws(workspace),
            workspace.numel() * workspace.element_size(), _flag(err_flag), _stream_ptr(stream))
        _check(st, "pa_paged_attention_decode_shared_prefix")
        return out
    _need(subgroup_starts, torch.int32, "subgroup_starts", 1)
    _need(subgroup_shared_lens, torch.int32, "subgroup_shared_lens", 1)
    st = load().pa_paged_attention_decode_shared_prefix2(
        _c.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens), ng,
        _ptr(group_starts), _ptr(group_prefix_lens), _ptr(prefix_tables), int(prefix_tables.shape[1]),
        int(max_group_size), int(max_prefix_len), int(subgroup_shared_lens.shape[0]), _ptr(subgroup_starts),
        _ptr(subgroup_shared_lens), int(max_subgroup_size), _ptr(out), _ws(workspace),
        workspace.numel() * workspace.element_size(), _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_paged_attention_decode_shared_prefix2")
    return out


def paged_attention_decode_noalloc(q, k_pool, v_pool, block_tables, context_lens, out=None, *, scale=None,
                                   max_context_len=None, err_flag=None, stream=None):
    """Decode attention without a workspace (fixed device scratch array; for
    callers that cannot allocate device memory -- see pagedattn.h)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, q.shape[0])
    desc = make_desc(q, k_pool, block_tables, scale=scale, max_context_len=max_context_len)
    st = load().pa_paged_attention_decode_noalloc(_c.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                  _ptr(block_tables), _ptr(context_lens), _ptr(out),
                                                  _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_paged_attention_decode_noalloc")
    return out


def paged_attention_prefill_chunk(q, cu_q, k_pool, v_pool, block_tables, context_lens, out=None, *,
                                  max_q_len, scale=None, max_context_len=None, err_flag=None, stream=None):
    """Causal chunked-prefill attention (see pagedattn.h)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    R = context_lens.shape[0]
    _attn_shapes(q, k_pool, v_pool, block_tables, context_lens, out, R)
    _shapes(q=q, cu_q=cu_q, rows=(("cu_q", R + 1),))
    desc = make_desc(q, k_pool, block_tables, num_seqs=context_lens.shape[0], scale=scale,
                     max_context_len=max_context_len)
    st = load().pa_paged_attention_prefill_chunk(_c.byref(desc), _ptr(q), _ptr(cu_q), int(max_q_len),
                                                 int(q.shape[0]), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                                 _ptr(context_lens), _ptr(out), _flag(err_flag),
                                                 _stream_ptr(stream))
    _check(st, "pa_paged_attention_prefill_chunk")
    return out


def paged_attention_mixed(prefill_q, cu_q, prefill_tables, prefill_context_lens, decode_q, decode_tables,
                          decode_context_lens, k_pool, v_pool, prefill_out=None, decode_out=None, *, max_q_len,
                          scale=None, prefill_max_context_len=None, decode_max_context_len=None, workspace=None,
                          err_flag=None, stream=None):
    """A continuous-batching step's chunked prefill and decode in one launch,
    side by side (see pagedattn.h); returns (prefill_out, decode_out)."""
    import torch
    _need(prefill_q, torch.bfloat16, "prefill_q", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    _need(prefill_tables, torch.int32, "prefill_tables", 2)
    _need(prefill_context_lens, torch.int32, "prefill_context_lens", 1)
    _need(decode_q, torch.bfloat16, "decode_q", 3)
    _need(decode_tables, torch.int32, "decode_tables", 2)
    _need(decode_context_lens, torch.int32, "decode_context_lens", 1)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    if prefill_out is None:
        prefill_out = torch.empty_like(prefill_q)
    if decode_out is None:
        decode_out = torch.empty_like(decode_q)
    _need(prefill_out, torch.bfloat16, "prefill_out", 3)
    _need(decode_out, torch.bfloat16, "decode_out", 3)
    R = prefill_context_lens.shape[0]
    _attn_shapes(prefill_q, k_pool, v_pool, prefill_tables, prefill_context_lens, prefill_out, R, "prefill_q",
                 "prefill_out", "prefill_tables", "prefill_context_lens")
    _shapes(prefill_q=prefill_q, cu_q=cu_q, rows=(("cu_q", R + 1),))
    _attn_shapes(decode_q, k_pool, v_pool, decode_tables, decode_context_lens, decode_out, decode_q.shape[0],
                 "decode_q", "decode_out", "decode_tables", "decode_context_lens")
    _shapes(prefill_q=prefill_q, decode_q=decode_q)
    pdesc = make_desc(prefill_q, k_pool, prefill_tables, num_seqs=prefill_context_lens.shape[0], scale=scale,
                      max_context_len=prefill_max_context_len)
    ddesc = make_desc(decode_q, k_pool, decode_tables, scale=scale, max_context_len=decode_max_context_len)
    if workspace is None:
        workspace = decode_workspace(ddesc, decode_q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_paged_attention_mixed(_c.byref(pdesc), _ptr(prefill_q), _ptr(cu_q), int(max_q_len),
                                         int(prefill_q.shape[0]), _ptr(prefill_tables), _ptr(prefill_context_lens),
                                         _ptr(prefill_out), _c.byref(ddesc), _ptr(decode_q), _ptr(decode_tables),
                                         _ptr(decode_context_lens), _ptr(decode_out), _ws(workspace), ws_bytes,
                                         _ptr(k_pool), _ptr(v_pool), _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_paged_attention_mixed")
    return prefill_out, decode_out


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, *, err_flag=None, stream=None):
    """k_pool[slot // B][h][slot % B] = k[t][h] (and v) for every token t."""
    import torch
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(k_pool, torch.bfloat16, "k_pool", 4)
    _need(v_pool, torch.bfloat16, "v_pool", 4)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    nblk, hkv, bs, d = k_pool.shape
    _shapes(k=k, v=v, k_pool=k_pool, v_pool=v_pool, slot_mapping=slot_mapping)
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, hkv, d) or tuple(v.shape) != (T, hkv, d):
        raise ValueError(f"k and v must be [{T}][{hkv}][{d}] (a row per slot_mapping entry)")
    st = load().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping),
                                     int(slot_mapping.shape[0]), int(hkv), int(d), int(bs), int(nblk),
                                     _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_reshape_and_cache")


def copy_blocks(k_pools: Sequence, v_pools: Sequence, block_pairs, *, err_flag=None, stream=None):
    """Block pairs[i][1] := block pairs[i][0] in every layer's K and V pool."""
    import torch
    L = len(k_pools)
    if L != len(v_pools) or L == 0:
        raise ValueError("k_pools and v_pools must be non-empty and of equal length")
    for t in list(k_pools) + list(v_pools):
        _need(t, torch.bfloat16, "pool", 4)
    _need(block_pairs, torch.int64, "block_pairs", 2)
    for t in list(k_pools) + list(v_pools):
        if tuple(t.shape) != tuple(k_pools[0].shape) or t.device != block_pairs.device:
            raise ValueError("every pool must have the first pool's shape, on block_pairs' device")
    if block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be [num_pairs][2]")
    nblk = k_pools[0].shape[0]
    blk_bytes = k_pools[0][0].numel() * 2
    kp = (_P * L)(*[t.data_ptr() for t in k_pools])
    vp = (_P * L)(*[t.data_ptr() for t in v_pools])
    st = load().pa_copy_blocks(kp, vp, L, _ptr(block_pairs), int(block_pairs.shape[0]), int(nblk),
                               int(blk_bytes), _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_copy_blocks")


def swap_blocks(src_k_pools: Sequence, src_v_pools: Sequence, dst_k_pools: Sequence, dst_v_pools: Sequence,
                block_pairs, *, err_flag=None, stream=None):
    """dst block pairs[i][1] := src block pairs[i][0] for every layer, K and V;
    pools are CUDA tensors or pinned host tensors (see pagedattn.h)."""
    import torch
    L = len(src_k_pools)
    pools = [list(src_k_pools), list(src_v_pools), list(dst_k_pools), list(dst_v_pools)]
    if L == 0 or any(len(p) != L for p in pools):
        raise ValueError("pool lists must be non-empty and of equal length")
    for p in pools:
        for t in p:
            if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
                raise TypeError("pools must be contiguous 4-D bf16 tensors")
            if not t.is_cuda and not t.is_pinned():
                raise ValueError("host pools must be pinned")
    _need(block_pairs, torch.int64, "block_pairs", 2)
    if block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be [num_pairs][2]")
    for p in pools:
        if any(tuple(t.shape) != tuple(p[0].shape) for t in p):
            raise ValueError("the pools of one side must all have the same shape")
    if tuple(src_k_pools[0].shape[1:]) != tuple(dst_k_pools[0].shape[1:]):
        raise ValueError("source and destination blocks must have the same shape")
    arr = [(_P * L)(*[t.data_ptr() for t in p]) for p in pools]
    st = load().pa_swap_blocks(arr[0], arr[1], arr[2], arr[3], L, _ptr(block_pairs), int(block_pairs.shape[0]),
                               int(src_k_pools[0].shape[0]), int(dst_k_pools[0].shape[0]),
                               int(src_k_pools[0][0].numel() * 2), _flag(err_flag), _stream_ptr(stream))
    _check(st, "pa_swap_blocks")


# --------------------------------------------------------------- block manager
class BlockManager:
    """Host block manager (free list, block tables, ref counts, copy-on-write)."""

    def __init__(self, num_blocks: int, block_size: int, num_host_blocks: int = 0):
        self._lib = load()
        self._h = self._lib.pa_bm_create_with_host(int(num_blocks), int(num_host_blocks), int(block_size))
        if not self._h:  # NULL: bad sizes, or no host memory for valid ones
            bad = int(num_blocks) <= 0 or int(num_host_blocks) < 0 or int(block_size) <= 0
            raise PaError(PA_ERR_INVALID if bad else PA_ERR_OOM, "pa_bm_create")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int, num_tokens: int):
        _check(self._lib.pa_bm_add_seq(self._h, int(seq_id), int(num_tokens)), "pa_bm_add_seq")

    def fork(self, parent: int, child: int):
        _check(self._lib.pa_bm_fork(self._h, int(parent), int(child)), "pa_bm_fork")

    def append(self, seq_id: int, token: Optional[int] = None):
        """Returns (slot, cow_pair or None).  With the token's id, a block it
        fills is registered in the prefix cache (pa_bm_append_token)."""
        slot = _c.c_int64()
        pair = (_c.c_int64 * 2)()
        if token is None:
            _check(self._lib.pa_bm_append(self._h, int(seq_id), _c.byref(slot), pair), "pa_bm_append")
        else:
            _check(self._lib.pa_bm_append_token(self._h, int(seq_id), int(token), _c.byref(slot), pair),
                   "pa_bm_append_token")
        return slot.value, (None if pair[0] < 0 else (pair[0], pair[1]))

    def append_batch(self, seq_ids, tokens=None):
        """One token onto each of `seq_ids` (distinct), in order, in one call;
        `tokens` (optional, one id per sequence) as in append.  Returns
        (slots int64 [n], cow_pairs int64 [n, 2]; -1 rows: no copy); on an
        error nothing has changed."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32).reshape(-1)
        tok = None
        if tokens is not None:
            tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
            if tok.size != ids.size:
                raise ValueError("tokens needs one id per sequence")
        slots = np.empty(ids.size, np.int64)
        cows = np.empty((ids.size, 2), np.int64)
        _check(self._lib.pa_bm_append_batch(self._h, ids.ctypes.data, None if tok is None else tok.ctypes.data,
                                            int(ids.size), slots.ctypes.data, cows.ctypes.data),
               "pa_bm_append_batch")
        return slots, cows

    def block_tables(self, seq_ids, max_blocks: int, pad: int = -1):
        """Padded block-table matrix int32 [n, max_blocks] and context lengths
        int32 [n] of `seq_ids`, as the attention calls take them.  The default
        pad is no block: an entry read past a context would be refused by the
        kernels' page check rather than read block 0."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32).reshape(-1)
        out = np.empty((ids.size, int(max_blocks)), np.int32)
        lens = np.empty(ids.size, np.int32)
        _check(self._lib.pa_bm_block_tables(self._h, ids.ctypes.data, int(ids.size), out.ctypes.data,
                                            int(max_blocks), int(pad), lens.ctypes.data), "pa_bm_block_tables")
        return out, lens

    def free_seq(self, seq_id: int):
        _check(self._lib.pa_bm_free_seq(self._h, int(seq_id)), "pa_bm_free_seq")

    def block_table(self, seq_id: int):
        n = _c.c_int()
        st = self._lib.pa_bm_block_table(self._h, int(seq_id), None, 0, _c.byref(n))
        if st not in (PA_OK, PA_ERR_INVALID):
            raise PaError(st, "pa_bm_block_table")
        buf = (_c.c_int32 * max(n.value, 1))()
        _check(self._lib.pa_bm_block_table(self._h, int(seq_id), buf, n.value, _c.byref(n)),
               "pa_bm_block_table")
        return list(buf[: n.value])

    def _swap(self, fn, seq_id):
        n = _c.c_int()
        cap = 1
        while True:
            buf = (_c.c_int64 * (2 * cap))()
            st = fn(self._h, int(seq_id), buf, cap, _c.byref(n))
            if st == PA_ERR_INVALID and n.value > cap:
                cap = n.value
                continue
            _check(st, fn.__name__)
            return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]

    def swap_out(self, seq_id: int):
        """Returns the (device block, host block) pairs to copy."""
        return self._swap(self._lib.pa_bm_swap_out, seq_id)

    def swap_in(self, seq_id: int):
        """Returns the (host block, device block) pairs to copy."""
        return self._swap(self._lib.pa_bm_swap_in, seq_id)

    def add_seq_tokens(self, seq_id: int, tokens) -> int:
        """New sequence holding the prompt `tokens` (a 1-D sequence of int32
        token ids; a contiguous int32 numpy array is passed without a copy);
        returns how many leading tokens were found in the prefix cache."""
        import numpy as np
        arr = np.ascontiguousarray(tokens, dtype=np.int32)
        if arr.ndim != 1:
            raise ValueError("tokens must be 1-D")
        cached = _c.c_int()
        ptr = arr.ctypes.data_as(_c.POINTER(_c.c_int32)) if arr.size else None
        _check(self._lib.pa_bm_add_seq_tokens(self._h, int(seq_id), ptr, int(arr.size), _c.byref(cached)),
               "pa_bm_add_seq_tokens")
        return cached.value

    def num_cached_blocks(self) -> int:
        return self._lib.pa_bm_num_cached_blocks(self._h)

    def num_free_host(self) -> int:
        return self._lib.pa_bm_num_free_host(self._h)

    def seq_len(self, seq_id: int) -> int:
        return self._lib.pa_bm_seq_len(self._h, int(seq_id))

    def ref_count(self, block: int) -> int:
        return self._lib.pa_bm_ref_count(self._h, int(block))

    def num_free(self) -> int:
        return self._lib.pa_bm_num_free(self._h)

    def wasted_slots(self) -> int:
        return self._lib.pa_bm_wasted_slots(self._h)


# ------------------------------------------------------------------ diagnostics
def hbm_probe(src, *, dst=None, sink=None, tma=False, gather=False, err_flag=None, stream=None):
    """Streams ``src`` (a contiguous CUDA tensor, nbytes a multiple of 16):
    read only through 16-byte vector loads (dst None; sink: a CUDA tensor of
    at least 16 bytes, allocated here when not given), read only through TMA
    bulk copies into shared memory (tma=True), read as paged decode reads
    (gather=True: 4 KB K/V runs at scattered places; the bytes read are the
    largest power-of-two number of runs fitting each half, times 2 x 4096), or
    copied into dst (same nbytes).  Asynchronous; returns nothing."""
    import torch
    if not isinstance(src, torch.Tensor) or not src.is_cuda or not src.is_contiguous():
        raise TypeError("src must be a contiguous CUDA tensor")
    nbytes = src.numel() * src.element_size()
    mode = 3 if gather else 2 if tma else 0 if dst is None else 1
    if mode >= 2:
        if dst is not None:
            raise ValueError("the TMA read modes take no dst")
    elif mode == 1:
        if not isinstance(dst, torch.Tensor) or not dst.is_cuda or not dst.is_contiguous() or \
                dst.numel() * dst.element_size() != nbytes or dst.device != src.device:
            raise ValueError("dst must be a contiguous CUDA tensor of src's size on src's device")
    elif sink is None:
        sink = torch.empty(16, dtype=torch.uint8, device=src.device)
    elif not isinstance(sink, torch.Tensor) or not sink.is_cuda or sink.numel() * sink.element_size() < 16:
        raise ValueError("sink must be a CUDA tensor of at least 16 bytes")
    _check(load().pa_hbm_probe(src.data_ptr(), _ptr(dst), nbytes, mode, _ptr(sink) if mode == 0 else None,
                               _flag(err_flag), _stream_ptr(stream)), "pa_hbm_probe")


def selftest_bounded_wait(limit_cycles: int, err_flag, done, *, stream=None):
    """Launches the bounded-wait self-test: one warp waits at most
    ``limit_cycles`` SM cycles on an mbarrier nothing arrives on, reports
    PA_DEVERR_TIMEOUT into ``err_flag`` and sets ``done`` (CUDA int32) to 1."""
    import torch
    _need(done, torch.int32, "done")
    _check(load().pa_selftest_bounded_wait(int(limit_cycles), _flag(err_flag), done.data_ptr(), _stream_ptr(stream)),
           "pa_selftest_bounded_wait")
