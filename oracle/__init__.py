"""fp64 CPU oracle of the paged-attention hot path (ctypes wrapper of pa_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the product package.  It
does not import the product package and the product package does not import it.

Every function here is a thin marshalling layer over the C oracle, whose
header comment gives the passage each step follows.  ``Oracle(path)`` can load
another build of the same source (the mutation tests use that).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_c = ctypes
_P = _c.c_void_p

OK, ERR_CTX, ERR_PAGE, ERR_SLOT, ERR_ARGS = 0, 1, 2, 4, 8


def _ptr(a: np.ndarray):
    return a.ctypes.data


class Oracle:
    def __init__(self, path: Optional[str] = None):
        if path is None:
            path = _build.LIB if os.path.exists(_build.LIB) else _build.build()
        lib = _c.CDLL(path)
        i, d = _c.c_int, _c.c_double
        lib.ora_bf16_to_f64.restype = d
        lib.ora_bf16_to_f64.argtypes = [_c.c_uint16]
        lib.ora_kv_bytes_per_token.restype = _c.c_int64
        lib.ora_kv_bytes_per_token.argtypes = [_c.c_int64] * 4
        dec = [i, i, i, i, i, i, i, _P, _P, _P, _P, _P, d]
        lib.ora_decode_head.restype = i
        lib.ora_decode_head.argtypes = dec + [i, i, _P]
        lib.ora_decode.restype = i
        lib.ora_decode.argtypes = dec + [_P, _P]
        lib.ora_prefill_row.restype = i
        lib.ora_prefill_row.argtypes = [i, i, i, i, i, i, i, _P, _P, _P, _P, _P, _P, d, i, i, i, _P]
        lib.ora_partial.restype = i
        lib.ora_partial.argtypes = dec + [i, i, i, i, _P, _P, _P]
        lib.ora_combine.restype = None
        lib.ora_combine.argtypes = [i, i, _P, _P, _P, _P]
        lib.ora_reshape_and_cache.restype = i
        lib.ora_reshape_and_cache.argtypes = [i, i, i, i, i, _P, _P, _P, _P, _P]
        lib.ora_copy_blocks.restype = i
        lib.ora_copy_blocks.argtypes = [i, _P, _P, i, _c.c_int64, _P, i]
        lib.ora_swap_blocks.restype = i
        lib.ora_swap_blocks.argtypes = [i, _P, _P, _P, _P, i, i, _c.c_int64, _P, i]
        self.lib = lib
        self.path = path

    # ---- helpers -------------------------------------------------------
    @staticmethod
    def _u16(a):
        return np.ascontiguousarray(a, dtype=np.uint16)

    @staticmethod
    def _i32(a):
        return np.ascontiguousarray(a, dtype=np.int32)

    def bf16_to_f64(self, bits: int) -> float:
        return self.lib.ora_bf16_to_f64(int(bits))

    def kv_bytes_per_token(self, layers, kv_heads, head_dim, elem_bytes) -> int:
        return self.lib.ora_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)

    # ---- decode --------------------------------------------------------
    def _dec_args(self, q, k_pool, v_pool, block_tables, context_lens, Hkv, B, scale):
        q = self._u16(q)
        k_pool = self._u16(k_pool)
        v_pool = self._u16(v_pool)
        bt = self._i32(block_tables)
        ctx = self._i32(context_lens)
        S, Hq, D = q.shape
        nblk = k_pool.shape[0]
        assert k_pool.shape == (nblk, Hkv, B, D) and v_pool.shape == k_pool.shape
        mb = bt.shape[1] if bt.ndim == 2 else 0
        keep = (q, k_pool, v_pool, bt, ctx)
        args = [S, Hq, Hkv, D, B, nblk, mb, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt), _ptr(ctx),
                float(scale)]
        return keep, args

    def decode(self, q, k_pool, v_pool, block_tables, context_lens, scale, *, num_kv_heads=None,
               block_size=None):
        """All heads of all sequences: returns (out fp64 [S][Hq][D], status int32 [S])."""
        Hkv = num_kv_heads if num_kv_heads is not None else np.asarray(k_pool).shape[1]
        B = block_size if block_size is not None else np.asarray(k_pool).shape[2]
        keep, args = self._dec_args(q, k_pool, v_pool, block_tables, context_lens, Hkv, B, scale)
        S, Hq, D = keep[0].shape
        out = np.zeros((S, Hq, D), dtype=np.float64)
        st = np.zeros(S, dtype=np.int32)
        self.lib.ora_decode(*args, _ptr(out), _ptr(st))
        return out, st

    def decode_head(self, q, k_pool, v_pool, block_tables, context_lens, scale, s, h):
        """One (sequence, query head): returns (out fp64 [D], status)."""
        Hkv, B = np.asarray(k_pool).shape[1], np.asarray(k_pool).shape[2]
        keep, args = self._dec_args(q, k_pool, v_pool, block_tables, context_lens, Hkv, B, scale)
        out = np.zeros(keep[0].shape[2], dtype=np.float64)
        st = self.lib.ora_decode_head(*args, int(s), int(h), _ptr(out))
        return out, st

    def decode_case(self, case, heads: Optional[Sequence] = None):
        """Decode a ``workloads.DecodeCase`` (all heads, or the listed (s, h) pairs)."""
        if heads is None:
            return self.decode(case.q, case.k_pool, case.v_pool, case.block_tables,
                               case.context_lens, case.scale)
        res = []
        for s, h in heads:
            res.append(self.decode_head(case.q, case.k_pool, case.v_pool, case.block_tables,
                                        case.context_lens, case.scale, s, h)[0])
        return np.stack(res) if res else np.zeros((0, case.head_dim))

    def partial(self, q, k_pool, v_pool, block_tables, context_lens, scale, s, h, j0, j1):
        Hkv, B = np.asarray(k_pool).shape[1], np.asarray(k_pool).shape[2]
        keep, args = self._dec_args(q, k_pool, v_pool, block_tables, context_lens, Hkv, B, scale)
        D = keep[0].shape[2]
        m, l = _c.c_double(), _c.c_double()
        o = np.zeros(D, dtype=np.float64)
        st = self.lib.ora_partial(*args, int(s), int(h), int(j0), int(j1), _c.addressof(m),
                                  _c.addressof(l), _ptr(o))
        return m.value, l.value, o, st

    def combine(self, m, l, o):
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        o = np.ascontiguousarray(o, dtype=np.float64)
        P, D = o.shape
        out = np.zeros(D, dtype=np.float64)
        self.lib.ora_combine(P, D, _ptr(m), _ptr(l), _ptr(o), _ptr(out))
        return out

    # ---- prefill -------------------------------------------------------
    def prefill_row(self, q, cu_q, k_pool, v_pool, block_tables, context_lens, scale, r, i, h):
        q = self._u16(q)
        cu = self._i32(cu_q)
        k_pool = self._u16(k_pool)
        v_pool = self._u16(v_pool)
        bt = self._i32(block_tables)
        ctx = self._i32(context_lens)
        _, Hq, D = q.shape
        nblk, Hkv, B, _ = k_pool.shape
        out = np.zeros(D, dtype=np.float64)
        st = self.lib.ora_prefill_row(len(cu) - 1, Hq, Hkv, D, B, nblk, bt.shape[1], _ptr(q), _ptr(cu),
                                      _ptr(k_pool), _ptr(v_pool), _ptr(bt), _ptr(ctx), float(scale),
                                      int(r), int(i), int(h), _ptr(out))
        return out, st

    # ---- cache writes --------------------------------------------------
    def reshape_and_cache(self, k, v, k_pool, v_pool, slot_mapping):
        """Applies the writes to (k_pool, v_pool) IN PLACE; returns the status."""
        k = self._u16(k)
        v = self._u16(v)
        assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
        assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        T = sm.shape[0]
        nblk, Hkv, B, D = k_pool.shape
        return self.lib.ora_reshape_and_cache(T, Hkv, D, B, nblk, _ptr(k), _ptr(v), _ptr(k_pool),
                                              _ptr(v_pool), _ptr(sm))

    def copy_blocks(self, k_pools, v_pools, pairs):
        """Applies the copies to every pool IN PLACE; returns the status."""
        L = len(k_pools)
        for a in list(k_pools) + list(v_pools):
            assert a.dtype == np.uint16 and a.flags.c_contiguous
        nblk = k_pools[0].shape[0]
        blk = int(np.prod(k_pools[0].shape[1:]))
        kp = (_P * L)(*[_ptr(a) for a in k_pools])
        vp = (_P * L)(*[_ptr(a) for a in v_pools])
        pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        return self.lib.ora_copy_blocks(L, kp, vp, nblk, blk, _ptr(pr), pr.shape[0])

    def swap_blocks(self, src_k_pools, src_v_pools, dst_k_pools, dst_v_pools, pairs):
        """Moves blocks between two sets of pools (e.g. device -> host) IN
        PLACE in the destination pools; returns the status."""
        L = len(src_k_pools)
        assert len(src_v_pools) == L and len(dst_k_pools) == L and len(dst_v_pools) == L
        for a in list(src_k_pools) + list(src_v_pools) + list(dst_k_pools) + list(dst_v_pools):
            assert a.dtype == np.uint16 and a.flags.c_contiguous
        blk = int(np.prod(src_k_pools[0].shape[1:]))
        assert int(np.prod(dst_k_pools[0].shape[1:])) == blk
        arr = lambda pools: (_P * L)(*[_ptr(a) for a in pools])  # noqa: E731
        pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        return self.lib.ora_swap_blocks(L, arr(src_k_pools), arr(src_v_pools), arr(dst_k_pools), arr(dst_v_pools),
                                        src_k_pools[0].shape[0], dst_k_pools[0].shape[0], blk, _ptr(pr),
                                        pr.shape[0])


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
