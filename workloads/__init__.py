"""Seeded synthetic inputs for the paged-attention hot path.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It holds random-number generation and the *shape* of each workload
(context lengths, page assignment, value distributions) and nothing of the
attention arithmetic itself.

Generator definitions
---------------------
* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014).  It is counter based: output ``i`` of stream
  ``(seed, stream)`` is ``mix64(base + (i + 1) * GAMMA)`` with
  ``base = mix64(seed ^ (stream * GAMMA2))``, so any slice of a stream can be
  drawn without walking the ones before it.
* Uniform doubles take the top 53 bits: ``(x >> 11) * 2**-53`` in [0, 1).
* Uniform integers in the inclusive range [lo, hi] are ``lo + floor(u * (hi-lo+1))``.
* Normal values use the Box-Muller transform in fp64: each pair of uniforms
  (u1, u2) gives ``r cos(2 pi u2)`` and ``r sin(2 pi u2)`` with
  ``r = sqrt(-2 ln(1-u1))``, emitted in that order.
* bf16 values: the fp64 normal is rounded to fp32 (round-to-nearest-even),
  then the fp32 value to bf16 (round-to-nearest-even on the bit pattern).
  Arrays of bf16 are carried as ``uint16`` bit patterns.
* A physical page assignment is a Fisher-Yates shuffle of [0, N_blk) driven by
  the same stream, consumed in order.

Pool layout (shared convention of both sides): ``k_pool``/``v_pool`` are
``bf16[N_blk][H_kv][B][D]``; block tables are ``int32[S][max_blocks]`` padded
with -1; slot mappings are ``int64`` with ``slot = page * B + offset``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import ctypes
import os

import numpy as np

_MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
GAMMA2 = 0xD1B54A32D192ED03


def _mix64_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


class Stream:
    """One SplitMix64 stream; ``draw(n)`` returns the next n raw 64-bit outputs."""

    def __init__(self, seed: int, stream: int = 0):
        self.base = _mix64_int((seed ^ ((stream * GAMMA2) & _MASK)) & _MASK)
        self.pos = 0

    def draw(self, n: int) -> np.ndarray:
        idx = np.arange(self.pos + 1, self.pos + 1 + n, dtype=np.uint64)
        self.pos += n
        with np.errstate(over="ignore"):
            z = np.uint64(self.base) + idx * np.uint64(GAMMA)
        return _mix64_np(z)

    def uniform(self, n: int) -> np.ndarray:
        return (self.draw(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def integers(self, lo: int, hi: int, n: int) -> np.ndarray:
        """n integers uniform on the inclusive range [lo, hi]."""
        u = self.uniform(n)
        return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)

    def normal(self, n: int) -> np.ndarray:
        npair = (n + 1) // 2
        out = np.empty(2 * npair, dtype=np.float64)
        step = 1 << 22
        for p0 in range(0, npair, step):
            m = min(step, npair - p0)
            u = self.uniform(2 * m)
            r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
            t = (2.0 * np.pi) * u[1::2]
            out[2 * p0: 2 * (p0 + m): 2] = r * np.cos(t)
            out[2 * p0 + 1: 2 * (p0 + m): 2] = r * np.sin(t)
        return out[:n]

    def permutation(self, n: int) -> np.ndarray:
        """Fisher-Yates shuffle of [0, n): for i = n-1 .. 1 swap a[i], a[j], j ~ U[0, i]."""
        a = np.arange(n, dtype=np.int64)
        if n < 2:
            return a
        u = self.uniform(n - 1)
        for k, i in enumerate(range(n - 1, 0, -1)):
            j = int(u[k] * (i + 1))
            a[i], a[j] = a[j], a[i]
        return a


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE on the bit pattern); returns uint16 bits."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (used for reporting only)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CLIB = None


def _clib():
    """The compiled fast path of the same generator (built on first use)."""
    global _CLIB
    if _CLIB is None:
        from . import build as _b
        path = _b.LIB
        if not os.path.exists(path):
            path = _b.build()
        lib = ctypes.CDLL(path)
        lib.wl_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        lib.wl_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        _CLIB = lib
    return _CLIB


def normal_bf16_numpy(st: Stream, shape) -> np.ndarray:
    """Reference (numpy) definition of the bf16 normal draw."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 22
    for i0 in range(0, n, step):
        m = min(step, n - i0)
        if m % 2 and i0 + m < n:
            m -= 1
        out[i0:i0 + m] = f64_to_bf16_bits(st.normal(m))
    return out.reshape(shape)


def normal_bf16(st: Stream, shape) -> np.ndarray:
    """n = prod(shape) bf16 normals from ``st`` (C fast path; same bits as the
    numpy definition).  Consumes 2*ceil(n/2) draws."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _clib().wl_normal_bf16(st.base, st.pos, n, out.ctypes.data)
    st.pos += 2 * ((n + 1) // 2)
    return out.reshape(shape)


@dataclasses.dataclass
class DecodeCase:
    """One paged decode problem: every array here is an *input* to the hot path."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    context_lens: np.ndarray      # int32 [S]   (includes this step's new token)
    block_tables: np.ndarray      # int32 [S][max_blocks], -1 padded
    q: np.ndarray                 # uint16 bf16 bits [S][Hq][D]
    k_pool: np.ndarray            # uint16 bf16 bits [N_blk][Hkv][B][D]
    v_pool: np.ndarray            # uint16 bf16 bits [N_blk][Hkv][B][D]
    new_k: Optional[np.ndarray] = None   # uint16 [T][Hkv][D]
    new_v: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None  # int64 [T]
    extra: Dict = dataclasses.field(default_factory=dict)

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if len(self.context_lens) else 0


def _assign_tables(perm: np.ndarray, ctx: np.ndarray, B: int, max_blocks: Optional[int] = None):
    """Consume ``perm`` in order, giving seq s its ceil(ctx_s / B) pages."""
    S = len(ctx)
    need = [(int(c) + B - 1) // B for c in ctx]
    mb = max(need) if max_blocks is None else max_blocks
    bt = np.full((S, max(mb, 1)), -1, dtype=np.int32)
    pos = 0
    for s in range(S):
        bt[s, : need[s]] = perm[pos : pos + need[s]]
        pos += need[s]
    return bt, pos


def _slots_for_last_token(bt: np.ndarray, ctx: np.ndarray, B: int) -> np.ndarray:
    """Slot of token ctx_s - 1 of every sequence (the token written this step)."""
    out = np.empty(len(ctx), dtype=np.int64)
    for s, c in enumerate(ctx):
        j = int(c) - 1
        out[s] = int(bt[s, j // B]) * B + (j % B)
    return out


def make_decode_case(name: str, ctx, Hq: int, Hkv: int, D: int, B: int, *,
                     seed: int = 0, stream: int = 0, pool_blocks: Optional[int] = None,
                     pool_factor: float = 1.25, scale: Optional[float] = None,
                     with_new_tokens: bool = True) -> DecodeCase:
    """Random paged decode problem with contexts ``ctx`` and a shuffled page pool.

    The pool is filled with N(0,1) bf16 values everywhere (allocated or not), the
    tables take pages from a Fisher-Yates permutation of the pool in order, and
    (optionally) one new K/V token per sequence is drawn whose slot is position
    ctx-1 of that sequence.
    """
    ctx = np.asarray(ctx, dtype=np.int32)
    S = len(ctx)
    st = Stream(seed, stream)
    used = int(sum((int(c) + B - 1) // B for c in ctx))
    nblk = pool_blocks if pool_blocks is not None else max(1, int(math.ceil(pool_factor * used)))
    perm = st.permutation(nblk)
    bt, _ = _assign_tables(perm, ctx, B)
    q = normal_bf16(st, (S, Hq, D))
    kp = normal_bf16(st, (nblk, Hkv, B, D))
    vp = normal_bf16(st, (nblk, Hkv, B, D))
    case = DecodeCase(name, S, Hq, Hkv, D, B, nblk, bt.shape[1],
                      float(scale if scale is not None else 1.0 / math.sqrt(D)),
                      ctx, bt, q, kp, vp)
    if with_new_tokens and S:
        case.new_k = normal_bf16(st, (S, Hkv, D))
        case.new_v = normal_bf16(st, (S, Hkv, D))
        case.slot_mapping = _slots_for_last_token(bt, ctx, B)
    return case


# --------------------------------------------------------------------------
# The five workloads.  Stream ids separate them; seed 0 throughout.
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 0) -> DecodeCase:
    """4 seqs, contexts {1,17,33,100}, 4 q heads = 4 kv heads, D=64, B=16,
    64-page pool, tables from a random permutation, scale 1/8, 4 new tokens."""
    return make_decode_case("tiny_decode", [1, 17, 33, 100], 4, 4, 64, 16,
                            seed=seed, stream=1, pool_blocks=64, scale=1.0 / 8.0)


def llama8b_decode(seed: int = 0, num_seqs: int = 64) -> DecodeCase:
    """Llama-3-8B-shaped decode layer: 64 seqs, ctx ~U[128,2048], 32q/8kv, D=128,
    B=16, pool 1.25x the pages used, 64 new tokens."""
    st = Stream(seed, 2)
    ctx = st.integers(128, 2048, num_seqs)
    return make_decode_case("llama8b_decode", ctx, 32, 8, 128, 16, seed=seed, stream=102)


def long_context_decode(seed: int = 0, num_seqs: int = 8, ctx_len: int = 32768) -> DecodeCase:
    """8 seqs x 32768 tokens, 64q/8kv (GQA 8), D=128, B=16, scattered pages."""
    return make_decode_case("long_context_decode", [ctx_len] * num_seqs, 64, 8, 128, 16,
                            seed=seed, stream=3)


@dataclasses.dataclass
class PrefixSharingPlan:
    """Prompt/sample structure of the prefix-sharing workload (no tables: the
    block manager under test builds those)."""
    num_prompts: int
    samples_per_prompt: int
    prefix_len: int
    suffix_lens: np.ndarray   # int64 [num_prompts]
    Hq: int
    Hkv: int
    D: int
    B: int
    num_blocks: int
    seed: int
    independent_suffixes: bool = False


def prefix_sharing_plan(seed: int = 0, num_prompts: int = 64, samples: int = 4,
                        prefix_len: int = 2048, independent_suffixes: bool = False) -> PrefixSharingPlan:
    """64 prompts x 4 samples share one 2048-token prefix; suffix ~U[1,512] per
    prompt (or per sample when ``independent_suffixes``)."""
    st = Stream(seed, 4)
    n_suf = num_prompts * (samples if independent_suffixes else 1)
    suf = st.integers(1, 512, n_suf)
    B = 16
    # pages: prefix + per-suffix pages + one page per sample for CoW / append
    pages = prefix_len // B + 1
    pages += int(sum((int(s) + B) // B + 1 for s in suf))
    pages += num_prompts * samples * 2
    nblk = int(math.ceil(1.25 * pages))
    return PrefixSharingPlan(num_prompts, samples, prefix_len, suf, 32, 8, 128, B, nblk, seed,
                             independent_suffixes)


def parallel_sampling_plan(seed: int = 0, num_prompts: int = 64, samples: int = 4, lo: int = 1024,
                           hi: int = 4096) -> PrefixSharingPlan:
    """64 prompts of U[lo, hi] tokens, 4 samples each and no prefix common to
    all prompts: the samples of a prompt share the prompt's blocks."""
    st = Stream(seed, 7)
    suf = st.integers(lo, hi, num_prompts)
    B = 16
    pages = int(sum((int(s) + B) // B + 1 for s in suf)) + num_prompts * samples * 2
    nblk = int(math.ceil(1.25 * pages))
    return PrefixSharingPlan(num_prompts, samples, 0, suf, 32, 8, 128, B, nblk, seed, False)


def prefix_sharing_values(plan: PrefixSharingPlan):
    """Pool contents, per-sequence queries and new tokens for the plan."""
    st = Stream(plan.seed, 104)
    S = plan.num_prompts * plan.samples_per_prompt
    kp = normal_bf16(st, (plan.num_blocks, plan.Hkv, plan.B, plan.D))
    vp = normal_bf16(st, (plan.num_blocks, plan.Hkv, plan.B, plan.D))
    q = normal_bf16(st, (S, plan.Hq, plan.D))
    nk = normal_bf16(st, (S, plan.Hkv, plan.D))
    nv = normal_bf16(st, (S, plan.Hkv, plan.D))
    return kp, vp, q, nk, nv


@dataclasses.dataclass
class MixedStepCase:
    """Chunked-prefill requests plus decode sequences sharing one page pool."""
    decode: DecodeCase           # the decode part (its pool is the shared pool)
    chunk_lens: np.ndarray       # int32 [R]  query tokens per chunk
    chunk_ctx: np.ndarray        # int32 [R]  context incl. the chunk
    chunk_tables: np.ndarray     # int32 [R][max_blocks]
    cu_q: np.ndarray             # int32 [R+1]
    q_chunk: np.ndarray          # uint16 [sum C][Hq][D]
    chunk_new_k: np.ndarray      # uint16 [sum C][Hkv][D]
    chunk_new_v: np.ndarray
    chunk_slots: np.ndarray      # int64 [sum C]


def make_mixed_step(name: str, chunk_lens, chunk_ctx, dec_ctx, Hq: int, Hkv: int, D: int, B: int,
                    *, seed: int = 0, stream: int = 5, pool_factor: float = 1.25) -> MixedStepCase:
    chunk_lens = np.asarray(chunk_lens, dtype=np.int32)
    chunk_ctx = np.asarray(chunk_ctx, dtype=np.int32)
    dec_ctx = np.asarray(dec_ctx, dtype=np.int32)
    assert np.all(chunk_lens <= chunk_ctx)
    st = Stream(seed, stream)
    all_ctx = np.concatenate([chunk_ctx, dec_ctx])
    used = int(sum((int(c) + B - 1) // B for c in all_ctx))
    nblk = max(1, int(math.ceil(pool_factor * used)))
    perm = st.permutation(nblk)
    mb = max((int(c) + B - 1) // B for c in all_ctx)
    bt_all, _ = _assign_tables(perm, all_ctx, B, mb)
    R = len(chunk_lens)
    kp = normal_bf16(st, (nblk, Hkv, B, D))
    vp = normal_bf16(st, (nblk, Hkv, B, D))
    Sd = len(dec_ctx)
    q_dec = normal_bf16(st, (Sd, Hq, D))
    dec = DecodeCase(name, Sd, Hq, Hkv, D, B, nblk, mb, 1.0 / math.sqrt(D), dec_ctx,
                     bt_all[R:].copy(), q_dec, kp, vp)
    dec.new_k = normal_bf16(st, (Sd, Hkv, D))
    dec.new_v = normal_bf16(st, (Sd, Hkv, D))
    dec.slot_mapping = _slots_for_last_token(dec.block_tables, dec_ctx, B)
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(chunk_lens)
    T = int(cu[-1])
    qc = normal_bf16(st, (T, Hq, D))
    ck = normal_bf16(st, (T, Hkv, D))
    cv = normal_bf16(st, (T, Hkv, D))
    slots = np.empty(T, dtype=np.int64)
    for r in range(R):
        c0 = int(chunk_ctx[r]) - int(chunk_lens[r])
        for i in range(int(chunk_lens[r])):
            j = c0 + i
            slots[cu[r] + i] = int(bt_all[r, j // B]) * B + j % B
    return MixedStepCase(dec, chunk_lens, chunk_ctx, bt_all[:R].copy(), cu, qc, ck, cv, slots)


def mixed_step(seed: int = 0, num_chunks: int = 16, chunk: int = 512, num_decode: int = 240) -> MixedStepCase:
    """16 prefill chunks of 512 query tokens over contexts ~U[512,8192] plus 240
    decode seqs with ctx ~U[64,4096]; 32q/8kv, D=128, B=32."""
    st = Stream(seed, 6)
    cctx = st.integers(chunk, 8192, num_chunks)
    dctx = st.integers(64, 4096, num_decode)
    return make_mixed_step("mixed_step", [chunk] * num_chunks, cctx, dctx, 32, 8, 128, 32,
                           seed=seed, stream=105)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "llama8b_decode": llama8b_decode,
    "long_context_decode": long_context_decode,
    "prefix_sharing": prefix_sharing_plan,
    "mixed_step": mixed_step,
}

