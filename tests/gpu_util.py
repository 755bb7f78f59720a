"""Helpers shared by the GPU parity tests: upload seeded inputs, compare the
CUDA path's bf16 output with the fp64 oracle."""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import pytest

# Attention tolerance against the fp64 oracle (bf16 output, fp32 accumulation).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_262_gb300 import build as pbuild
    pbuild.build()
    return torch


def bf16_dev(a, torch, device="cuda"):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def bf16_host(t):
    """Device bf16 tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(gpu_bits, ref, what=""):
    g = to_f64(gpu_bits)
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max|err|={mx:.3g} mean|err|={mean:.3g}"
    return mx, mean


def upload_case(case, torch):
    d = {}
    d["q"] = bf16_dev(case.q, torch)
    d["k_pool"] = bf16_dev(case.k_pool, torch)
    d["v_pool"] = bf16_dev(case.v_pool, torch)
    d["bt"] = torch.from_numpy(np.ascontiguousarray(case.block_tables, dtype=np.int32)).cuda()
    d["ctx"] = torch.from_numpy(np.ascontiguousarray(case.context_lens, dtype=np.int32)).cuda()
    if case.new_k is not None:
        d["new_k"] = bf16_dev(case.new_k, torch)
        d["new_v"] = bf16_dev(case.new_v, torch)
        d["slots"] = torch.from_numpy(np.ascontiguousarray(case.slot_mapping, dtype=np.int64)).cuda()
    return d


def oracle_rows(ora, case, heads=None):
    """The oracle's output rows of a decode case for the listed (sequence,
    query head) pairs (every pair when None), [len(heads)][D], computed on a
    thread pool over the host cores (the oracle's C calls release the GIL).
    The case's pools must already hold what the GPU path read."""
    if heads is None:
        heads = [(s, h) for s in range(case.num_seqs) for h in range(case.num_q_heads)]
    if not heads:
        return np.zeros((0, case.head_dim))
    try:
        n = max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        n = max(1, os.cpu_count() or 1)

    def row(sh):
        out, st = ora.decode_head(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                                  case.scale, sh[0], sh[1])
        assert st == 0, f"oracle status {st} for {sh}"
        return out

    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        return np.stack(list(ex.map(row, heads)))
