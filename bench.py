"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

One step = one pass of the hot path over one batch of synthetic input from the
seeded generator in ``workloads``:

* decode workloads (default ``llama8b_decode``: 64 seqs, ctx ~U[128,2048],
  32q/8kv heads, D=128, B=16; also ``long_context_decode``, ``tiny_decode``):
  each sequence's new token stored in the cache and paged decode attention, in
  one decode-with-append launch (``--separate-append``: reshape_and_cache,
  then decode);
* ``prefix_sharing``: 64 prompts x 4 samples over a 2048-token prefix built by
  the host block manager; copy_blocks of the copy-on-write pairs,
  reshape_and_cache of the appended tokens, decode over the shared tables;
* ``parallel_sampling``: 64 prompts of U[1024,4096] tokens x 4 samples, no
  prefix common to all: each prompt's blocks shared by its samples
  (sub-groups; ``--sharing one-level``: each prompt a group;
  ``--plain-decode``);
* ``swap``: preemption -- 16 sequences x 2048 tokens (8 kv heads, D=128,
  B=16, 4 layers; blocks scattered over the pool) to a pinned host pool and
  back to new device blocks, pairs from the block manager (swap_blocks; the
  link's reference rate is a copy-engine copy of the same bytes, measured in
  the same run);
* ``block_manager``: the host block manager alone (no GPU): 64 prompts x 4
  samples admitted with prefix-cache lookups (a 2048-token system prompt
  common to all, then each prompt's U[1,512] tokens), forked per sample, one
  append each (copy-on-write); 64 unshared sequences swapped out and in;
  everything freed; operations per second of host time;
* ``mixed_step``: one reshape_and_cache of every new token, then chunked
  prefill of 16 x 512 query tokens (tensor cores) and decode of 240 sequences
  (B=32) in one mixed-step launch whose CTAs run the two side by side
  (``--mixed-launch separate``: two launches).

To keep reads coming from HBM, each step uses the next of NL layer pools
(separate copies of the cache, together several times the 129 MB L2).

Prints ONE JSON line.  ``value`` is algorithmic HBM bytes per second over the
device-timed step: every cached K/V byte a step must read once (shared
prefix pages once), q read, out written, new tokens and copied pages read and
written.  ``e2e`` is the same metric through the C-ABI calls with the step's
inputs copied from pinned host memory and the outputs copied back inside the
timed region.  ``roofline`` covers the step's dominant kernel, timed with CUDA
events on its launch stream.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the pages publish no runnable implementation to compare with).
Multi-GPU (torchrun): independent replicas, one per rank, no collective on the
data path; max time over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Callable, Dict, List, Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

CSRC = os.path.join(ROOT, "paged_kv_cache_262_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
METRIC = "paged decode attention: KV HBM GB/s (% of GB300 peak), decode tokens/s"
L2_BYTES = 129e6
WORKLOADS = ["llama8b_decode", "long_context_decode", "tiny_decode", "prefix_sharing", "parallel_sampling",
             "mixed_step", "swap", "block_manager"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_decode", choices=WORKLOADS)
    ap.add_argument("--chunks", type=int, default=16, help="mixed_step: prefill chunks")
    ap.add_argument("--decodes", type=int, default=240, help="mixed_step: decode sequences")
    ap.add_argument("--block-size", type=int, default=32, choices=[16, 32], help="mixed_step: tokens per page")
    ap.add_argument("--mixed-launch", default="fused", choices=["separate", "fused"],
                    help="mixed_step: one mixed-step launch whose CTAs run the prefill and the decode side by "
                         "side (default), or the two as separate launches")
    ap.add_argument("--overlap", default="none", choices=["none", "decode", "decode-hi", "prefill-hi"],
                    help="mixed_step: run prefill and decode on two streams (forked and joined in the step); "
                         "which one goes to the side stream and whether that stream has high priority")
    ap.add_argument("--sharing", default="auto", choices=["auto", "one-level", "subgroups"],
                    help="prefix_sharing / parallel_sampling: groups only (one level), or each prompt's samples "
                         "as sub-groups too (auto: sub-groups; each prompt's blocks are read once for its "
                         "samples)")
    ap.add_argument("--separate-append", action="store_true",
                    help="decode workloads: reshape_and_cache and decode as two launches instead of one "
                         "decode-with-append launch")
    ap.add_argument("--layers", type=int, default=0, help="layer pools to rotate (0 = auto, > 4x L2)")
    ap.add_argument("--plain-decode", action="store_true",
                    help="prefix_sharing: plain decode instead of the shared-prefix path")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every timed step from the host (default: replay the K steps from a CUDA graph)")
    ap.add_argument("--no-long-context", action="store_true",
                    help="llama8b_decode: leave out the long-context (8 x 32768) sub-record measured after it")
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the HBM read/copy probe (its launches would crowd a profiler's launch list)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline sample budget")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            return {"hbm": float(j["hbm_gbs"]), "bf16": float(j["bf16_tflops"]),
                    "bf16_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    "source": "measured"}
        except Exception:
            pass
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch of `kernel` on `workload` from the
    committed ncu capture, or None when the kernel's source changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    j = json.load(open(TRAFFIC_FILE)).get(f"{kernel}@{workload}")
    if not j:
        return None
    srcs = j["source"] if isinstance(j["source"], list) else [j["source"]]
    h = hashlib.sha256()
    for f in srcs:  # the kernel's sources, hashed in the listed order
        path = os.path.join(CSRC, f)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return j.get("bytes_per_launch") if h.hexdigest() == j["sha256"] else None


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.limit")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [(t, [x.strip() for x in line.split(",")]) for t, line in self.samples]
        rows = [(t, f) for t, f in rows if len(f) >= 9]
        win = [f for t, f in rows if t0 - 0.05 <= t <= t1 + 0.05]
        label = "timed"
        if not win:
            win = [f for t, f in rows if t <= t1 + 0.05][-10:]
            label = "nearest"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(f[1]) for f in win if num(f[1]) is not None]
        reasons = set()
        for f in win:
            for n, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"], f[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        pw = [num(f[3]) for f in win if num(f[3]) is not None]
        lim = [num(f[9]) for f in win if len(f) > 9 and num(f[9]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(win[0][2]),
                "reasons": sorted(reasons), "samples": len(win), "window": label,
                "power_w": statistics.median(pw) if pw else None,
                "power_limit_w": statistics.median(lim) if lim else None}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (ranks run independent replicas; the job
    takes as long as its slowest rank)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


# ------------------------------------------------------------------ workloads
@dataclasses.dataclass
class Bench:
    """One workload's step: what it reads per step, what it launches, what it counts."""
    name: str
    describe: str
    host_inputs: Dict[str, np.ndarray]        # per-step inputs (copied H2D in e2e)
    step: Callable                            # step(i, inputs: dict of device tensors, ev) -> outputs list
    step_bytes: int                           # algorithmic HBM bytes per step
    launches: int                             # our kernels per step
    kernel: str                               # dominant kernel
    bound: str                                # "hbm" or "tensor"
    kernel_work: float                        # bytes (hbm) or flops (tensor) per dominant launch
    seqs: int
    extra: Dict = dataclasses.field(default_factory=dict)
    layers: int = 1
    pool_mb: float = 0.0
    # launches of each timed kernel alone: name -> fn(i, inputs) (the interval
    # between consecutive events of step); [0] is the dominant kernel
    kernels: Dict[str, Callable] = dataclasses.field(default_factory=dict)


def decode_bytes(ctx, Hq, Hkv, D, B):
    ctx = np.asarray(ctx, dtype=np.int64)
    return int(ctx.sum()) * Hkv * D * 2 * 2 + 2 * len(ctx) * Hq * D * 2 + int(((ctx + B - 1) // B).sum()) * 4 \
        + len(ctx) * 4


def cache_bytes(T, Hkv, D):
    return T * Hkv * D * 2 * 2 * 2 + T * 8


def n_layers(args, pool_bytes):
    n = args.layers or max(2, int(math.ceil(5 * L2_BYTES / max(pool_bytes, 1))))
    return min(n, 64)


def decode_describe(case, fused):
    T = len(case.slot_mapping)
    what = (f"decode with append of {T} tokens (one launch)" if fused
            else f"reshape_and_cache of {T} tokens + decode")
    return (f"{case.name}: {case.num_seqs} seqs, ctx {int(case.context_lens.min())}.."
            f"{int(case.context_lens.max())} (mean {case.context_lens.mean():.0f}), {case.num_q_heads}q/"
            f"{case.num_kv_heads}kv heads, D={case.head_dim}, B={case.block_size}, {what}")


def build_decode(args, torch, pa, dev, case):
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    NL = n_layers(args, case.k_pool.nbytes * 2)
    kp0, vp0 = up(case.k_pool), up(case.v_pool)
    kps = [kp0] + [kp0.clone() for _ in range(NL - 1)]
    vps = [vp0] + [vp0.clone() for _ in range(NL - 1)]
    desc = pa.make_desc(up(case.q), kp0, torch.from_numpy(case.block_tables), scale=case.scale,
                        max_context_len=case.max_context_len)
    ws = pa.decode_workspace(desc, dev)
    outs = {"out": torch.empty((case.num_seqs, case.num_q_heads, case.head_dim), dtype=torch.bfloat16, device=dev)}

    fused = not args.separate_append  # each sequence's new token written by the decode launch itself

    def decode(i, x, out=None):
        l = i % NL
        out = out if out is not None else outs["out"]
        if fused:
            pa.paged_attention_decode_append(x["q"], x["new_k"], x["new_v"], x["slots"], kps[l], vps[l], x["bt"],
                                             x["ctx"], out, scale=case.scale, max_context_len=case.max_context_len,
                                             workspace=ws)
        else:
            pa.paged_attention_decode(x["q"], kps[l], vps[l], x["bt"], x["ctx"], out, scale=case.scale,
                                      max_context_len=case.max_context_len, workspace=ws)

    def step(i, x, ev, o=None):  # on the current stream
        l = i % NL
        out = o[0] if o else outs["out"]
        if not fused:
            pa.reshape_and_cache(x["new_k"], x["new_v"], kps[l], vps[l], x["slots"])
        ev and ev[0].record()
        decode(i, x, out)
        ev and ev[1].record()
        return [out]

    dec = decode_bytes(case.context_lens, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size)
    T = len(case.slot_mapping)
    cache = cache_bytes(T, case.num_kv_heads, case.head_dim)
    return Bench(case.name, decode_describe(case, fused),
                 {"q": case.q, "new_k": case.new_k, "new_v": case.new_v, "slots": case.slot_mapping,
                  "bt": case.block_tables, "ctx": case.context_lens},
                 step, dec + cache, 1 if fused else 2, "decode_kernel", "hbm", dec + (cache if fused else 0),
                 case.num_seqs, layers=NL, pool_mb=case.k_pool.nbytes * 2 / 1e6, kernels={"decode_kernel": decode})


def prefix_sharing_setup(pa, plan=None):
    """Tables, copy-on-write pairs and slots of the prefix-sharing workload (or
    another plan of the same shape), produced by the host block manager (fork
    per prompt and per sample, then one appended token per sample)."""
    plan = plan or wl.prefix_sharing_plan()
    B, R = plan.B, plan.samples_per_prompt
    bm = pa.BlockManager(plan.num_blocks, B)
    root = 10 ** 6
    bm.add_seq(root, plan.prefix_len)
    for p in range(plan.num_prompts):
        bm.fork(root, p * R)
        for _ in range(int(plan.suffix_lens[p])):
            bm.append(p * R)
        for i in range(1, R):
            bm.fork(p * R, p * R + i)
    bm.free_seq(root)
    S = plan.num_prompts * R
    slots, pairs = [], []
    for s in range(S):
        slot, pair = bm.append(s)
        slots.append(slot)
        if pair is not None:
            pairs.append(pair)
    ctx = np.array([bm.seq_len(s) for s in range(S)], np.int32)
    tables = [bm.block_table(s) for s in range(S)]
    bt = np.full((S, max(len(t) for t in tables)), -1, np.int32)
    for s, t in enumerate(tables):
        bt[s, : len(t)] = t
    return plan, bt, ctx, np.array(slots, np.int64), np.array(pairs, np.int64).reshape(-1, 2)


def prefix_sharing_subgroups(plan, bt, ctx):
    """The second sharing level of the prefix-sharing workload: the samples of
    one prompt (consecutive sequences) as a sub-group sharing their common
    leading blocks (the prompt prefix and the prompt's full suffix blocks;
    the partial block each sample copied on write is its own)."""
    B, R = plan.B, plan.samples_per_prompt
    S = len(ctx)
    starts, shared = [0], []
    for a in range(0, S, R):
        rows = bt[a: a + R]
        n = 0
        while n < rows.shape[1] and rows[0, n] >= 0 and np.all(rows[:, n] == rows[0, n]):
            n += 1
        shared.append(min(n, int(ctx[a: a + R].min()) // B) * B)
        starts.append(min(a + R, S))
    return np.array(starts, np.int32), np.array(shared, np.int32)


def prefix_modes(args, plan):
    """(shared-prefix path?, sub-groups as a second level?) for a sharing plan."""
    name = "prefix_sharing" if plan.prefix_len > 0 else "parallel_sampling"
    shared = not args.plain_decode
    sharing = args.sharing if args.sharing != "auto" else "subgroups"
    return shared, shared and sharing == "subgroups"


def prefix_describe(args, plan, n_pairs):
    name = "prefix_sharing" if plan.prefix_len > 0 else "parallel_sampling"
    shared, two = prefix_modes(args, plan)
    S = plan.num_prompts * plan.samples_per_prompt
    if plan.prefix_len > 0:
        mode = ("shared-prefix decode, two levels (prefix attended once on the tensor cores; each prompt's "
                "suffix blocks once for its samples, each sample's own block for it alone)" if two else
                "shared-prefix decode (prefix attended once on the tensor cores + per-sequence suffix)" if shared
                else "plain decode")
    else:
        mode = ("sub-group decode (each prompt's blocks read once for its samples, each sample's own block "
                "for it alone)" if two else
                "shared-prefix decode, each prompt a group (prompt attended once on the tensor cores)" if shared
                else "plain decode")
    shape = (f"{plan.prefix_len}-token shared prefix (ref_count {S}), suffix U[1,512]" if plan.prefix_len > 0
             else f"prompts of {int(plan.suffix_lens.min())}..{int(plan.suffix_lens.max())} tokens, no common prefix")
    return (f"{name}: {plan.num_prompts} prompts x {plan.samples_per_prompt} samples, "
            f"{shape}, {plan.Hq}q/{plan.Hkv}kv, D={plan.D}, B={plan.B}; "
            f"copy_blocks of {n_pairs} CoW pairs + reshape_and_cache of {S} tokens + {mode}")


def build_prefix(args, torch, pa, dev, plan=None):
    plan, bt, ctx, slots, pairs = prefix_sharing_setup(pa, plan)
    name = "prefix_sharing" if plan.prefix_len > 0 else "parallel_sampling"
    kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    NL = n_layers(args, kp.nbytes * 2)
    kp0, vp0 = up(kp), up(vp)
    kps = [kp0] + [kp0.clone() for _ in range(NL - 1)]
    vps = [vp0] + [vp0.clone() for _ in range(NL - 1)]
    S, Hq, Hkv, D, B = len(ctx), plan.Hq, plan.Hkv, plan.D, plan.B
    desc = pa.make_desc(up(q), kp0, torch.from_numpy(bt), max_context_len=int(ctx.max()))
    ws = pa.decode_workspace(desc, dev)
    outs = {"out": torch.empty((S, Hq, D), dtype=torch.bfloat16, device=dev)}

    shared, two = prefix_modes(args, plan)
    ss, sh = prefix_sharing_subgroups(plan, bt, ctx)
    if plan.prefix_len > 0:  # one group: the prefix every prompt starts with
        npre = plan.prefix_len // B
        groups = {"gs": np.array([0, S], np.int32), "gp": np.array([plan.prefix_len], np.int32),
                  "pt": np.ascontiguousarray(bt[:1, :npre])}
        gmax, gplen = S, plan.prefix_len
    elif two:  # no group: the sub-groups alone
        groups = {"gs": np.zeros(1, np.int32), "gp": np.zeros(0, np.int32), "pt": np.zeros((1, 1), np.int32)}
        gmax, gplen = 0, 0
    else:  # one level: each prompt's samples a group
        groups = {"gs": ss, "gp": sh, "pt": np.ascontiguousarray(bt[ss[:-1], : int(sh.max()) // B])}
        gmax, gplen = plan.samples_per_prompt, int(sh.max())
    if two:
        groups.update({"ss": ss, "sh": sh})
    sp_ws = torch.empty(pa._binding.load().pa_shared_prefix_workspace_bytes(pa._binding._c.byref(desc)),
                        dtype=torch.uint8, device=dev)

    def attend(i, x, out=None):
        l = i % NL
        out = out if out is not None else outs["out"]
        if shared:
            sub = dict(subgroup_starts=x["ss"], subgroup_shared_lens=x["sh"],
                       max_subgroup_size=plan.samples_per_prompt) if two else {}
            pa.paged_attention_decode_shared_prefix(
                x["q"], kps[l], vps[l], x["bt"], x["ctx"], x["gs"], x["gp"], x["pt"], out, max_group_size=gmax,
                max_prefix_len=gplen, max_context_len=int(ctx.max()), workspace=sp_ws, **sub)
        else:
            pa.paged_attention_decode(x["q"], kps[l], vps[l], x["bt"], x["ctx"], out,
                                      max_context_len=int(ctx.max()), workspace=ws)

    def step(i, x, ev, o=None):  # on the current stream
        l = i % NL
        out = o[0] if o else outs["out"]
        pa.copy_blocks([kps[l]], [vps[l]], x["pairs"])
        pa.reshape_and_cache(x["new_k"], x["new_v"], kps[l], vps[l], x["slots"])
        ev and ev[0].record()
        attend(i, x, out)
        ev and ev[1].record()
        return [out]

    unique_pages = np.unique(bt[bt >= 0])
    # unique KV bytes: every distinct page's tokens in use, once (pages are full except last ones)
    uniq_tokens = 0
    seen = set()
    for s in range(S):
        n = int(ctx[s])
        for k, pg in enumerate(bt[s]):
            if pg < 0 or pg in seen:
                continue
            seen.add(int(pg))
            uniq_tokens += min(B, n - k * B)
    kv_unique = uniq_tokens * Hkv * D * 2 * 2
    dec_unique = kv_unique + 2 * S * Hq * D * 2 + int(((ctx.astype(np.int64) + B - 1) // B).sum()) * 4 + S * 4
    dec_logical = decode_bytes(ctx, Hq, Hkv, D, B)
    copy = len(pairs) * Hkv * B * D * 2 * 2 * 2
    inputs = {"q": q, "new_k": nk, "new_v": nv, "slots": slots, "pairs": pairs, "bt": bt, "ctx": ctx}
    if shared:
        inputs.update(groups)
    return Bench(name, prefix_describe(args, plan, len(pairs)),
                 inputs, step, dec_unique + copy + cache_bytes(S, Hkv, D),
                 3 + (1 if shared and len(groups["gp"]) else 0),  # copy, reshape, [prefix pass,] decode
                 "shared_prefix_decode" if shared else "decode_kernel", "hbm", dec_unique, S,
                 extra={"unique_pages": int(len(unique_pages)), "logical_decode_bytes": dec_logical,
                        "unique_decode_bytes": dec_unique, "cow_pairs": int(len(pairs))},
                 layers=NL, pool_mb=kp.nbytes * 2 / 1e6,
                 kernels={"shared_prefix_decode" if shared else "decode_kernel": attend})


def mixed_describe(cctx, dctx, B, n_new, fused):
    what = "one mixed-step launch (prefill and decode side by side)" if fused else "prefill + decode"
    return (f"mixed_step: {len(cctx)} prefill chunks x 512 tokens (ctx {int(min(cctx))}..{int(max(cctx))})"
            f" + {len(dctx)} decodes (ctx {int(min(dctx))}..{int(max(dctx))}), 32q/8kv, D=128, B={B}; "
            f"reshape_and_cache of {n_new} tokens + {what}")


def build_mixed(args, torch, pa, dev):
    st = wl.Stream(0, 6)
    cctx = st.integers(512, 8192, 16)[: args.chunks]
    dctx = st.integers(64, 4096, 240)[: args.decodes]
    B = args.block_size
    m = wl.make_mixed_step("mixed_step", [512] * len(cctx), cctx, dctx, 32, 8, 128, B, seed=0, stream=105)
    dec = m.decode
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    NL = n_layers(args, dec.k_pool.nbytes * 2)
    kp0, vp0 = up(dec.k_pool), up(dec.v_pool)
    kps = [kp0] + [kp0.clone() for _ in range(NL - 1)]
    vps = [vp0] + [vp0.clone() for _ in range(NL - 1)]
    desc = pa.make_desc(up(dec.q), kp0, torch.from_numpy(dec.block_tables), max_context_len=dec.max_context_len)
    ws = pa.decode_workspace(desc, dev)
    T = int(m.cu_q[-1])
    outs = {"pout": torch.empty((T, 32, 128), dtype=torch.bfloat16, device=dev),
            "dout": torch.empty((dec.num_seqs, 32, 128), dtype=torch.bfloat16, device=dev)}
    max_cctx = int(m.chunk_ctx.max())

    def prefill(i, x, pout=None):
        l = i % NL
        pa.paged_attention_prefill_chunk(x["q_chunk"], x["cu_q"], kps[l], vps[l], x["chunk_bt"], x["chunk_ctx"],
                                         pout if pout is not None else outs["pout"], max_q_len=512,
                                         max_context_len=max_cctx)

    def decode(i, x, dout=None):
        l = i % NL
        pa.paged_attention_decode(x["q"], kps[l], vps[l], x["bt"], x["ctx"], dout if dout is not None else outs["dout"],
                                  max_context_len=dec.max_context_len, workspace=ws)

    fused = args.mixed_launch == "fused"

    def mixed(i, x, pout=None, dout=None):
        l = i % NL
        pa.paged_attention_mixed(x["q_chunk"], x["cu_q"], x["chunk_bt"], x["chunk_ctx"], x["q"], x["bt"], x["ctx"],
                                 kps[l], vps[l], pout if pout is not None else outs["pout"],
                                 dout if dout is not None else outs["dout"], max_q_len=512,
                                 prefill_max_context_len=max_cctx, decode_max_context_len=dec.max_context_len,
                                 workspace=ws)

    side = None
    if args.overlap != "none":
        side = torch.cuda.Stream(device=dev, priority=-1 if args.overlap.endswith("-hi") else 0)
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        side_fn = prefill if args.overlap == "prefill-hi" else decode
        main_fn = decode if args.overlap == "prefill-hi" else prefill

    def step(i, x, ev, o=None):  # on the current stream
        l = i % NL
        pout, dout = o if o else (outs["pout"], outs["dout"])
        pa.reshape_and_cache(x["new_k"], x["new_v"], kps[l], vps[l], x["slots"])
        ev and ev[0].record()
        if fused:
            mixed(i, x, pout, dout)
            ev and ev[1].record()
            return [pout, dout]
        if side is not None:  # the two attention launches side by side, joined before the step ends
            cur = torch.cuda.current_stream()
            fork.record(cur)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                side_fn(i, x, pout if side_fn is prefill else dout)
            main_fn(i, x, pout if main_fn is prefill else dout)
            join.record(side)
            cur.wait_event(join)
            ev and ev[1].record()
        else:
            prefill(i, x, pout)
            ev and ev[1].record()
            decode(i, x, dout)
        ev and ev[2].record()
        return [pout, dout]

    flops = 0
    for r in range(len(cctx)):
        c = int(cctx[r])
        pos = np.arange(c - 512, c, dtype=np.int64)
        flops += 4 * 128 * 32 * int((pos + 1).sum())
    pre_bytes = int(np.asarray(cctx, np.int64).sum()) * 8 * 128 * 4 + 2 * T * 32 * 128 * 2
    dbytes = decode_bytes(dec.context_lens, 32, 8, 128, B)
    Tn = T + dec.num_seqs
    new_k = np.concatenate([m.chunk_new_k, dec.new_k])
    new_v = np.concatenate([m.chunk_new_v, dec.new_v])
    slots = np.concatenate([m.chunk_slots, dec.slot_mapping])
    return Bench("mixed_step", mixed_describe(cctx, dctx, B, Tn, fused),
                 {"q_chunk": m.q_chunk, "cu_q": m.cu_q, "chunk_bt": m.chunk_tables, "chunk_ctx": m.chunk_ctx,
                  "q": dec.q, "bt": dec.block_tables, "ctx": dec.context_lens, "new_k": new_k, "new_v": new_v,
                  "slots": slots},
                 step, pre_bytes + dbytes + cache_bytes(Tn, 8, 128), 2 if fused else 3,
                 "mixed_kernel" if fused else "prefill_kernel", "hbm" if fused else "tensor",
                 pre_bytes + dbytes if fused else flops,
                 dec.num_seqs, extra={"prefill_flops": flops, "decode_bytes": dbytes, "prefill_kv_bytes": pre_bytes},
                 layers=NL, pool_mb=dec.k_pool.nbytes * 2 / 1e6,
                 kernels=({"mixed_kernel": mixed} if fused else {}) | {"prefill_kernel": prefill, "decode_kernel": decode})


def build_swap(args, torch, pa, dev):
    B, Hkv, D, L = 16, 8, 128, 4
    nseq, ntok = 16, 2048
    per = ntok // B
    ndev, nhost = int(1.25 * nseq * per), nseq * per
    bm = pa.BlockManager(ndev, B, num_host_blocks=nhost)
    for s in range(nseq):
        bm.add_seq(s, 0)
    for _ in range(ntok):  # round-robin appends: every sequence's blocks scattered over the pool
        for s in range(nseq):
            bm.append(s)
    out_pairs = np.array([p for s in range(nseq) for p in bm.swap_out(s)], np.int64)
    in_pairs = np.array([p for s in range(nseq) for p in bm.swap_in(s)], np.int64)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    dk = [torch.randn((ndev, Hkv, B, D), generator=gen, device=dev).to(torch.bfloat16) for _ in range(L)]
    dv = [torch.randn((ndev, Hkv, B, D), generator=gen, device=dev).to(torch.bfloat16) for _ in range(L)]
    hk = [torch.empty((nhost, Hkv, B, D), dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    hv = [torch.empty_like(h).pin_memory() for h in hk]
    blk = Hkv * B * D * 2
    moved = 2 * len(out_pairs) * L * blk  # K and V of every block and layer, one way

    def swap(i, x):
        pa.swap_blocks(dk, dv, hk, hv, x["out_pairs"])  # preempt: device -> host
        pa.swap_blocks(hk, hv, dk, dv, x["in_pairs"])   # resume: host -> new device blocks

    def step(i, x, ev, o=None):
        ev and ev[0].record()
        swap(i, x)
        ev and ev[1].record()
        return []

    # the link's reference: one contiguous copy-engine copy of the same bytes each way
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for r in range(4):
        if r == 1:
            e0.record()
        hbuf.copy_(dbuf, non_blocking=True)
        dbuf.copy_(hbuf, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    link_gbs = 3 * 2 * moved / (e0.elapsed_time(e1) / 1e3) / 1e9
    return Bench("swap", f"swap: {nseq} sequences x {ntok} tokens, {Hkv} kv heads, D={D}, B={B}, {L} layers "
                 f"({len(out_pairs)} scattered blocks) to pinned host memory and back to new device blocks",
                 {"out_pairs": out_pairs, "in_pairs": in_pairs}, step, 2 * moved, 2, "swap_blocks", "link",
                 2 * moved, nseq, extra={"link_gbs": round(link_gbs, 1), "blocks": int(len(out_pairs)),
                                         "bytes_each_way": moved},
                 layers=L, pool_mb=2 * L * ndev * blk / 1e6, kernels={"swap_blocks": swap})


def build(args, torch, pa, dev):
    if args.workload == "prefix_sharing":
        return build_prefix(args, torch, pa, dev)
    if args.workload == "parallel_sampling":
        return build_prefix(args, torch, pa, dev, wl.parallel_sampling_plan())
    if args.workload == "swap":
        return build_swap(args, torch, pa, dev)
    if args.workload == "mixed_step":
        return build_mixed(args, torch, pa, dev)
    case = {"llama8b_decode": wl.llama8b_decode, "long_context_decode": wl.long_context_decode,
            "tiny_decode": wl.tiny_decode}[args.workload]()
    return build_decode(args, torch, pa, dev, case)


# ------------------------------------------------------------------ our arm
def hbm_probe(torch, pa, dev):
    """This GPU's HBM stream rates from the library's own probe kernels
    (pa_hbm_probe): read-only streams over 2 GiB through 16-byte vector loads
    and through TMA bulk copies into shared memory, and a 16-byte vector copy
    of 1 GiB (read + write bytes); best of 10 launches each, CUDA events on
    the launch stream; and the same bytes read as paged decode reads them
    (4 KB runs at scattered places, the decode kernel's concurrency).  Decode
    is a read stream of page gathers, so it is also reported against the
    faster read rate and against the gather rate."""
    src = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    src.random_(0, 256)  # nonzero data, so the probe's never-taken store stays never taken
    sink = torch.zeros(16, dtype=torch.uint8, device=dev)
    half = src[: 1 << 30]
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def best(fn, nbytes):
        for _ in range(3):
            fn()
        out = 0.0
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            out = max(out, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
        return out

    err = torch.zeros(1, dtype=torch.int32, device=dev)
    read = best(lambda: pa.hbm_probe(src, sink=sink), src.numel())
    tma = best(lambda: pa.hbm_probe(src, tma=True, err_flag=err), src.numel())
    runs = 1 << (int(src.numel() // 2 // 4096).bit_length() - 1)  # 4 KB runs read in each half
    gather = best(lambda: pa.hbm_probe(src, gather=True, err_flag=err), 2 * 4096 * runs)
    copy = best(lambda: pa.hbm_probe(half, dst=dst), 2 * half.numel())
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"HBM probe: device error flag {int(err.item())}")
    del src, dst, half, sink
    torch.cuda.empty_cache()
    return {"read_gbs": round(max(read, tma), 1), "read_lsu_gbs": round(read, 1), "read_tma_gbs": round(tma, 1),
            "gather_gbs": round(gather, 1), "copy_gbs": round(copy, 1)}


def tensor_probe(torch, dev, sampler):
    """This GPU's dense bf16 tensor rate from cuBLAS (torch.matmul, 8192^3,
    fp32 accumulate): best of 10 single GEMMs (burst), and GEMMs back to back
    for about 1.5 s under the board's power limit (sustained), with the clocks
    and power sampled over the sustained loop."""
    n = 8192
    a = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
    b = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
    c = torch.empty((n, n), device=dev, dtype=torch.bfloat16)
    flop = 2.0 * n * n * n
    stream = torch.cuda.current_stream()
    for _ in range(5):
        torch.matmul(a, b, out=c)
    torch.cuda.synchronize()
    burst = 0.0
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        torch.matmul(a, b, out=c)
        e1.record(stream)
        torch.cuda.synchronize()
        burst = max(burst, flop / (e0.elapsed_time(e1) / 1e3) / 1e12)
    reps = max(1, int(1.5 / (flop / (burst * 1e12))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(reps):
        torch.matmul(a, b, out=c)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sustained = flop * reps / (e0.elapsed_time(e1) / 1e3) / 1e12
    clk = sampler.summary(t0 + (t1 - t0) / 3, t1) if sampler else None
    del a, b, c
    torch.cuda.empty_cache()
    return {"burst_tflops": round(burst, 1), "sustained_tflops": round(sustained, 1), "gemm": f"bf16 {n}^3, cuBLAS",
            "sustained_reps": reps, "clocks": clk}


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_262_gb300 as pa
    from paged_kv_cache_262_gb300 import build as pbuild

    pbuild.build()
    pa.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    probe = None if args.no_probe else hbm_probe(torch, pa, dev)
    if probe is not None and args.workload == "mixed_step":  # the tensor side's own ceiling, this run
        probe["tensor"] = tensor_probe(torch, dev, sampler)
    b = build(args, torch, pa, dev)
    res = measure(args, b, torch, dev, world, rank, sampler, probe)
    long_ctx = None
    if args.workload == "llama8b_decode" and not args.no_long_context:
        # the long-context decode target beside it, in the same process and clock record
        del b
        torch.cuda.empty_cache()
        long_ctx = measure(args, build_decode(args, torch, pa, dev, wl.long_context_decode()), torch, dev, world,
                           rank, sampler, probe)
    if sampler:
        sampler.stop()
    if rank != 0:
        return None
    if long_ctx is not None:
        res["long_context_decode"] = long_ctx
    if not args.no_cpu_baseline and args.workload != "swap":  # (no attention arithmetic to time there)
        res["cpu_baseline"] = cpu_baseline(args, args.cpu_seconds)
    return res


def measure(args, b, torch, dev, world, rank, sampler, probe):
    """Warm-up, the K timed steps, each timed kernel's launch duration, e2e;
    the JSON fields of one workload (rank 0; None elsewhere)."""
    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16)
        t = t.to(dev)
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    x = {k: to_dev(v) for k, v in b.host_inputs.items()}
    stream = torch.cuda.current_stream()
    nev = 3 if b.kernel == "prefill_kernel" else 2
    idle = None
    if sampler and b.kernel == "mixed_kernel":  # the power drawn with nothing running, for the power bound
        torch.cuda.synchronize()
        t_i0 = time.time()
        time.sleep(0.6)
        idle = sampler.summary(t_i0, time.time())

    for i in range(args.warmup):
        b.step(i, x, None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    side = {}
    per, per_clk = {}, {}  # per-kernel launch time and clocks (graph mode)
    if args.eager:
        # every launch from the host, an event pair around each timed kernel
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_wall0 = time.time()
        e0.record(stream)
        for i in range(args.steps):
            b.step(i, x, evs[i])
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        ms = e0.elapsed_time(e1)
        k_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]
        k_mean, k_median = statistics.mean(k_ms), statistics.median(k_ms)
        if nev == 3:
            d_ms = [ev[1].elapsed_time(ev[2]) for ev in evs]
            side["decode_launch_ms_mean"] = statistics.mean(d_ms)
        timing = "eager launches, CUDA events around each timed kernel"
    else:
        # the K steps replayed from one CUDA graph (the launches of a serving
        # loop); each timed kernel from a graph of its K launches alone
        cap = torch.cuda.Stream(device=dev)

        def capture(fn):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                for i in range(args.steps):
                    fn(i)
            stream.wait_stream(cap)
            return g

        g_step = capture(lambda i: b.step(i, x, None))
        g_kern = [(name, capture(lambda i, f=f: f(i, x))) for name, f in b.kernels.items()]
        g_step.replay()  # untimed: first replay of each graph
        for _, g in g_kern:
            g.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_wall0 = time.time()
        e0.record(stream)
        g_step.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        ms = e0.elapsed_time(e1)
        for name, g in g_kern:
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            kw0 = time.time()
            k0.record(stream)
            g.replay()
            k1.record(stream)
            torch.cuda.synchronize()
            per[name] = k0.elapsed_time(k1) / args.steps
            if sampler:  # (the first third of the window: the board's draw still settling)
                kw1 = time.time()
                per_clk[name] = sampler.summary(kw0 + (kw1 - kw0) / 3, kw1)
        k_mean, k_median = per[b.kernel], None  # one event pair around K launches: a mean, no median
        if "decode_kernel" in per and b.kernel != "decode_kernel":
            side["decode_launch_ms_mean"] = per["decode_kernel"]
        if "prefill_kernel" in per and b.kernel != "prefill_kernel":
            side["prefill_launch_ms_mean"] = per["prefill_kernel"]
            side["prefill_tflops"] = round(b.extra["prefill_flops"] / (per["prefill_kernel"] / 1e3) / 1e12, 1)
            if probe and probe.get("tensor"):  # the prefill alone against this run's sustained cuBLAS rate
                side["prefill_frac_of_probe_sustained"] = round(
                    side["prefill_tflops"] / probe["tensor"]["sustained_tflops"], 4)
        timing = (f"CUDA graph of the {args.steps} steps; per-kernel launch time from a graph of the kernel's "
                  f"{args.steps} launches alone (a mean)")
    if "decode_launch_ms_mean" in side:
        side["decode_gbs"] = round(b.extra["decode_bytes"] / (side["decode_launch_ms_mean"] / 1e3) / 1e9, 1)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, b, torch, dev, stream, world)
    ms = max_over_ranks(ms, world, dev)
    if rank != 0:
        return None
    peaks = load_peaks()
    if b.bound == "hbm":
        achieved = b.kernel_work / (k_mean / 1e3) / 1e9
        peak, unit = peaks["hbm"], "GB/s"
        peak_note = f"{peaks['source']} hbm_gbs (copy, read+write bytes)"
    elif b.bound == "link":
        achieved = b.kernel_work / (k_mean / 1e3) / 1e9
        peak, unit = b.extra["link_gbs"], "GB/s"
        peak_note = ("chip-to-chip link: contiguous copy-engine copies (cudaMemcpyAsync, pinned host <-> device) "
                     "of the same bytes each way, measured in this run")
    else:
        achieved = b.kernel_work / (k_mean / 1e3) / 1e12
        peak, unit = peaks["bf16_sustained"], "TFLOP/s"
        peak_note = f"{peaks['source']} bf16_tflops_sustained (kernel timed inside a long step); burst {peaks['bf16']}"
    value = job_throughput(b.step_bytes, args.steps, world, ms)
    roof = {"bound": b.bound, "kernel": b.kernel, "achieved": round(achieved, 1), "peak": peak,
            "peak_source": peak_note, "unit": unit, "frac": round(achieved / peak, 4),
            "traffic": kernel_traffic(b.kernel, b.name), "algorithmic_per_launch": b.kernel_work,
            "launch_ms_mean": k_mean}
    if k_median is not None:
        roof["launch_ms_median"] = k_median
    if b.bound == "hbm" and probe:
        roof["read_peak"] = {"peak": probe["read_gbs"], "unit": "GB/s",
                             "frac": round(achieved / probe["read_gbs"], 4),
                             "source": "this run's pa_hbm_probe, the faster of two read-only streams over 2 GiB "
                                       "(16-byte vector loads; TMA bulk copies into shared memory), best of 10 "
                                       "(decode streams reads only)",
                             "read_lsu_gbs": probe["read_lsu_gbs"], "read_tma_gbs": probe["read_tma_gbs"],
                             "copy_probe_gbs": probe["copy_gbs"]}
        roof["gather_peak"] = {"peak": probe["gather_gbs"], "unit": "GB/s",
                               "frac": round(achieved / probe["gather_gbs"], 4),
                               "source": "this run's pa_hbm_probe mode 3: 4 KB K/V runs at scattered places with "
                                         "the decode kernel's concurrency and no arithmetic (what paged reads can "
                                         "reach), best of 10"}
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": b.describe, "seqs": b.seqs, "layer_pools": b.layers,
                   "l2": f"inputs larger than L2: {b.layers} layer pools of {b.pool_mb:.0f} MB rotated",
                   "parallelism": f"replicas{world}"},
        "decode_tokens_per_s": round(b.seqs * args.steps * world / (ms / 1e3), 1),
        "gpu_launches": b.launches * args.steps,
        "roofline": roof,
        "clocks": clocks,
        "timing": timing,
    }
    tp = (probe or {}).get("tensor")
    if tp and b.bound == "tensor":  # the prefill against this run's cuBLAS rate too
        res["roofline"]["tensor_probe"] = dict(tp, frac_sustained=round(achieved / tp["sustained_tflops"], 4),
                                               frac_burst=round(achieved / tp["burst_tflops"], 4))
    if b.kernel == "mixed_kernel":  # one launch doing both: the prefill's tensor work in the same time
        tf = b.extra["prefill_flops"] / (k_mean / 1e3) / 1e12
        res["roofline"]["tensor"] = {"achieved": round(tf, 1), "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                                     "frac": round(tf / peaks["bf16_sustained"], 4)}
        if tp:
            res["roofline"]["tensor"]["probe"] = dict(tp, frac_sustained=round(tf / tp["sustained_tflops"], 4))
        lower = max(b.extra["prefill_flops"] / (peaks["bf16_sustained"] * 1e12),
                    b.kernel_work / (peaks["hbm"] * 1e9)) * 1e3
        res["roofline"]["lower_bound_ms"] = round(lower, 4)
        # The step under the board power limit: the energy the two halves draw
        # above idle when each runs alone back to back, spent at the limit's
        # headroom above idle.  An estimate, not a bound: energy per unit of
        # work falls somewhat with the clock a capped GPU settles at.
        clk_p, clk_d = per_clk.get("prefill_kernel"), per_clk.get("decode_kernel")
        if idle and clk_p and clk_d and all(c.get("power_w") for c in (idle, clk_p, clk_d)) \
                and clk_p.get("power_limit_w"):
            p0, lim = idle["power_w"], clk_p["power_limit_w"]
            e_dyn = (clk_p["power_w"] - p0) * per["prefill_kernel"] + (clk_d["power_w"] - p0) * per["decode_kernel"]
            t_pow = e_dyn / (lim - p0)
            res["roofline"]["power_estimate"] = {
                "ms": round(t_pow, 4), "frac": round(t_pow / k_mean, 4), "idle_w": p0, "limit_w": lim,
                "prefill_alone": {"ms": round(per["prefill_kernel"], 4), "power_w": clk_p["power_w"],
                                  "sm_mhz": clk_p["sm_mhz"], "reasons": clk_p["reasons"]},
                "decode_alone": {"ms": round(per["decode_kernel"], 4), "power_w": clk_d["power_w"],
                                 "sm_mhz": clk_d["sm_mhz"], "reasons": clk_d["reasons"]},
                "mixed": per_clk.get("mixed_kernel")}
    res.update(side)
    if b.extra:
        res["workload_extra"] = b.extra
    if e2e:
        res["e2e"] = e2e
    return res


def run_e2e(args, b, torch, dev, stream, world):
    """The same steps through the C ABI with host buffers: each step's inputs
    are packed in one pinned staging buffer and copied host->device, and its
    outputs copied device->host, inside the timed region.  Two staging slots,
    an upload stream and a download stream let step i+1's inputs and step
    i-1's outputs move while step i's kernels run, as a serving loop would."""
    names = list(b.host_inputs)
    arrs = [np.ascontiguousarray(b.host_inputs[k]) for k in names]
    offs, pos = [], 0
    for a in arrs:
        offs.append(pos)
        pos += (a.nbytes + 255) // 256 * 256
    staged = np.zeros(pos, np.uint8)
    for a, o in zip(arrs, offs):
        staged[o: o + a.nbytes] = a.view(np.uint8).reshape(-1)
    h_stage = torch.from_numpy(staged).pin_memory()
    d_stage = [torch.empty(pos, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        x = {}
        for k, a, o in zip(names, arrs, offs):
            dt = {np.uint16: torch.bfloat16, np.int32: torch.int32, np.int64: torch.int64}[a.dtype.type]
            x[k] = buf[o: o + a.nbytes].view(dt).view(a.shape)
        return x

    xs = [views(d) for d in d_stage]
    probe = b.step(0, xs[0], None)
    d_out = [[torch.empty_like(t) for t in probe] for _ in range(2)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in probe] for _ in range(2)]
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        k = i & 1
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(comp_done[k])     # slot k's inputs no longer in use (step i-2)
            d_stage[k].copy_(h_stage, non_blocking=True)
            h2d_done[k].record(up)
        cur = torch.cuda.current_stream()
        cur.wait_event(h2d_done[k])
        if i >= 2:
            cur.wait_event(d2h_done[k])         # slot k's outputs of step i-2 copied out
        b.step(i, xs[k], None, d_out[k])
        comp_done[k].record(cur)
        with torch.cuda.stream(down):
            down.wait_event(comp_done[k])
            for hd, dd in zip(h_out[k], d_out[k]):
                hd.copy_(dd, non_blocking=True)
            d2h_done[k].record(down)

    def run_steps(n):
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        up.wait_event(start)  # the transfer streams fork from (and, in a capture, join) this stream
        down.wait_event(start)
        for i in range(n):
            e2e_step(i)
        for k in range(min(n, 2)):
            cur.wait_event(d2h_done[k])         # every transfer joins the stream

    run_steps(max(args.warmup, 2))
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.eager:
        if world > 1:
            torch.distributed.barrier()
        f0.record(stream)
        run_steps(args.steps)
        f1.record(stream)
    else:  # the same calls captured once and replayed, as a serving loop would
        cap = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            run_steps(args.steps)
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        f0.record(stream)
        g.replay()
        f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    h2d = int(pos)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    return {"value": round(job_throughput(b.step_bytes, args.steps, world, e2e_ms), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms / args.steps,
            "transfers": "one pinned staging buffer H2D + outputs D2H per step, double-buffered on upload and download streams",
            "launch": "host launches" if args.eager else "the K steps' copies and kernels captured in one CUDA graph"}


# ------------------------------------------------------------------ oracle (CPU) arm
def oracle_units(args):
    """The workload as a list of oracle work units, each returning the
    algorithmic bytes it covered, with the kind of unit and the workload's
    description (the GPU arm's config.workload).  Units are whole (sequence,
    kv head) decode units or whole prefill rows (all heads of one query
    position)."""
    import oracle
    ora = oracle.default()
    units: List[Callable[[], int]] = []
    if args.workload == "mixed_step":
        st = wl.Stream(0, 6)
        cctx = st.integers(512, 8192, 16)[: args.chunks]
        dctx = st.integers(64, 4096, 240)[: args.decodes]
        m = wl.make_mixed_step("mixed_step", [512] * len(cctx), cctx, dctx, 32, 8, 128, args.block_size, seed=0,
                               stream=105)
        kp, vp = m.decode.k_pool.copy(), m.decode.v_pool.copy()
        ora.reshape_and_cache(m.chunk_new_k, m.chunk_new_v, kp, vp, m.chunk_slots)
        for r in range(len(cctx)):
            for i in range(512):
                def u(r=r, i=i):
                    for h in range(32):
                        ora.prefill_row(m.q_chunk, m.cu_q, kp, vp, m.chunk_tables, m.chunk_ctx, m.decode.scale, r, i, h)
                    return (int(cctx[r]) - 512 + i + 1) * 8 * 128 * 4
                units.append(u)
        return units, "prefill rows (all 32 heads of one query position)", mixed_describe(
            cctx, dctx, args.block_size, int(m.cu_q[-1]) + len(dctx), args.mixed_launch == "fused")
    if args.workload in ("prefix_sharing", "parallel_sampling"):
        import paged_kv_cache_262_gb300 as pa
        plan, bt, ctx, slots, pairs = prefix_sharing_setup(
            pa, wl.parallel_sampling_plan() if args.workload == "parallel_sampling" else None)
        kp, vp, q, nk, nv = wl.prefix_sharing_values(plan)
        if len(pairs):
            ora.copy_blocks([kp], [vp], pairs)
        ora.reshape_and_cache(nk, nv, kp, vp, slots)
        case = wl.DecodeCase("prefix_sharing", len(ctx), plan.Hq, plan.Hkv, plan.D, plan.B, plan.num_blocks,
                             bt.shape[1], 1 / math.sqrt(plan.D), ctx, bt, q, kp, vp)
        describe = prefix_describe(args, plan, len(pairs))
    else:
        case = {"llama8b_decode": wl.llama8b_decode, "long_context_decode": wl.long_context_decode,
                "tiny_decode": wl.tiny_decode}[args.workload]()
        describe = decode_describe(case, not args.separate_append)
        if case.new_k is not None:
            ora.reshape_and_cache(case.new_k, case.new_v, case.k_pool, case.v_pool, case.slot_mapping)
    G = case.num_q_heads // case.num_kv_heads
    for s in range(case.num_seqs):
        for g in range(case.num_kv_heads):
            def u(s=s, g=g):
                for h in range(g * G, (g + 1) * G):
                    ora.decode_head(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                                    case.scale, s, h)
                return int(case.context_lens[s]) * case.head_dim * 2 * 2 + 2 * G * case.head_dim * 2
            units.append(u)
    return units, "(sequence, kv head) decode units (all query heads of the group)", describe


def _run_parallel(ex, n, units, start, count):
    """Runs units[start .. start+count) (wrapping) on the n-thread pool `ex`,
    one block of units per thread; the oracle's C calls release the GIL.
    Returns (bytes, wall seconds)."""
    idx = [(start + i) % len(units) for i in range(count)]
    blocks = [idx[i::n] for i in range(n)]  # one task per thread
    t0 = time.perf_counter()
    nbytes = sum(ex.map(lambda blk: sum(units[k]() for k in blk), blocks))
    return nbytes, time.perf_counter() - t0


def host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_baseline(args, budget_s):
    """The fp64 oracle on the host: single thread for half the budget, then
    every host core (independent units in parallel) for the other half."""
    units, kind, _ = oracle_units(args)
    secs, nbytes, done = 0.0, 0, 0
    while done < len(units) and secs < budget_s / 2:
        t0 = time.perf_counter()
        nbytes += units[done]()
        secs += time.perf_counter() - t0
        done += 1
    single = {"value": round(nbytes / secs / 1e9, 6), "unit": "GB/s", "cores": 1,
              "sample": f"first {done} of {len(units)} {kind}, {secs:.1f} s"}
    n = host_threads()
    count = max(n, int(n * (budget_s / 2) / (secs / done)))
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        _run_parallel(ex, n, units, 0, n)  # start the threads
        pbytes, wall = _run_parallel(ex, n, units, done % len(units), count)
    return {"value": round(pbytes / wall / 1e9, 6), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"fp64 C oracle on {n} host threads: {count} {kind} of {args.workload} "
                      f"(from unit {done % len(units)}, wrapping), {wall:.1f} s wall",
            "single_thread": single}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step a bounded sample of the
    workload's units, run on every host core."""
    if rank != 0:
        return None
    from oracle import build as obuild
    obuild.build()
    units, kind, describe = oracle_units(args)
    n = host_threads()
    t0 = time.perf_counter()
    units[0]()
    t_unit = max(time.perf_counter() - t0, 1e-6)
    per_step = max(n, min(len(units), int(n * (120.0 / max(args.steps + args.warmup, 1)) / t_unit)))
    k = 1
    secs, nbytes = 0.0, 0
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        for _ in range(args.warmup):
            _run_parallel(ex, n, units, k, per_step)
            k += per_step
        for _ in range(args.steps):
            b, w = _run_parallel(ex, n, units, k, per_step)
            k += per_step
            nbytes += b
            secs += w
    value = nbytes / secs / 1e9
    sample = f"fp64 C oracle on {n} host threads: {per_step} {kind} of {args.workload} per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe, "parallelism": f"{n} host threads"},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": n, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_block_manager(args):
    """Host throughput of the block manager's operations (prefix caching,
    fork, copy-on-write append, swap, free) over the prefix-sharing plan."""
    import paged_kv_cache_262_gb300 as pa
    plan = wl.prefix_sharing_plan()
    st = wl.Stream(0, 8)
    system = np.asarray(st.integers(0, 32000, plan.prefix_len), np.int32)
    prompts = [np.concatenate([system, np.asarray(st.integers(0, 32000, int(n)), np.int32)])
               for n in plan.suffix_lens]
    R, B = plan.samples_per_prompt, plan.B
    nblk = 4 * plan.num_blocks
    times = {k: 0.0 for k in ("admit", "fork", "append", "steady", "swap", "free")}
    counts = {"tokens": 0, "cached_tokens": 0, "forks": 0, "appends": 0, "cow": 0, "swapped_blocks": 0, "frees": 0,
              "steps": 0, "turn_tokens": 0, "turn_cached": 0, "turn_generated": 0}
    message = np.asarray(st.integers(0, 32000, 32), np.int32)
    ids = np.arange(len(prompts) * R, dtype=np.int32)
    step_tokens = np.asarray(st.integers(0, 32000, len(ids)), np.int32)
    DECODE_STEPS = 8
    max_blocks = (max(len(p) for p in prompts) + DECODE_STEPS + B - 1) // B

    def one_pass():
        bm = pa.BlockManager(nblk, B, num_host_blocks=nblk)
        t0 = time.perf_counter()
        for p, toks in enumerate(prompts):
            counts["cached_tokens"] += bm.add_seq_tokens(p * R, toks)
            counts["tokens"] += len(toks)
        t1 = time.perf_counter()
        for p in range(len(prompts)):
            for i in range(1, R):
                bm.fork(p * R, p * R + i)
                counts["forks"] += 1
        def decode_step():
            # one decode step's host work: a token onto every sequence, then the
            # padded block-table matrix and context lengths the attention call takes
            _, cows = bm.append_batch(ids, step_tokens)  # with ids: filled blocks enter the prefix cache
            bm.block_tables(ids, max_blocks)
            return int((cows[:, 0] >= 0).sum())

        t2 = time.perf_counter()
        counts["cow"] += decode_step()  # the first step after the forks: copy-on-write of the shared blocks
        counts["appends"] += len(ids)
        t3 = time.perf_counter()
        for _ in range(DECODE_STEPS - 1):
            decode_step()
        times["steady"] += time.perf_counter() - t3
        counts["steps"] += DECODE_STEPS - 1
        base = len(prompts) * R  # swapping needs unshared blocks: 64 separate 1024-token sequences
        for j in range(64):
            bm.add_seq(base + j, 1024)
        t3s = time.perf_counter()  # the swap phase starts after that set-up
        for j in range(64):
            counts["swapped_blocks"] += len(bm.swap_out(base + j))
            bm.swap_in(base + j)
        t4 = time.perf_counter()
        for s_ in range(base + 64):
            bm.free_seq(s_)
            counts["frees"] += 1
        t5 = time.perf_counter()
        for k, a, b in (("admit", t0, t1), ("fork", t1, t2), ("append", t2, t3), ("swap", t3s, t4), ("free", t4, t5)):
            times[k] += b - a
        # the next turn of each prompt's first sample: its history (the prompt and the tokens
        # its decode steps appended, ids given) and a new message, after every sequence was freed
        for p, toks in enumerate(prompts):
            hist = np.concatenate([toks, np.full(DECODE_STEPS, step_tokens[p * R], np.int32), message])
            got = bm.add_seq_tokens(base + 64 + p, hist)
            counts["turn_tokens"] += len(hist)
            counts["turn_cached"] += got
            counts["turn_generated"] += max(0, got - len(toks) // B * B)  # in blocks the decode steps filled

    for _ in range(args.warmup):
        one_pass()
    for k in times:
        times[k] = 0.0
    for k in counts:
        counts[k] = 0
    w0 = time.perf_counter()
    for _ in range(args.steps):
        one_pass()
    wall = time.perf_counter() - w0
    rate = lambda n, t: round(n / t, 1) if t > 0 else None  # noqa: E731
    return {"metric": "host block manager: prompt tokens admitted per second (prefix-cache lookups)",
            "value": rate(counts["tokens"], times["admit"]), "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True,
            "scaling": "none", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": f"block_manager: {len(prompts)} prompts x {R} samples, {plan.prefix_len}-token "
                                   f"system prompt + U[1,512] tokens, B={B}; admit, fork, {DECODE_STEPS} decode steps (each one "
                                   f"append_batch with token ids + block_tables call over all {len(ids)} sequences); 64 unshared "
                                   f"1024-token sequences swapped out and in; free all; per step (host only, "
                                   f"through the C ABI from Python; prompts held as int32 arrays)"},
            "cached_fraction": round(counts["cached_tokens"] / max(counts["tokens"], 1), 4),
            "ops_per_s": {"fork": rate(counts["forks"], times["fork"]),
                          "append": rate(counts["appends"], times["append"]),
                          "copy_on_write_share": round(counts["cow"] / max(counts["appends"], 1), 4),
                          "swap_blocks_out_and_in": rate(counts["swapped_blocks"], times["swap"]),
                          "free": rate(counts["frees"], times["free"])},
            "next_turn": {"cached_fraction": round(counts["turn_cached"] / max(counts["turn_tokens"], 1), 4),
                          "tokens_found_in_blocks_decode_filled_per_prompt": round(counts["turn_generated"] / max(
                              args.steps * len(prompts), 1), 2)},
            "decode_step_host_us": {"first_after_fork": round(times["append"] / args.steps * 1e6, 2),
                                    "steady": round(times["steady"] / max(counts["steps"], 1) * 1e6, 2)},
            "gpu_launches": 0}


def main():
    args = parse()
    if args.workload == "block_manager":  # host only
        print(json.dumps(run_block_manager(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        res = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
