// Shared-prefix decode as a queue of small tasks, for sm_103a.
//
// "Configuring vLLM and PagedAttention for High Throughput Enterprise LLM
// Serving" ("Zero-Copy Prefix Caching & Shared Sampling") lets requests that
// share leading blocks point at the same physical pages, and decode is bound
// by reading the cache from HBM ("Memory Bottlenecks in Autoregressive LLM
// Inference").  After the tensor-core pass over a group's common prefix
// (pa_shared_prefix.cu), what is left per sequence is short: the blocks
// written since the prefix, shared by the samples of one prompt up to each
// sample's copy-on-write block ("vLLM Guide: High-Throughput Multi-GPU LLM
// Serving with PagedAttention", "What Is PagedAttention?").  Short pieces of
// work each paying a whole CTA's start-up (block-table read, first gather
// round trip) and end (merge, prefix fold, stores) leave HBM idle most of the
// time; this kernel hides both under streaming:
//  * A unit is one (sub-group, kv head): the sub-group's shared keys past the
//    group prefix, then each member's own keys.  Its query rows (members x
//    heads, at most 16) are the N side of warp MMAs, so a shared page read
//    serves every member (a sequence alone is a sub-group of one).
//  * A unit's page list is cut into parts of at least 8 pages (at most 16
//    parts); a task is one part.  Tasks are numbered sub-group, kv head,
//    part, and handed out by a global counter, so that the parts of one unit
//    run at the same time on different warps and work balances dynamically.
//  * A persistent grid (one CTA per SM) of independent warps; no CTA barrier
//    after the start.  Each warp owns a ring of NST page slots gathered by
//    2-D TMA (128-byte swizzle, L2 evict-first).  The ring runs across task
//    boundaries: the next task's pages are in flight while the current one is
//    finished.
//  * Products as in the decode kernel: S^T = K Q^T and O^T = V^T P^T as
//    m16n8k16 warp MMAs, online softmax in fp32 (base 2), probabilities
//    rounded to bf16 once for both the product and the running sum.
//  * Every part writes its partial softmax state (o/l, m, l) per query row;
//    a second, short launch (a half-warp per query row, its sources' loads
//    in flight together) merges the parts of the row's unit in part order and
//    then the group prefix's partial states, and writes the bf16 row --
//    deterministic.
//  * The task counter is a plain atomic increment (a compare-and-swap loop on
//    one address serialises thousands of warps); it and the per-row merge
//    descriptors are zeroed, stream-ordered, before the launch (before the
//    prefix pass, so that this grid can start beside the pass as its
//    programmatic dependent).
//  * Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_units.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

constexpr int kTD = 128;  // head_dim of this kernel
constexpr int kTMaxSources = kTaskMaxParts + kMaxPrefixParts;  // partial states merged into one row at most
// The plan reads the contexts and prefix groups from shared memory (one round
// of loads per CTA) when they fit: up to kStageSeqs sequences and
// kStageGroups groups.
constexpr int kStageSeqs = 2048;
constexpr int kStageGroups = 256;

struct TaskArgs {
  const __nv_bfloat16 *q;
  const int32_t *bt;
  const int32_t *ctx;
  __nv_bfloat16 *out;
  const int32_t *sub_start;   // null: every sequence is a sub-group of one
  const int32_t *sub_shared;
  int nsg;                    // sub-groups (sequences when sub_start is null)
  const int32_t *grp_start;
  const int32_t *grp_prefix;
  int ngroups;
  const float *pre_o;         // [npre][S][Hq][D]
  const float *pre_ml;        // [npre][S][Hq][2]
  int npre;
  float *ws_o;                // [kTaskMaxParts][S][Hq][D] o/l of each part
  float *ws_ml;               // [kTaskMaxParts][S][Hq][2] (m, l) of each part
  unsigned int *ws_ctr;       // tasks handed out (zeroed per launch)
  int *row_info;              // [S][Hq]: parts of the row's unit | 256 if a prefix is folded in; 0 = none
  int32_t *err;
  int S, Hq, Hkv, G, rows, num_blocks, max_blocks, max_ctx;
  int part_pages;             // least pages of a part
  float scale_log2;
};

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int B, int W, int NST>
struct TaskSmem {
  static constexpr int kBoxBytes = B * 128;          // B rows x 64 bf16
  static constexpr int kPageBytes = 2 * kBoxBytes;   // one K (or V) run of D = 128
  static constexpr int kSlotBytes = 2 * kPageBytes;  // K then V
  static constexpr int kRingBytes = W * NST * kSlotBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kPlanOff = kBarOff + W * NST * 8;
  // plan: task base [kTaskMaxSub + 1], first sequence [kTaskMaxSub + 1],
  // pages [kTaskMaxSub], group prefix [kTaskMaxSub], shared length
  // [kTaskMaxSub], warp sums [W]
  static constexpr int kStageOff = kPlanOff + (5 * kTaskMaxSub + 2 + W) * 4;
  // staged plan inputs: contexts [kStageSeqs], group starts [kStageGroups + 1], group prefixes [kStageGroups]
  static constexpr int kBytes = kStageOff + (kStageSeqs + 2 * kStageGroups + 1) * 4;
  static constexpr int kAlloc = kBytes + 1024;
};

// Pages per part of a unit of n pages: at least min_pages, at most 16 parts
// (a part's entries fit the 32 lanes: n <= 512).
__device__ __forceinline__ int part_len(int n, int min_pages) {
  return max(min_pages, (n + kTaskMaxParts - 1) / kTaskMaxParts);
}

struct Task {
  int t;       // task number; >= total: none
  int kvh, part, nparts, s0, nm, kstart, np;
  int bad;     // the unit is invalid: its rows are zeroed
};

// The plan of a launch in shared memory (every CTA builds the same one).
struct TaskPlan {
  int *sg_base;    // [kTaskMaxSub + 1] first task of each sub-group
  int *sg_s0;      // [kTaskMaxSub + 1] first sequence of each sub-group
  int *sg_pages;   // [kTaskMaxSub] pages past the group prefix (-1: invalid)
  int *sg_kstart;  // [kTaskMaxSub] the group prefix (first key of the unit)
  int *sg_kshared; // [kTaskMaxSub] keys every member shares
  int *wsum;       // [warps] scan scratch
  int *ctx_s;      // [kStageSeqs] staged contexts
  int *gstart_s;   // [kStageGroups + 1] staged group starts
  int *gprefix_s;  // [kStageGroups] staged group prefixes
  bool staged;     // the contexts and groups fit the staging arrays
};

// Builds the plan on all NTH threads of the CTA: each sub-group's data, tasks
// per sub-group (one per part and kv head) and their prefix sums.  Its inputs
// are read in one round of independent loads, into shared memory when they
// fit.  The caller synchronises the CTA before reading it.
template <int B, int NTH>
__device__ __forceinline__ void build_task_plan(const TaskArgs &a, const TaskPlan &p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // every input load is issued before the first store waits for one: a
  // single round trip
  constexpr int kC = (kStageSeqs + NTH - 1) / NTH, kG = (kStageGroups + NTH) / NTH, kS = (kTaskMaxSub + NTH) / NTH;
  int vc[kC], vgs[kG], vgp[kG], vs0[kS], vsh[kS];
  if (p.staged) {
#pragma unroll
    for (int k = 0; k < kC; ++k) {
      const int i = tid + k * NTH;
      vc[k] = i < a.S ? __ldg(a.ctx + i) : 0;
    }
#pragma unroll
    for (int k = 0; k < kG; ++k) {
      const int i = tid + k * NTH;
      vgs[k] = i <= a.ngroups && a.ngroups > 0 ? __ldg(a.grp_start + i) : 0;
      vgp[k] = i < a.ngroups ? __ldg(a.grp_prefix + i) : 0;
    }
  }
#pragma unroll
  for (int k = 0; k < kS; ++k) {
    const int sg = tid + k * NTH;
    vs0[k] = sg <= a.nsg ? (a.sub_start ? __ldg(a.sub_start + sg) : sg) : 0;
    vsh[k] = sg < a.nsg ? (a.sub_start ? __ldg(a.sub_shared + sg) : -1) : 0;
  }
  if (p.staged) {
#pragma unroll
    for (int k = 0; k < kC; ++k)
      if (tid + k * NTH < a.S) p.ctx_s[tid + k * NTH] = vc[k];
#pragma unroll
    for (int k = 0; k < kG; ++k) {
      const int i = tid + k * NTH;
      if (i <= a.ngroups && a.ngroups > 0) p.gstart_s[i] = vgs[k];
      if (i < a.ngroups) p.gprefix_s[i] = vgp[k];
    }
  }
#pragma unroll
  for (int k = 0; k < kS; ++k) {
    const int sg = tid + k * NTH;
    if (sg <= a.nsg) p.sg_s0[sg] = vs0[k];
    if (sg < a.nsg) p.sg_kshared[sg] = vsh[k];
  }
  __syncthreads();
  const UnitShape us{a.S, a.G, a.rows, a.max_blocks, a.max_ctx, a.ngroups};
  for (int sg = tid; sg < a.nsg; sg += NTH) {
    int ks, n;
    if (p.staged)
      subgroup_plan(
          us, B, p.sg_s0[sg], p.sg_s0[sg + 1], p.sg_kshared[sg], [&](int i) { return p.ctx_s[i]; },
          [&](int i) { return p.gstart_s[i]; }, [&](int i) { return p.gprefix_s[i]; }, &ks, &n);
    else
      subgroup_plan(
          us, B, p.sg_s0[sg], p.sg_s0[sg + 1], p.sg_kshared[sg], [&](int i) { return __ldg(a.ctx + i); },
          [&](int i) { return __ldg(a.grp_start + i); }, [&](int i) { return __ldg(a.grp_prefix + i); }, &ks, &n);
    if (p.sg_kshared[sg] < 0) p.sg_kshared[sg] = ks;
    p.sg_kstart[sg] = ks;
    p.sg_pages[sg] = n;
    p.sg_base[sg + 1] =
        a.Hkv * (n < 0 ? 1 : (n + part_len(n, a.part_pages) - 1) / part_len(n, a.part_pages) + (n == 0));
  }
  __syncthreads();
  constexpr int kPer = (kTaskMaxSub + NTH - 1) / NTH;
  int c[kPer], sum = 0;
  const int lo = tid * kPer;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    c[k] = lo + k < a.nsg ? p.sg_base[lo + k + 1] : 0;
    sum += c[k];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) p.wsum[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += p.wsum[w];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    run += c[k];
    if (lo + k < a.nsg) p.sg_base[lo + k + 1] = run;
  }
  if (tid == 0) p.sg_base[0] = 0;
}

// Task t -> its description, on a whole warp; lane j < np holds page j of
// the part: its table entry (CHECK: validated here, -1 if bad; else raw, to
// be checked where it is used, so that the load is waited for only then),
// first token, owner member (-1: shared) and the context that bounds its
// keys.  Also warms L2 with the unit's query rows.
template <int B, bool CHECK>
__device__ __forceinline__ void describe_task(const TaskArgs &a, const TaskPlan &p, int total, int t, Task &T,
                                              int &e_pg, int &e_tok, int &e_own, int &e_octx) {
  const int lane = threadIdx.x & 31;
  T.t = t;
  T.np = 0;
  T.bad = 0;
  e_pg = -1;
  e_tok = 0;
  e_own = -1;
  e_octx = 0;
  if (t >= total) return;
  int lo = 0, hi = a.nsg;  // sg_base[lo] <= t < sg_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.sg_base[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int sg = lo;
  T.nparts = (p.sg_base[sg + 1] - p.sg_base[sg]) / a.Hkv;
  const int rem = t - p.sg_base[sg];
  T.kvh = rem / T.nparts;
  T.part = rem - T.kvh * T.nparts;
  const int n = p.sg_pages[sg];
  T.kstart = p.sg_kstart[sg];
  T.s0 = p.sg_s0[sg];
  T.nm = p.sg_s0[sg + 1] - T.s0;
  if (n < 0) {
    T.bad = 1;
    return;
  }
  const int kshared = p.sg_kshared[sg];
  const int plen = part_len(n, a.part_pages);
  const int p0 = T.part * plen;
  T.np = max(0, min(n, p0 + plen) - p0);
  // members' contexts and the end of each member's own pages (after the shared ones)
  const int c = lane < T.nm ? (p.staged ? p.ctx_s[T.s0 + lane] : __ldg(a.ctx + T.s0 + lane)) : 0;
  const int own = lane < T.nm ? (c + B - 1) / B - kshared / B : 0;
  int incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int shared_pages = (kshared - T.kstart) / B;
  const int i = p0 + lane;
  int m = -1, lb = T.kstart / B + i;
  for (int mm = 0; mm < T.nm; ++mm) {
    const int e = __shfl_sync(0xffffffffu, incl, mm), o = __shfl_sync(0xffffffffu, own, mm);
    if (i >= shared_pages && m < 0 && i < shared_pages + e) {
      m = mm;
      lb = kshared / B + (i - (shared_pages + e - o));
    }
  }
  const int cm = __shfl_sync(0xffffffffu, c, max(m, 0));
  if (lane < T.np) {
    int pg = __ldg(a.bt + (size_t)(T.s0 + max(m, 0)) * a.max_blocks + lb);
    if (CHECK && (pg < 0 || pg >= a.num_blocks)) {
      if (a.err) atomicOr(a.err, PA_DEVERR_PAGE);
      pg = -1;
    }
    e_pg = pg;
    e_tok = lb * B;
    e_own = m;
    e_octx = m >= 0 ? cm : kshared;
  }
  for (int g = lane; g < T.nm * a.G; g += 32) {
    const __nv_bfloat16 *qr = a.q + ((size_t)(T.s0 + g / a.G) * a.Hq + (size_t)T.kvh * a.G + g % a.G) * kTD;
    prefetch_l2(qr);
    prefetch_l2(qr + 64);
  }
}

template <int B, int NT, int W, int NST>
__global__ void __launch_bounds__(W * 32, 1)
    decode_tasks_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const TaskArgs a) {
  using L = TaskSmem<B, W, NST>;
  constexpr int MT = B / 16;  // 16-token tiles per page
  constexpr int KS = kTD / 16, DT = kTD / 16;
  constexpr int NTH = W * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
  int *sg_base = reinterpret_cast<int *>(smem + L::kPlanOff);
  int *sg_s0 = sg_base + kTaskMaxSub + 1;
  int *sg_pages = sg_s0 + kTaskMaxSub + 1;
  int *sg_kstart = sg_pages + kTaskMaxSub;
  int *sg_kshared = sg_kstart + kTaskMaxSub;
  int *wsum = sg_kshared + kTaskMaxSub;
  int *ctx_s = reinterpret_cast<int *>(smem + L::kStageOff);
  int *gstart_s = ctx_s + kStageSeqs;
  int *gprefix_s = gstart_s + kStageGroups + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the merge launch behind this grid may be scheduled at once (it waits for
  // this grid's completion before reading anything)
  asm volatile("griddepcontrol.launch_dependents;");

  // the first task of each warp: handed out while the plan is made
  unsigned int first = 0;
  if (lane == 0) first = atomicAdd(a.ws_ctr, 1u);

  // ---- plan (every CTA the same)
  const TaskPlan plan{sg_base, sg_s0, sg_pages, sg_kstart, sg_kshared, wsum, ctx_s, gstart_s, gprefix_s,
                      a.S <= kStageSeqs && a.ngroups <= kStageGroups};
  build_task_plan<B, NTH>(a, plan);
  uint64_t *bars = bars_all + warp * NST;
  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int total = sg_base[a.nsg];
  const int G = a.G;
  const size_t slab = (size_t)a.S * a.Hq;
  uint8_t *ring = smem + warp * NST * L::kSlotBytes;
  const uint64_t pol = policy_evict_first();

  auto describe = [&](int t, Task &T, int &e_pg, int &e_tok, int &e_own, int &e_octx) {
    describe_task<B, true>(a, plan, total, t, T, e_pg, e_tok, e_own, e_octx);
  };
  auto fetch = [&]() -> int {
    int t = 0;
    if (lane == 0) t = (int)atomicAdd(a.ws_ctr, 1u);
    return __shfl_sync(0xffffffffu, t, 0);
  };

  // cur: the task being consumed; nxt: the one after it, described once the
  // first page of cur has been consumed (its table reads overlap the gathers
  // in flight); more: the counter may still hand out tasks
  Task cur, nxt;
  int c_pg, c_tok, c_own, c_octx, n_pg = -1, n_tok = 0, n_own = -1, n_octx = 0;
  describe((int)__shfl_sync(0xffffffffu, first, 0), cur, c_pg, c_tok, c_own, c_octx);
  bool more = cur.t < total, nxt_ready = false;
  nxt.t = total;
  nxt.np = 0;
  auto describe_next = [&]() {
    if (nxt_ready) return;
    if (more) {  // (table entries checked where they are used: no wait here)
      describe_task<B, false>(a, plan, total, fetch(), nxt, n_pg, n_tok, n_own, n_octx);
      more = nxt.t < total;
    } else {
      nxt.t = total;
      nxt.np = 0;
    }
    nxt_ready = true;
  };

  // a table entry of the next task, at its first use: -1 (and the error
  // flag) if it is outside the pool
  auto checked = [&](int pg, bool flag) {
    if (pg < 0 || pg >= a.num_blocks) {
      if (flag && a.err) atomicOr(a.err, PA_DEVERR_PAGE);
      pg = -1;
    }
    return pg;
  };

  // ring positions: pages issued / consumed so far; the issue pointer is in
  // the current task (which 0) or the next one (which 1) at page `at`
  long long issued = 0, consumed = 0;
  int which = 0, at = 0;
  auto issue_one = [&](int pg, int kvh) {  // whole warp; lane 0 issues
    __syncwarp();
    if (lane == 0) {
      const int slot = (int)(issued % NST);
      uint64_t *bar = &bars[slot];
      if (pg < 0) {
        mbar_arrive(bar);
      } else {  // (a slot's generic writes were fenced by their writers)
        mbar_arrive_expect_tx(bar, L::kSlotBytes);
        uint8_t *dst = ring + slot * L::kSlotBytes;
        const int row = (pg * a.Hkv + kvh) * B;
        tma_load_3d_hint(dst, &tmK, 0, row, 0, bar, pol);  // both 64-column halves
        tma_load_3d_hint(dst + L::kPageBytes, &tmV, 0, row, 0, bar, pol);
      }
    }
    ++issued;
  };
  auto top_up = [&]() {
    while (issued - consumed < NST) {
      if (which == 0) {
        if (at < cur.np) {
          issue_one(__shfl_sync(0xffffffffu, c_pg, at), cur.kvh);
          ++at;
          continue;
        }
        if (!nxt_ready || nxt.t >= total) return;
        which = 1;
        at = 0;
      }
      if (at >= nxt.np) return;
      issue_one(checked(__shfl_sync(0xffffffffu, n_pg, at), lane == 0), nxt.kvh);
      ++at;
    }
  };

  // Q^T fragments (MMA B operand) of a task: query row 8nt + lane/4 of its
  // unit, d pairs; loaded before the task's gathers are issued (which may
  // wait for its table entries), so that the two round trips overlap.  A
  // lane needs the bf16 pairs (words) c, c + 4, c + 8, ... of its two rows
  // (c = lane % 4); it loads their 16-byte blocks c + 4m (m < 4) instead,
  // a quarter of the load instructions, and the four lanes of a row trade
  // words in one 4 x 4 transpose per m: rotate the block left by c, take
  // word j from lane c - j, rotate back.
  uint32_t qf[NT][KS][2];
  static_assert(KS == 8, "a row is 16 blocks of 16 bytes");
  auto load_q = [&](const Task &T) {
    const int c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = nt * 8 + (lane >> 2);
      const bool ok = !T.bad && g < T.nm * G;
      const uint4 *qr = reinterpret_cast<const uint4 *>(
          a.q + ((size_t)(T.s0 + g / G) * a.Hq + (size_t)T.kvh * G + g % G) * kTD);
      uint4 v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) v[m] = ok ? __ldg(qr + c + 4 * m) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t r[4] = {v[m].x, v[m].y, v[m].z, v[m].w};  // words 4 (c + 4m) + k
        uint32_t t[4], p[4], u[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) t[j] = (c & 1) ? r[(j + 1) & 3] : r[j];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = (c & 2) ? t[(j + 2) & 3] : t[j];
        u[0] = p[0];
#pragma unroll
        for (int j = 1; j < 4; ++j) u[j] = __shfl_sync(0xffffffffu, p[j], (lane & ~3) | ((c - j) & 3));
        // u[j] = word 4 (((c - j) & 3) + 4m) + c; rotate (u0, u3, u2, u1) right by c
        const uint32_t w[4] = {u[0], u[3], u[2], u[1]};
#pragma unroll
        for (int j = 0; j < 4; ++j) t[j] = (c & 1) ? w[(j + 3) & 3] : w[j];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = (c & 2) ? t[(j + 2) & 3] : t[j];
#pragma unroll
        for (int j = 0; j < 4; ++j) qf[nt][(4 * m + j) >> 1][(4 * m + j) & 1] = p[j];  // word 4 (4m + j) + c
      }
    }
  };

  bool timed_out = false;
  while (cur.t < total && !timed_out) {
    const int ncols = cur.nm * G;
    auto row_of = [&](int g) -> size_t {
      return (size_t)(cur.s0 + g / G) * a.Hq + (size_t)cur.kvh * G + g % G;
    };
    load_q(cur);
    if (cur.np == 0) describe_next();  // nothing of cur to overlap it with
    top_up();
    float m_run[NT][2], l_run[NT][2], o[NT][DT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) o[nt][dt][0] = o[nt][dt][1] = o[nt][dt][2] = o[nt][dt][3] = 0.f;
    }

    for (int k = 0; k < cur.np; ++k) {
      const int stg = (int)(consumed % NST);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[stg], (uint32_t)((consumed / NST) & 1)))) {
        timed_out = true;
        break;
      }
      const int pg = __shfl_sync(0xffffffffu, c_pg, k);
      const int tok0 = __shfl_sync(0xffffffffu, c_tok, k);
      const int owner = __shfl_sync(0xffffffffu, c_own, k);
      const int octx = __shfl_sync(0xffffffffu, c_octx, k);
      if (pg >= 0) {
        const uint32_t kb = smem_u32(ring + stg * L::kSlotBytes);
        const uint32_t vb = kb + L::kPageBytes;
        // S^T[token][row] = K Q^T
        float sc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) sc[mt][nt][0] = sc[mt][nt][1] = sc[mt][nt][2] = sc[mt][nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int c = 2 * kk + (lane >> 4);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            uint32_t af[4];
            ldsm_x4(kb + (c >> 3) * L::kBoxBytes + sw128(r, c & 7), af);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sc[mt][nt], af, qf[nt][kk][0], qf[nt][kk][1]);
          }
        }
        // online softmax: a member's own page counts only for its rows; keys
        // past the bounding context are masked.  The running maximum moves
        // only when a row's page maximum passes it by more than kSlack (a
        // factor 2^kSlack), so that the probabilities can be taken against it
        // while the page maxima are still being reduced, and the rescale of
        // the row's state is rare.
        constexpr float kSlack = 8.f;
        float t[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          t[nt][0] = t[nt][1] = -INFINITY;
          const bool own0 = owner < 0 || (nt * 8 + 2 * (lane & 3)) / G == owner;
          const bool own1 = owner < 0 || (nt * 8 + 2 * (lane & 3) + 1) / G == owner;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int j = tok0 + mt * 16 + (lane >> 2);
            const bool v0 = j < octx, v1 = j + 8 < octx;
            sc[mt][nt][0] = v0 && own0 ? sc[mt][nt][0] * a.scale_log2 : -INFINITY;
            sc[mt][nt][1] = v0 && own1 ? sc[mt][nt][1] * a.scale_log2 : -INFINITY;
            sc[mt][nt][2] = v1 && own0 ? sc[mt][nt][2] * a.scale_log2 : -INFINITY;
            sc[mt][nt][3] = v1 && own1 ? sc[mt][nt][3] * a.scale_log2 : -INFINITY;
            t[nt][0] = fmaxf(t[nt][0], fmaxf(sc[mt][nt][0], sc[mt][nt][2]));
            t[nt][1] = fmaxf(t[nt][1], fmaxf(sc[mt][nt][1], sc[mt][nt][3]));
          }
        }
        // P (bf16 pairs) against the running maxima; a row that has seen no
        // key yet (maximum -inf) takes 0, so that no -inf - -inf appears
        uint32_t plo[MT][NT], phi[MT][NT];
        auto probabilities = [&]() {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float e0 = m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0];
            const float e1 = m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              plo[mt][nt] = pack_bf16(ex2_ftz(sc[mt][nt][0] - e0), ex2_ftz(sc[mt][nt][1] - e1));
              phi[mt][nt] = pack_bf16(ex2_ftz(sc[mt][nt][2] - e0), ex2_ftz(sc[mt][nt][3] - e1));
            }
          }
        };
        probabilities();
        bool grow = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            t[nt][0] = fmaxf(t[nt][0], __shfl_xor_sync(0xffffffffu, t[nt][0], off));
            t[nt][1] = fmaxf(t[nt][1], __shfl_xor_sync(0xffffffffu, t[nt][1], off));
          }
          grow |= t[nt][0] > m_run[nt][0] + kSlack || t[nt][1] > m_run[nt][1] + kSlack;
        }
        if (__any_sync(0xffffffffu, grow)) {  // new maxima: rescale the state, retake P
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float mn0 = fmaxf(m_run[nt][0], t[nt][0]), mn1 = fmaxf(m_run[nt][1], t[nt][1]);
            const float su0 = mn0 == -INFINITY ? 0.f : mn0, su1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2f(m_run[nt][0] - su0), al1 = exp2f(m_run[nt][1] - su1);
            m_run[nt][0] = mn0;
            m_run[nt][1] = mn1;
            l_run[nt][0] *= al0;
            l_run[nt][1] *= al1;
#pragma unroll
            for (int dt = 0; dt < DT; ++dt) {
              o[nt][dt][0] *= al0;
              o[nt][dt][1] *= al1;
              o[nt][dt][2] *= al0;
              o[nt][dt][3] *= al1;
            }
          }
          probabilities();
        }
        // value rows past the bounding context may hold any bits (NaN
        // included) and would meet a zero probability: clear them
        if (tok0 + B > octx) {
          uint8_t *vslot = ring + stg * L::kSlotBytes + L::kPageBytes;
          const int r0 = octx - tok0;
          for (int idx = lane; idx < (B - r0) * 16; idx += 32) {
            const int row = r0 + idx / 16, rem = idx % 16;
            *reinterpret_cast<uint4 *>(vslot + (rem >> 3) * L::kBoxBytes + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the slot is refilled by TMA afterwards
          __syncwarp();
        }
        // O^T[d][row] += V^T P^T, one 16-token k-tile at a time
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t pb[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            l_run[nt][0] += bf16_lo(plo[mt][nt]) + bf16_lo(phi[mt][nt]);
            l_run[nt][1] += bf16_hi(plo[mt][nt]) + bf16_hi(phi[mt][nt]);
            pb[nt][0] = movmatrix_t(plo[mt][nt]);
            pb[nt][1] = movmatrix_t(phi[mt][nt]);
          }
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            const int r = mt * 16 + (lane & 7) + (lane >> 4) * 8;
            const int c = 2 * dt + ((lane >> 3) & 1);
            uint32_t af[4];
            ldsm_x4_t(vb + (c >> 3) * L::kBoxBytes + sw128(r, c & 7), af);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(o[nt][dt], af, pb[nt][0], pb[nt][1]);
          }
        }
      }
      ++consumed;
      if (k == 0) describe_next();
      top_up();  // the freed slot takes the next page (of this task or the next)
    }
    if (timed_out) break;

    // ---- finish the task: its partial state for every row of the unit
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l_run[nt][e] += __shfl_xor_sync(0xffffffffu, l_run[nt][e], off);
    if (cur.bad) {
      const bool in_range = cur.s0 >= 0 && cur.nm > 0 && cur.s0 + cur.nm <= a.S;
      if (in_range)
        for (int g = 0; g < ncols; ++g)
          reinterpret_cast<uint2 *>(a.out + row_of(g) * kTD)[lane] = make_uint2(0u, 0u);
      if (lane == 0 && a.err) atomicOr(a.err, PA_DEVERR_CTX);
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int g = nt * 8 + 2 * (lane & 3) + e;
          if (g >= ncols) continue;
          const size_t pr = (size_t)cur.part * slab + row_of(g);
          const float l = l_run[nt][e];
          const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            const int d = dt * 16 + (lane >> 2);
            a.ws_o[pr * kTD + d] = o[nt][dt][e] * inv;
            a.ws_o[pr * kTD + d + 8] = o[nt][dt][2 + e] * inv;
          }
          if (lane < 4) {
            a.ws_ml[2 * pr] = m_run[nt][e];
            a.ws_ml[2 * pr + 1] = l;
          }
        }
      }
      if (cur.part == 0)  // the merge's descriptor of the unit's rows
        for (int g = lane; g < ncols; g += 32) a.row_info[row_of(g)] = cur.nparts | (cur.kstart > 0 ? 256 : 0);
    }

    // ---- the next task becomes current
    describe_next();
    cur = nxt;
    c_pg = lane < nxt.np ? checked(n_pg, true) : n_pg;
    c_tok = n_tok;
    c_own = n_own;
    c_octx = n_octx;
    nxt_ready = false;
    if (which == 1) {
      which = 0;  // the issue pointer keeps its place, now in the current task
    } else {
      at = 0;     // nothing of the new task was issued yet
    }
  }
  if (timed_out) {
    if (lane == 0 && a.err) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    for (long long p = consumed; p < issued; ++p) mbar_wait(&bars[p % NST], (uint32_t)((p / NST) & 1));
  }
  // Launched as a programmatic dependent of the prefix pass, this grid may
  // run beside it (it reads nothing the pass writes): it completes only after
  // the pass has, so that the merge launch behind it sees the pass's states.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Two query rows a warp (a half-warp each): the row's partial states -- its
// unit's parts in part order, then the group prefix's key ranges -- merged
// with weights l_p 2^(m_p - M) / sum, written as bf16.  Lane: 8 output
// elements of its half's row; sources' loads four at a time.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeWarps * 32) merge_rows_kernel(const TaskArgs a) {
  // a programmatic dependent of the task grid: resident early, it starts
  // merging once every task (and the prefix pass before them) is complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const size_t R = (size_t)a.S * a.Hq;
  const size_t row = ((size_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5)) * 2 + half;
  const int info = row < R ? a.row_info[row] : 0;  // 0: no unit covered this row (refused, or past the end)
  const int nparts = info & 255, nsrc = info ? nparts + ((info & 256) ? a.npre : 0) : 0;
  // (m, l) of sources hl and hl + 16 of this half's row
  auto ml_of = [&](int k) -> float2 {
    if (k < nparts) return __ldcg(reinterpret_cast<const float2 *>(a.ws_ml) + (size_t)k * R + row);
    if (k < nsrc) return __ldg(reinterpret_cast<const float2 *>(a.pre_ml) + (size_t)(k - nparts) * R + row);
    return make_float2(-INFINITY, 0.f);
  };
  const float2 s0 = ml_of(hl), s1 = ml_of(hl + 16);
  float M = fmaxf(s0.y > 0.f ? s0.x : -INFINITY, s1.y > 0.f ? s1.x : -INFINITY);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float w0 = s0.y > 0.f ? s0.y * exp2f(s0.x - M) : 0.f, w1 = s1.y > 0.f ? s1.y * exp2f(s1.x - M) : 0.f;
  float den = w0 + w1;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  w0 *= inv;
  w1 *= inv;
  const int nmax = max(nsrc, __shfl_xor_sync(0xffffffffu, nsrc, 16));  // the warp's loop bound
  float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
  for (int k0 = 0; k0 < nmax; k0 += 4) {
    float4 v[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + j;
      const float4 *src = k < nparts ? reinterpret_cast<const float4 *>(a.ws_o + ((size_t)k * R + row) * kTD)
                                     : reinterpret_cast<const float4 *>(a.pre_o + ((size_t)(k - nparts) * R + row) * kTD);
      v[j][0] = v[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < nsrc) {
        v[j][0] = __ldcg(src + 2 * hl);
        v[j][1] = __ldcg(src + 2 * hl + 1);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + j;
      const float wk = __shfl_sync(0xffffffffu, k < 16 ? w0 : w1, (half << 4) | (k & 15));
      if (k < nsrc) {
        acc0.x += wk * v[j][0].x;
        acc0.y += wk * v[j][0].y;
        acc0.z += wk * v[j][0].z;
        acc0.w += wk * v[j][0].w;
        acc1.x += wk * v[j][1].x;
        acc1.y += wk * v[j][1].y;
        acc1.z += wk * v[j][1].z;
        acc1.w += wk * v[j][1].w;
      }
    }
  }
  if (info) {
    uint4 packed;
    packed.x = pack_bf16(acc0.x, acc0.y);
    packed.y = pack_bf16(acc0.z, acc0.w);
    packed.z = pack_bf16(acc1.x, acc1.y);
    packed.w = pack_bf16(acc1.z, acc1.w);
    reinterpret_cast<uint4 *>(a.out + row * kTD)[hl] = packed;
  }
}

template <int B, int NT>
int launch_tasks(const CUtensorMap &tk, const CUtensorMap &tv, const TaskArgs &a, int sms, cudaStream_t st) {
  // 16-token pages: 8 warps with three 8 KB slots each; 32-token pages: 6
  // warps with two 16 KB slots -- about 192 KB of pages in flight per SM.
  constexpr int W = B == 16 ? 8 : 6;
  constexpr int NST = B == 16 ? 3 : 2;
  using L = TaskSmem<B, W, NST>;
  static_assert(L::kAlloc <= 227 * 1024, "task decode shared memory over the per-CTA limit");
  static_assert(kTaskMaxSub <= 8 * W * 32, "plan scan: at most 8 sub-groups a thread");
  auto kern = decode_tasks_kernel<B, NT, W, NST>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
    return PA_ERR_CUDA;
  // a programmatic dependent of the kernel before it on the stream (the
  // prefix pass): its CTAs may start as soon as that kernel allows
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tk, tv, a) != cudaSuccess) return PA_ERR_CUDA;
  const size_t R = (size_t)a.S * a.Hq;
  cfg.gridDim = dim3((unsigned)((R + 2 * kMergeWarps - 1) / (2 * kMergeWarps)));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, merge_rows_kernel, a) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t task_workspace_bytes(const pa_decode_desc *d) {
  const size_t rows = (size_t)d->num_seqs * d->num_q_heads;
  return up256((size_t)kTaskMaxParts * rows * kTD * sizeof(float)) +
         up256((size_t)kTaskMaxParts * rows * 2 * sizeof(float)) + up256((1 + rows) * sizeof(int));
}

bool tasks_supported(const pa_decode_desc *d, int nsg, int rows) {
  return d->head_dim == kTD && nsg > 0 && nsg <= kTaskMaxSub && nsg <= d->num_seqs && rows > 0 && rows <= 16 &&
         (long long)d->num_kv_heads * nsg * (kTaskMaxParts + 1) < (1ll << 30) &&
         (long long)d->num_seqs * d->num_q_heads < (1ll << 31);
}

unsigned int *task_counter(const pa_decode_desc *d, void *workspace) {
  const size_t R = (size_t)d->num_seqs * d->num_q_heads;
  return reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(workspace) +
                                          up256(kTaskMaxParts * R * kTD * sizeof(float)) +
                                          up256(kTaskMaxParts * R * 2 * sizeof(float)));
}

int decode_tasks_clear(const pa_decode_desc *d, void *workspace, void *stream) {
  const size_t R = (size_t)d->num_seqs * d->num_q_heads;
  uint8_t *ctr = static_cast<uint8_t *>(workspace) + up256(kTaskMaxParts * R * kTD * sizeof(float)) +
                 up256(kTaskMaxParts * R * 2 * sizeof(float));
  return cudaMemsetAsync(ctr, 0, (1 + R) * sizeof(int), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int decode_tasks_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                        const int32_t *block_tables, const int32_t *context_lens, const DecodePrefix &pre, int rows,
                        void *out, void *workspace, int32_t *err_flag, void *stream) {
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const uint64_t nrows = (uint64_t)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tk, tv;
  if (!encode_kv_halves_3d(&tk, k_pool, nrows, d->block_size) ||
      !encode_kv_halves_3d(&tv, v_pool, nrows, d->block_size))
    return PA_ERR_CUDA;
  const size_t R = (size_t)d->num_seqs * d->num_q_heads;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  TaskArgs a{};
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.bt = block_tables;
  a.ctx = context_lens;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.sub_start = pre.nsub > 0 ? pre.sub_start : nullptr;
  a.sub_shared = pre.nsub > 0 ? pre.sub_shared : nullptr;
  a.nsg = pre.nsub > 0 ? pre.nsub : d->num_seqs;
  a.grp_start = pre.grp_start;
  a.grp_prefix = pre.grp_prefix;
  a.ngroups = pre.ngroups;
  a.pre_o = pre.pre_o;
  a.pre_ml = pre.pre_ml;
  a.npre = pre.npre;
  a.ws_o = reinterpret_cast<float *>(ws);
  a.ws_ml = reinterpret_cast<float *>(ws + up256(kTaskMaxParts * R * kTD * sizeof(float)));
  a.ws_ctr = reinterpret_cast<unsigned int *>(ws + up256(kTaskMaxParts * R * kTD * sizeof(float)) +
                                              up256(kTaskMaxParts * R * 2 * sizeof(float)));
  a.row_info = reinterpret_cast<int *>(a.ws_ctr + 1);
  a.err = err_flag;
  a.S = d->num_seqs;
  a.Hq = d->num_q_heads;
  a.Hkv = d->num_kv_heads;
  a.G = d->num_q_heads / d->num_kv_heads;
  a.rows = rows;
  a.num_blocks = d->num_blocks;
  a.max_blocks = d->max_blocks_per_seq;
  a.max_ctx = d->max_context_len;
  a.scale_log2 = d->scale * 1.4426950408889634f;
  a.part_pages = 8;
  const char *env = getenv("PA_TASK_PART_PAGES");  // tuning
  if (env && atoi(env) > 0 && atoi(env) <= 32) a.part_pages = atoi(env);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->block_size == 16)
    return rows <= 8 ? launch_tasks<16, 1>(tk, tv, a, sms, s) : launch_tasks<16, 2>(tk, tv, a, sms, s);
  return rows <= 8 ? launch_tasks<32, 1>(tk, tv, a, sms, s) : launch_tasks<32, 2>(tk, tv, a, sms, s);
}

}  // namespace pa
