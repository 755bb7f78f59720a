// The paged decode unit of libpagedattn (sm_103a): argument block, shared
// memory layout and the per-unit device code, included by the decode kernel
// (pa_decode.cu) and the mixed-step kernel (pa_mixed.cu).  The design notes
// are at the top of pa_decode.cu.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

// Barrier `bar` over the N threads of one unit (bar 0 with N = the CTA's
// threads is __syncthreads).
template <int N>
__device__ __forceinline__ void unit_sync(int bar) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(N) : "memory");
}

struct DecodeArgs {
  const __nv_bfloat16 *q;
  const int32_t *bt;
  const int32_t *ctx;
  __nv_bfloat16 *out;
  float *ws_o;
  float *ws_ml;
  unsigned long long *ws_cnt;  // per (sequence, kv head): epoch << 32 | arrivals
  int32_t *err;
  int S, Hq, Hkv, G, num_blocks, max_blocks, max_ctx, part_pages, max_parts;
  float scale_log2;
  unsigned int epoch;  // unique per call, never 0
  int lpt;             // order CTAs longest context first
  // Shared-prefix groups (optional): sequences grp_start[k] .. grp_start[k+1]-1
  // share their first grp_prefix[k] tokens (whole blocks), whose attention was
  // computed by a separate pass into the partial states pre_o / pre_ml; this
  // kernel then covers keys grp_prefix[k] .. ctx-1 and folds that partial in.
  const int32_t *grp_start;
  const int32_t *grp_prefix;
  int ngroups;
  const float *pre_o;   // [npre][S][Hq][D] o/l of the prefix's key ranges
  const float *pre_ml;  // [npre][S][Hq][2] (m, l) of the prefix's key ranges
  int npre;
  // Sub-groups (GRP launches): sequences sub_start[k] .. sub_start[k+1]-1
  // share keys 0 .. sub_shared[k]-1 (whole blocks; the first grp_prefix of
  // them attended by the prefix pass).  One unit per (sub-group, kv head)
  // attends the shared keys once for all members' query rows and each
  // member's own keys for its rows only.
  const int32_t *sub_start;
  const int32_t *sub_shared;
  int nsub;
  int sub_rows;  // bound on a sub-group's query rows (members x G)
  // Append (optional): app_k/app_v [S][Hkv][D] hold each sequence's newest
  // token, which belongs at position ctx-1 in slot app_slots[s] (< 0: none).
  const uint4 *app_k;
  const uint4 *app_v;
  const int64_t *app_slots;
  uint4 *kp;  // the pools, written through for the append
  uint4 *vp;
};

// Counts one arrival of this call at *c and returns the arrivals so far.  A
// counter whose epoch tag is not this call's (left by another call or holding
// stale data) restarts at 1, so the workspace needs no zero-fill.
__device__ __forceinline__ unsigned int arrive_count(unsigned long long *c, unsigned int epoch) {
  const unsigned long long tag = (unsigned long long)epoch << 32;
  unsigned long long old = atomicAdd(c, 0ull), prev;
  for (;;) {
    const unsigned long long nv = ((old >> 32) == epoch) ? old + 1 : (tag | 1ull);
    prev = atomicCAS(c, old, nv);
    if (prev == old) return (unsigned int)(nv & 0xffffffffull);
    old = prev;
  }
}

template <int D, int B, int NW, int NST>
struct DecodeSmem {
  static constexpr int kHalves = D / 64;           // 64-column TMA boxes per row
  static constexpr int kBoxBytes = B * 128;        // B rows x 128 bytes
  static constexpr int kPageBytes = kHalves * kBoxBytes;
  static constexpr int kSlotBytes = 2 * kPageBytes;  // K then V
  static constexpr int kRingBytes = NW * NST * kSlotBytes;
  // After streaming, the ring is reused for the merge buffers (floats):
  // red_o [NW][16][D], red_m [NW][16], red_l [NW][16], wts [kMaxParts][16].
  static constexpr int kRedBytes = (NW * 16 * D + 2 * NW * 16 + kMaxParts * 16) * 4;
  static constexpr int kRegion0 = kRingBytes > kRedBytes ? kRingBytes : kRedBytes;
  static constexpr int kBarOff = (kRegion0 + 1023) & ~1023;
  static constexpr int kTblOff = kBarOff + NW * NST * 8;
  static constexpr int kMiscOff = kTblOff + kMaxPartPages * 4;
  // misc: [0..3] broadcast words, [4..7] warp totals, [8..135] length histogram
  static constexpr int kStageOff = kMiscOff + 4 * 136;  // appended token's K then V row
  static constexpr int kMetaOff = kStageOff + 2 * D * 2;  // GRP: per page, owner + 1 << 24 | logical block
  static constexpr int kBytes = kMetaOff + kMaxPartPages * 4;
  static constexpr int kAlloc = kBytes + 1024;  // base re-aligned to 1024 in the kernel
};

// Length class of a sequence for longest-first ordering: quarter-octave
// buckets of its page count (1 .. 68), 0 for an invalid context.
__device__ __forceinline__ int length_bucket(int ctx, int B, int max_blocks, int max_ctx) {
  if (ctx <= 0 || ctx > max_blocks * B || ctx > max_ctx) return 0;
  const int p = (ctx + B - 1) / B;
  const int msb = 31 - __clz(p);
  const int frac = msb >= 2 ? (p >> (msb - 2)) & 3 : (p << (2 - msb)) & 3;
  return 4 * msb + frac + 1;
}

// Index of the sequence of rank r when sequences are ordered by decreasing
// length bucket, ties in index order.  Whole CTA; misc holds 136 ints.
template <int NT_>
__device__ int seq_of_rank(int r, const int32_t *ctx, int S, int B, int max_blocks, int max_ctx, int *misc,
                           int tid, int bar) {
  constexpr int kThreads = NT_;
  int *hist = misc + 8;
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 128; i += kThreads) hist[i] = 0;
  unit_sync<kThreads>(bar);
  for (int i = tid; i < S; i += kThreads) atomicAdd(&hist[length_bucket(__ldg(ctx + i), B, max_blocks, max_ctx)], 1);
  unit_sync<kThreads>(bar);
  if (warp == 0) {  // bucket holding rank r, scanning buckets from the longest down
    int c[4], t = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[j] = hist[127 - 4 * lane - j];
      t += c[j];
    }
    int incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - t;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (r >= run && r < run + c[j]) {
        misc[0] = 127 - 4 * lane - j;
        misc[1] = r - run;
      }
      run += c[j];
    }
  }
  unit_sync<kThreads>(bar);
  const int bstar = misc[0], k = misc[1];
  const int chunk = (S + kThreads - 1) / kThreads;
  const int beg = min(S, tid * chunk), end = min(S, beg + chunk);
  int cnt = 0;
  for (int i = beg; i < end; ++i) cnt += length_bucket(__ldg(ctx + i), B, max_blocks, max_ctx) == bstar;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) misc[4 + warp] = incl;
  unit_sync<kThreads>(bar);
  int excl = incl - cnt;
  for (int w = 0; w < warp; ++w) excl += misc[4 + w];
  if (k >= excl && k < excl + cnt) {
    int left = k - excl;
    for (int i = beg; i < end; ++i)
      if (length_bucket(__ldg(ctx + i), B, max_blocks, max_ctx) == bstar && left-- == 0) misc[2] = i;
  }
  unit_sync<kThreads>(bar);
  return misc[2];
}

// One decode unit: (sequence part, kv head, sequence) number `lin` in launch
// order, on NW warps whose thread index within the unit is `tid`, with the
// unit's shared memory at `smem` (1024-aligned, DecodeSmem<...>::kBytes) and
// barrier `bar` for its own NW * 32 threads.  The decode kernel runs one unit
// per CTA; the mixed-step kernel runs several side by side in one CTA.
template <int D, int B, int NT, int NW, int NST, bool PRE, bool APP, bool GRP = false, bool TMA3 = false>
__device__ __forceinline__ void decode_unit(const CUtensorMap *tmK, const CUtensorMap *tmV, const DecodeArgs &a,
                                            int lin, int tid, uint8_t *smem, int bar) {
  using L = DecodeSmem<D, B, NW, NST>;
  static_assert(NW <= 4, "misc holds four warp totals");
  constexpr int KS = D / 16;  // k-steps of S^T = K Q^T
  constexpr int MT = B / 16;  // 16-token tiles per page
  constexpr int DT = D / 16;  // 16-row d tiles of O^T = V^T P^T

  constexpr bool FOLD = PRE || GRP;  // shared-prefix states to fold in at the end
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
  int32_t *tbl = reinterpret_cast<int32_t *>(smem + L::kTblOff);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);
  int32_t *meta = reinterpret_cast<int32_t *>(smem + L::kMetaOff);

  // Units are dispatched in linear order; map that order to (sequence rank,
  // part, kv head), ranks longest context first when a.lpt is set.  GRP: to
  // (sub-group rank, kv head), sub-groups ranked by their shared length when
  // a.lpt is set; s is the sub-group's first member.
  const int per_seq = a.max_parts * a.Hkv;
  const int rank = GRP ? lin / a.Hkv : lin / per_seq;
  const int part = GRP ? 0 : (lin - rank * per_seq) / a.Hkv;
  const int kvh = GRP ? lin - rank * a.Hkv : lin - rank * per_seq - part * a.Hkv;
  const bool rank_it = a.lpt && (GRP ? a.nsub : a.S) > 1;
  const int sg = GRP && rank_it
                     ? seq_of_rank<NW * 32>(rank, a.sub_shared, a.nsub, B, a.max_blocks, a.max_ctx, misc, tid, bar)
                     : rank;  // GRP: the sub-group
  const int s = GRP ? __ldg(a.sub_start + sg)
                    : rank_it ? seq_of_rank<NW * 32>(rank, a.ctx, a.S, B, a.max_blocks, a.max_ctx, misc, tid, bar)
                              : rank;
  const int nm = GRP ? __ldg(a.sub_start + sg + 1) - s : 1;  // members (query-row groups) of the unit
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  const int ncols = nm * G;  // query rows of the unit: member g / G, head g % G
  // GRP: a sub-group outside the batch is refused before anything is read
  const bool in_range = !GRP || (s >= 0 && nm > 0 && s + nm <= a.S);
  const int ctx = in_range ? __ldg(a.ctx + s) : 0;
  int kstart = 0;  // first key this kernel covers (end of a shared prefix; PRE and GRP launches only)
  if (FOLD && a.ngroups > 0 && s >= __ldg(a.grp_start) && s < __ldg(a.grp_start + a.ngroups)) {
    int lo = 0, hi = a.ngroups;  // grp_start[lo] <= s < grp_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(a.grp_start + mid) <= s) lo = mid;
      else hi = mid;
    }
    kstart = __ldg(a.grp_prefix + lo);
  }
  const bool has_pre = kstart > 0;
  // query row g of the unit: (sequence, head) -> row of q / out / the prefix states
  auto row_of = [&](int g) -> size_t {
    return GRP ? (size_t)(s + g / G) * a.Hq + (size_t)kvh * G + g % G : (size_t)s * a.Hq + (size_t)kvh * G + g;
  };
  int kshared = 0;  // GRP: end of the keys every member shares
  bool bad_grp = false;
  int npages_grp = 0;
  if constexpr (GRP) {
    // members' contexts in misc[8 ..], the start of each member's own pages
    // in the unit's page list in misc[24 ..] (the shared pages come first)
    kshared = __ldg(a.sub_shared + sg);
    if (in_range && tid < nm && tid < 16) misc[8 + tid] = __ldg(a.ctx + s + tid);
    unit_sync<NW * 32>(bar);
    if (tid == 0) {
      int ok = in_range && ncols <= NT * 8 && kshared >= kstart && kshared % B == 0 && kstart % B == 0;
      int at = ok ? (kshared - kstart) / B : 0;
      for (int m = 0; ok && m < nm; ++m) {
        const int c = misc[8 + m];
        ok = c >= kshared && c > 0 && c <= a.max_blocks * B && c <= a.max_ctx;
        misc[24 + m] = at;
        at += (c + B - 1) / B - kshared / B;
      }
      if (ok) misc[24 + nm] = at;
      misc[0] = ok && at <= kMaxPartPages;
    }
    unit_sync<NW * 32>(bar);
    bad_grp = !misc[0];
    npages_grp = bad_grp ? 0 : misc[24 + nm];
  }
  const bool bad = GRP ? bad_grp
                       : ctx <= 0 || ctx > a.max_blocks * B || ctx > a.max_ctx || kstart < 0 || kstart > ctx ||
                             kstart % B != 0;
  const int npages = GRP ? npages_grp : bad ? 0 : (ctx + B - 1) / B - kstart / B;
  const int kp0 = bad ? 0 : kstart / B;  // first page of this kernel's key range
  const int nparts = (bad || GRP) ? 1 : max(1, (npages + a.part_pages - 1) / a.part_pages);
  if (part >= nparts) return;
  __nv_bfloat16 *out_base = a.out + ((size_t)s * a.Hq + (size_t)kvh * G) * D;
  if (bad) {
    if (GRP) {
      if (in_range)
        for (int i = tid; i < ncols * D; i += NW * 32) a.out[row_of(i / D) * D + i % D] = __float2bfloat16(0.f);
    } else
      for (int i = tid; i < G * D; i += NW * 32) out_base[i] = __float2bfloat16(0.f);
    if (tid == 0 && a.err) atomicOr(a.err, PA_DEVERR_CTX);
    return;
  }

  // ---- stage this part's block-table entries; init this warp's barriers
  const int p0 = part * a.part_pages;
  const int np = GRP ? npages : max(0, min(npages - p0, a.part_pages));  // GRP units are never split
  const int32_t *bt_row = a.bt + (size_t)s * a.max_blocks + kp0 + p0;
  // append: the new token's slot, loaded with the table entries (checked
  // once the first gathers are out)
  const bool app_unit = APP && part == nparts - 1 && np > 0;
  const int64_t app_slot = app_unit ? __ldg(a.app_slots + s) : -1;
  for (int i = tid; i < np; i += NW * 32) {
    int pg;
    if constexpr (GRP) {  // shared pages from the first member's row, then each member's own
      int m = -1, lb = kp0 + i;
      if (i >= misc[24]) {
        m = 0;
        while (m + 1 < nm && i >= misc[24 + m + 1]) ++m;
        lb = kshared / B + (i - misc[24 + m]);
      }
      pg = __ldg(a.bt + (size_t)(s + max(m, 0)) * a.max_blocks + lb);
      meta[i] = ((m + 1) << 24) | lb;
    } else {
      pg = __ldg(bt_row + i);
    }
    if (pg < 0 || pg >= a.num_blocks) {
      if (a.err) atomicOr(a.err, PA_DEVERR_PAGE);
      pg = -1;
    }
    tbl[i] = pg;
  }
  uint64_t *my_bars = bars + warp * NST;
  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&my_bars[i], 1);
    fence_mbar_init();
  }
  unit_sync<NW * 32>(bar);

  uint8_t *ring = smem + warp * NST * L::kSlotBytes;
  const int nmine = np > warp ? (np - warp + NW - 1) / NW : 0;
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int i) {  // lane 0: gather local page i of this warp into its slot
    const int pg = tbl[warp + i * NW];
    uint64_t *bar = &my_bars[i % NST];
    uint8_t *slot = ring + (i % NST) * L::kSlotBytes;
    if (pg < 0) {
      mbar_arrive(bar);  // nothing to load; keep the phase sequence intact
      return;
    }
    mbar_arrive_expect_tx(bar, L::kSlotBytes);
    const int row = (pg * a.Hkv + kvh) * B;
    if constexpr (TMA3) {  // both halves in one copy (maps from encode_kv_halves_3d)
      tma_load_3d_hint(slot, tmK, 0, row, 0, bar, pol);
      tma_load_3d_hint(slot + L::kPageBytes, tmV, 0, row, 0, bar, pol);
    } else {
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h)
        tma_load_2d_hint(slot + h * L::kBoxBytes, tmK, h * 64, row, bar, pol);
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h)
        tma_load_2d_hint(slot + L::kPageBytes + h * L::kBoxBytes, tmV, h * 64, row, bar, pol);
    }
  };
  if (lane == 0)
    for (int i = 0; i < NST && i < nmine; ++i) issue(i);

  // ---- append: the part holding the last page owns the new token.  Its slot
  // must be the one of position ctx-1; any other slot (out of the pool or
  // elsewhere in it) is refused, so nothing this launch reads is written.
  // (Checked after the first gathers are issued: the token is written only
  // below, and the streamed copy of its page is patched from the stage.)
  constexpr int kRowChunks = D / 8;  // 16-byte chunks in one K or V row: lane c < 2 kRowChunks moves chunk c
  static_assert(2 * kRowChunks <= 32, "one K and one V row fit a warp's lanes");
  int app_row = -1;                  // the new token's row in the last page, for the warp streaming it
  if (app_unit) {
    const int pg = tbl[np - 1];
    if (app_slot >= 0 && pg >= 0) {
      if (app_slot == (int64_t)pg * B + (ctx - 1) % B) {
        if (warp == (np - 1) % NW) app_row = (ctx - 1) % B;
      } else if (tid == 0 && a.err) {
        atomicOr(a.err, PA_DEVERR_SLOT);
      }
    }
  }

  // ---- Q^T fragments (MMA B operand): head 8nt + lane/4, d pairs
  uint32_t qf[NT][KS][2];
  const __nv_bfloat16 *qb = a.q + ((size_t)s * a.Hq + (size_t)kvh * G) * D;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = nt * 8 + (lane >> 2);
    const __nv_bfloat16 *qg = GRP ? a.q + row_of(g) * D : qb + (size_t)g * D;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int d0 = kk * 16 + 2 * (lane & 3);
      if (g < (GRP ? ncols : G)) {
        qf[nt][kk][0] = __ldg(reinterpret_cast<const uint32_t *>(qg + d0));
        qf[nt][kk][1] = __ldg(reinterpret_cast<const uint32_t *>(qg + d0 + 8));
      } else {
        qf[nt][kk][0] = qf[nt][kk][1] = 0u;
      }
    }
  }

  uint4 *stage = reinterpret_cast<uint4 *>(smem + L::kStageOff);
  if (APP && app_row >= 0) {  // the new token: into its slot, and staged for the patch below
    const size_t src = ((size_t)s * a.Hkv + kvh) * kRowChunks;
    const size_t dst = (((size_t)tbl[np - 1] * a.Hkv + kvh) * B + app_row) * kRowChunks;
    if (lane < 2 * kRowChunks) {
      const bool isv = lane >= kRowChunks;
      const int cc = isv ? lane - kRowChunks : lane;
      const uint4 val = __ldg((isv ? a.app_v : a.app_k) + src + cc);
      stage[lane] = val;
      (isv ? a.vp : a.kp)[dst + cc] = val;
    }
  }

  // A whole context in one CTA after a shared prefix folds the prefix's
  // partial states in at the end: load them now, so that their latency hides
  // under the streaming (thread tid: output elements tid + j NW 32, and the
  // (m, l) of head tid), when a thread's share is small enough for registers.
  constexpr int kPreElems = 4;
  const int npre = (FOLD && has_pre && nparts == 1) ? a.npre : 0;
  // (PRE: the shared-prefix launch; groups of more than 8 heads never qualify)
  const bool pre_early = PRE && NT == 1 && npre > 0 && G * D <= kPreElems * NW * 32;
  const size_t slab = (size_t)a.S * a.Hq;
  float pre_o_r[kPreElems][kMaxPrefixParts], pre_m_r[kMaxPrefixParts], pre_l_r[kMaxPrefixParts];
  if (pre_early) {
#pragma unroll
    for (int j = 0; j < kPreElems; ++j) {
      const int idx = tid + j * NW * 32;
      const size_t row = (size_t)s * a.Hq + (size_t)kvh * G + idx / D;
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p)
        pre_o_r[j][p] = (idx < G * D && p < npre) ? __ldg(a.pre_o + (p * slab + row) * D + idx % D) : 0.f;
    }
    const size_t row = (size_t)s * a.Hq + (size_t)kvh * G + tid;
#pragma unroll
    for (int p = 0; p < kMaxPrefixParts; ++p) {
      pre_m_r[p] = (tid < G && p < npre) ? __ldg(a.pre_ml + 2 * (p * slab + row)) : -INFINITY;
      pre_l_r[p] = (tid < G && p < npre) ? __ldg(a.pre_ml + 2 * (p * slab + row) + 1) : 0.f;
    }
  }

  // Running state.  Lane holds heads 8nt + 2(lane%4) + e (e = 0, 1) and, in o,
  // the O^T rows d = 16dt + lane/4 (+8).
  float m_run[NT][2], l_run[NT][2], o[NT][DT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[nt][dt][0] = o[nt][dt][1] = o[nt][dt][2] = o[nt][dt][3] = 0.f;
  }

  bool timed_out = false;
  int i = 0;
  for (; i < nmine; ++i) {
    const int stg = i % NST;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&my_bars[stg], (uint32_t)((i / NST) & 1)));
    if (!ok) {
      timed_out = true;
      break;
    }
    const int lp = warp + i * NW;
    if (tbl[lp] >= 0) {
      const uint32_t kb = smem_u32(ring + stg * L::kSlotBytes);
      const uint32_t vb = kb + L::kPageBytes;
      // the page's first token; GRP: and its owner (-1: shared by every member) with that member's context
      int tok0 = (kp0 + p0 + lp) * B, owner = -1, octx = ctx;
      if constexpr (GRP) {
        const int mt_ = meta[lp];
        tok0 = (mt_ & 0xffffff) * B;
        owner = (mt_ >> 24) - 1;
        octx = owner >= 0 ? misc[8 + owner] : kshared;
      }
      if (APP && app_row >= 0 && lp == np - 1) {
        // The gather may have seen the slot before or after the store above:
        // overwrite the row with the staged copy (each lane its own chunks).
        uint8_t *slot = ring + stg * L::kSlotBytes;
        if (lane < 2 * kRowChunks) {
          const bool isv = lane >= kRowChunks;
          const int cc = isv ? lane - kRowChunks : lane;
          *reinterpret_cast<uint4 *>(slot + (isv ? L::kPageBytes : 0) + (cc >> 3) * L::kBoxBytes +
                                     sw128(app_row, cc & 7)) = stage[lane];
        }
        __syncwarp();
      }

      // S^T[token][head] = K Q^T
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

      // online softmax: mask tokens past the context, page max.  The running
      // maximum moves only when a column's page maximum passes it by more
      // than kSlack (a factor 2^kSlack): the probabilities are taken against
      // it while the page maxima are still being reduced, and the rescale of
      // the column's state is rare.
      constexpr float kSlack = 8.f;
      float t[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        t[nt][0] = t[nt][1] = -INFINITY;
        // GRP: a member's own page counts only for its columns
        const bool own0 = !GRP || owner < 0 || (nt * 8 + 2 * (lane & 3)) / G == owner;
        const bool own1 = !GRP || owner < 0 || (nt * 8 + 2 * (lane & 3) + 1) / G == owner;
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
      // P (bf16 pairs) against the running maxima; a column that has seen no
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

      // Value rows past the context (the tail of the last page) may hold
      // anything a slot was never written with, NaN included, and 0 * NaN
      // would reach the output: clear them before the product.
      if (tok0 + B > octx) {
        uint8_t *vslot = ring + stg * L::kSlotBytes + L::kPageBytes;
        const int r0 = octx - tok0;
        for (int idx = lane; idx < (B - r0) * L::kHalves * 8; idx += 32) {
          const int row = r0 + idx / (L::kHalves * 8), rem = idx % (L::kHalves * 8);
          *reinterpret_cast<uint4 *>(vslot + (rem >> 3) * L::kBoxBytes + row * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the slot is refilled by TMA afterwards
        __syncwarp();
      }

      // O^T[d][head] += V^T P^T, one 16-token k-tile at a time
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
    __syncwarp();
    if (lane == 0 && i + NST < nmine) {
      fence_proxy_async_smem();
      issue(i + NST);
    }
  }
  if (timed_out) {
    if (lane == 0 && a.err) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    for (int k = i; k < nmine && k < i + NST; ++k) mbar_wait(&my_bars[k % NST], (uint32_t)((k / NST) & 1));
  }

  // ---- per-warp sums across the lanes that share a head
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) l_run[nt][e] += __shfl_xor_sync(0xffffffffu, l_run[nt][e], off);

  // ---- merge the warps (ring memory is reused)
  unit_sync<NW * 32>(bar);
  float *red_o = reinterpret_cast<float *>(smem);
  float *red_m = red_o + NW * 16 * D;
  float *red_l = red_m + NW * 16;
  float *wts = red_l + NW * 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = nt * 8 + 2 * (lane & 3);
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 16 + (lane >> 2);
      red_o[(warp * 16 + g) * D + d] = o[nt][dt][0];
      red_o[(warp * 16 + g + 1) * D + d] = o[nt][dt][1];
      red_o[(warp * 16 + g) * D + d + 8] = o[nt][dt][2];
      red_o[(warp * 16 + g + 1) * D + d + 8] = o[nt][dt][3];
    }
    if (lane < 4) {
      red_m[warp * 16 + g] = m_run[nt][0];
      red_m[warp * 16 + g + 1] = m_run[nt][1];
      red_l[warp * 16 + g] = l_run[nt][0];
      red_l[warp * 16 + g + 1] = l_run[nt][1];
    }
  }
  unit_sync<NW * 32>(bar);

  const bool split = nparts > 1;
  const size_t unit = (size_t)s * a.Hkv + kvh;
  // Whole context in one CTA with a shared prefix before it: per query head,
  // the weight of this CTA's (unnormalised) sum and of each prefix state,
  // both divided by the total weight -- computed once per head, so that every
  // output element only adds up its prefix states (loads issued together).
  float *coef = wts;  // [0..15] this CTA's sum, [16 (p + 1) + g] prefix state p
  if (npre > 0) {
    if (tid < ncols) {
      const int g = tid;
      const size_t row = row_of(g);
      float mx = -INFINITY, l = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red_m[w * 16 + g]);
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) l += red_l[w * 16 + g] * exp2f(red_m[w * 16 + g] - mx);
      }
      float mp[kMaxPrefixParts], lp[kMaxPrefixParts];
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p) {
        mp[p] = pre_early ? pre_m_r[p] : p < npre ? __ldg(a.pre_ml + 2 * (p * slab + row)) : -INFINITY;
        lp[p] = pre_early ? pre_l_r[p] : p < npre ? __ldg(a.pre_ml + 2 * (p * slab + row) + 1) : 0.f;
      }
      float M = l > 0.f ? mx : -INFINITY;
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p)
        if (lp[p] > 0.f) M = fmaxf(M, mp[p]);
      const float c = l > 0.f ? exp2f(mx - M) : 0.f;  // on the sum, whose normaliser is l
      float den = c * l;
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p) {
        lp[p] = lp[p] > 0.f ? lp[p] * exp2f(mp[p] - M) : 0.f;
        den += lp[p];
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      coef[g] = c * inv;
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p) coef[16 * (p + 1) + g] = lp[p] * inv;
    }
    unit_sync<NW * 32>(bar);
  }
  for (int idx = tid, j = 0; idx < ncols * D; idx += NW * 32, ++j) {
    const int g = idx / D, d = idx - g * D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red_m[w * 16 + g]);
    float l = 0.f, acc = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(red_m[w * 16 + g] - mx);
        l += red_l[w * 16 + g] * f;
        acc += red_o[(w * 16 + g) * D + d] * f;
      }
    }
    if (!split) {
      float res;
      if (npre > 0) {  // fold in the shared prefix's partial states
        const size_t row = row_of(g);
        float po[kMaxPrefixParts];
        if (pre_early) {
#pragma unroll
          for (int jj = 0; jj < kPreElems; ++jj)
            if (jj == j)
#pragma unroll
              for (int p = 0; p < kMaxPrefixParts; ++p) po[p] = pre_o_r[jj][p];
        } else {
#pragma unroll
          for (int p = 0; p < kMaxPrefixParts; ++p) po[p] = p < npre ? __ldg(a.pre_o + (p * slab + row) * D + d) : 0.f;
        }
        res = coef[g] * acc;
#pragma unroll
        for (int p = 0; p < kMaxPrefixParts; ++p) res += coef[16 * (p + 1) + g] * po[p];
      } else {
        res = l > 0.f ? acc / l : 0.f;
      }
      if (GRP)
        a.out[row_of(g) * D + d] = __float2bfloat16(res);
      else
        out_base[idx] = __float2bfloat16(res);
    } else {
      const size_t u = (unit * a.max_parts + part) * G + g;
      a.ws_o[u * D + d] = l > 0.f ? acc / l : 0.f;
      if (d == 0) {
        a.ws_ml[2 * u] = mx;
        a.ws_ml[2 * u + 1] = l;
      }
    }
  }
  if (!split) return;

  // ---- split-K: the last part of this (sequence, kv head) merges all parts
  __threadfence();
  unit_sync<NW * 32>(bar);
  if (tid == 0) misc[0] = (arrive_count(a.ws_cnt + unit, a.epoch) == (unsigned int)nparts);
  unit_sync<NW * 32>(bar);
  if (!misc[0]) return;
  __threadfence();
  const size_t ubase = unit * a.max_parts;
  float *wpre = reinterpret_cast<float *>(misc + 8);  // [npre][16] prefix weights (histogram area, free now)
  if (tid < G) {
    const int g = tid;
    const size_t row = (size_t)s * a.Hq + (size_t)kvh * G + g;
    const int npre = (PRE && has_pre) ? a.npre : 0;
    float M = -INFINITY;
    for (int p = 0; p < npre; ++p) {
      const float lp = __ldg(a.pre_ml + 2 * (p * slab + row) + 1);
      if (lp > 0.f) M = fmaxf(M, __ldg(a.pre_ml + 2 * (p * slab + row)));
    }
    for (int p = 0; p < nparts; ++p) {
      const float l = __ldcg(a.ws_ml + 2 * ((ubase + p) * G + g) + 1);
      if (l > 0.f) M = fmaxf(M, __ldcg(a.ws_ml + 2 * ((ubase + p) * G + g)));
    }
    float den = 0.f;
    for (int p = 0; p < nparts; ++p) {
      const float m = __ldcg(a.ws_ml + 2 * ((ubase + p) * G + g));
      const float l = __ldcg(a.ws_ml + 2 * ((ubase + p) * G + g) + 1);
      const float w = l > 0.f ? l * exp2f(m - M) : 0.f;
      wts[p * 16 + g] = w;
      den += w;
    }
    for (int p = 0; p < npre; ++p) {
      const float lp = __ldg(a.pre_ml + 2 * (p * slab + row) + 1);
      const float w = lp > 0.f ? lp * exp2f(__ldg(a.pre_ml + 2 * (p * slab + row)) - M) : 0.f;
      wpre[p * 16 + g] = w;
      den += w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int p = 0; p < nparts; ++p) wts[p * 16 + g] *= inv;
    for (int p = 0; p < npre; ++p) wpre[p * 16 + g] *= inv;
  }
  unit_sync<NW * 32>(bar);
  for (int idx = tid; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float acc = 0.f;
    for (int p = 0; p < nparts; ++p) acc += wts[p * 16 + g] * __ldcg(a.ws_o + ((ubase + p) * G + g) * D + d);
    if (PRE && has_pre)
      for (int p = 0; p < a.npre; ++p)
        acc += wpre[p * 16 + g] * __ldg(a.pre_o + (p * slab + (size_t)s * a.Hq + (size_t)kvh * G + g) * D + d);
    out_base[idx] = __float2bfloat16(acc);
  }
  if (tid == 0) a.ws_cnt[unit] = 0ull;
}

// Host: the argument block of a decode launch over a validated desc with
// split plan `plan` (no shared prefix, no append; the caller sets those).
// Longest-first order pays when the units fill a few waves of the `slots`
// resident units: in one wave there is no order to choose, and with many
// short units greedy dispatch already balances while every unit would still
// pay ~1.4 us for its rank (measured: 1.7 units a slot 50.7 vs 59.2 us, 4.2 a
// slot 283 vs 291 us, 6.7 a slot 99 vs 89 us, one wave 4.6 vs 3.6 us).
// PA_DECODE_LPT=0 / 1 in the environment forces it off / on.
inline void fill_decode_args(DecodeArgs *a, const pa_decode_desc *d, const DecodePlan &plan, const void *q,
                             const int32_t *block_tables, const int32_t *context_lens, void *out, void *workspace,
                             int32_t *err_flag, long long slots) {
  *a = DecodeArgs{};
  a->q = static_cast<const __nv_bfloat16 *>(q);
  a->bt = block_tables;
  a->ctx = context_lens;
  a->out = static_cast<__nv_bfloat16 *>(out);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a->ws_o = plan.total() ? reinterpret_cast<float *>(ws) : nullptr;
  a->ws_ml = plan.total() ? reinterpret_cast<float *>(ws + plan.ws_o_bytes) : nullptr;
  a->ws_cnt = plan.total() ? reinterpret_cast<unsigned long long *>(ws + plan.ws_o_bytes + plan.ws_ml_bytes)
                           : nullptr;
  a->epoch = next_decode_epoch();
  const long long units = (long long)d->num_seqs * d->num_kv_heads * plan.max_parts;
  a->lpt = units > slots && units <= 5 * slots;
  const char *env = getenv("PA_DECODE_LPT");
  if (env && (env[0] == '0' || env[0] == '1')) a->lpt = env[0] - '0';
  a->err = err_flag;
  a->S = d->num_seqs;
  a->Hq = d->num_q_heads;
  a->Hkv = d->num_kv_heads;
  a->G = d->num_q_heads / d->num_kv_heads;
  a->num_blocks = d->num_blocks;
  a->max_blocks = d->max_blocks_per_seq;
  a->max_ctx = d->max_context_len;
  a->part_pages = plan.part_pages;
  a->max_parts = plan.max_parts;
  a->scale_log2 = d->scale * 1.4426950408889634f;
}

}  // namespace
}  // namespace pa
