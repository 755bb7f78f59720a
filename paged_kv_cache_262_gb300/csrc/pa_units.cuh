// Decode units of the shared-prefix decode (sm_103a): a unit is one
// (sub-group, kv head) -- the sub-group's keys past its group prefix, shared
// by every member, then each member's own keys.  Shared by the task-queue
// decode (pa_decode_tasks.cu) and the wide-group decode (pa_decode_wide.cu).
#pragma once

#include "pa_internal.h"

namespace pa {
namespace {

// Most pages a unit may hold (shared plus every member's own).
constexpr int kUnitMaxPages = 512;

struct UnitShape {
  int S, G, rows, max_blocks, max_ctx, ngroups;
};

// Sub-group of sequences s0 .. s1-1 whose members share keys 0 .. kshared-1
// (-1: a sequence alone, sharing only its group prefix): its group prefix
// (the unit's first key) and its page count past that prefix (-1: invalid --
// members outside the batch, more query rows than the launch takes, a shared
// length that is not whole blocks or past a member's context, a bad context,
// or more than kUnitMaxPages pages).  One thread; contexts and the prefix
// groups through the accessors (shared or global memory).
template <class Ctx, class Gs, class Gp>
__device__ void subgroup_plan(const UnitShape &u, int B, int s0, int s1, int kshared, Ctx ctx_at, Gs gstart_at,
                              Gp gprefix_at, int *kstart_out, int *pages_out) {
  const int nm = s1 - s0;
  int kstart = 0;
  if (u.ngroups > 0 && s0 >= 0 && s0 < u.S && s0 >= gstart_at(0) && s0 < gstart_at(u.ngroups)) {
    int lo = 0, hi = u.ngroups;  // grp_start[lo] <= s0 < grp_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (gstart_at(mid) <= s0) lo = mid;
      else hi = mid;
    }
    kstart = gprefix_at(lo);
  }
  if (kshared < 0) kshared = kstart;
  bool ok = s0 >= 0 && nm > 0 && s1 <= u.S && nm * u.G <= u.rows && kstart >= 0 && kshared >= kstart &&
            kshared % B == 0 && kstart % B == 0;
  int own = 0;
  int c[16];  // a valid sub-group has at most 16 members (16 query rows); loads issued together
#pragma unroll
  for (int m = 0; m < 16; ++m) c[m] = ok && m < nm ? ctx_at(s0 + m) : 0;
#pragma unroll
  for (int m = 0; m < 16; ++m)
    if (m < nm) {
      ok = ok && c[m] >= kshared && c[m] > 0 && c[m] <= u.max_blocks * B && c[m] <= u.max_ctx;
      own += (c[m] + B - 1) / B - kshared / B;
    }
  const int n = (kshared - kstart) / B + own;
  *kstart_out = kstart;
  *pages_out = ok && n <= kUnitMaxPages ? n : -1;
}

// The same plan for one sub-group on a whole warp (lane 0 reads the
// sub-group's bounds and group prefix, lanes < 16 its members' contexts):
// returns the page count (-1: invalid) and sets the first sequence, member
// count, group prefix and shared length.  Every lane gets the same values.
__device__ __forceinline__ int subgroup_plan_warp(const UnitShape &u, int B, int sg, const int32_t *sub_start,
                                                  const int32_t *sub_shared, const int32_t *grp_start,
                                                  const int32_t *grp_prefix, const int32_t *ctx, int *s0_out,
                                                  int *nm_out, int *kstart_out, int *kshared_out) {
  const int lane = threadIdx.x & 31;
  int s0 = 0, s1 = 0, ksh = -1, kstart = 0;
  if (lane == 0) {
    s0 = sub_start ? __ldg(sub_start + sg) : sg;
    s1 = sub_start ? __ldg(sub_start + sg + 1) : sg + 1;
    ksh = sub_start ? __ldg(sub_shared + sg) : -1;
    if (u.ngroups > 0 && s0 >= 0 && s0 < u.S && s0 >= __ldg(grp_start) && s0 < __ldg(grp_start + u.ngroups)) {
      int lo = 0, hi = u.ngroups;  // grp_start[lo] <= s0 < grp_start[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(grp_start + mid) <= s0) lo = mid;
        else hi = mid;
      }
      kstart = __ldg(grp_prefix + lo);
    }
  }
  s0 = __shfl_sync(0xffffffffu, s0, 0);
  s1 = __shfl_sync(0xffffffffu, s1, 0);
  ksh = __shfl_sync(0xffffffffu, ksh, 0);
  kstart = __shfl_sync(0xffffffffu, kstart, 0);
  if (ksh < 0) ksh = kstart;
  const int nm = s1 - s0;
  bool ok = s0 >= 0 && nm > 0 && s1 <= u.S && nm * u.G <= u.rows && kstart >= 0 && ksh >= kstart &&
            ksh % B == 0 && kstart % B == 0;
  const int c = (ok && lane < nm) ? __ldg(ctx + s0 + lane) : 0;
  const bool mine = lane >= nm || (c >= ksh && c > 0 && c <= u.max_blocks * B && c <= u.max_ctx);
  ok = __all_sync(0xffffffffu, mine) && ok;
  int own = (ok && lane < nm) ? (c + B - 1) / B - ksh / B : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) own += __shfl_xor_sync(0xffffffffu, own, off);
  const int n = (ksh - kstart) / B + own;
  *s0_out = s0;
  *nm_out = nm;
  *kstart_out = kstart;
  *kshared_out = ksh;
  return ok && n <= kUnitMaxPages ? n : -1;
}

}  // namespace
}  // namespace pa
