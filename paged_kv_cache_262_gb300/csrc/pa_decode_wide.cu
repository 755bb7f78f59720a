// Wide-group paged decode on the tcgen05 tensor cores, for sm_103a.
//
// A decode unit whose query rows are many -- the samples of one prompt as a
// sub-group ("Configuring vLLM and PagedAttention for High Throughput
// Enterprise LLM Serving", "Zero-Copy Prefix Caching & Shared Sampling"),
// or a wide GQA group -- does two dense contractions per key: 16 rows x 128
// dims for the scores, 16 x 128 for the values.  On warp MMAs (m16n8k16)
// those take as long as the page takes to arrive from HBM, so such units are
// bound by the warp-MMA rate instead of by the cache reads that decode is
// about ("Memory Bottlenecks in Autoregressive LLM Inference").  Here they run
// on the 5th-generation tensor cores with the tokens as the MMA M side:
//  * key tile = 128 tokens (8 pages of 16 or 4 of 32), gathered by 2-D TMA
//    exactly as the prefill gathers its key tiles (K and V, 128-byte swizzle,
//    L2 evict-first), into a ring of kWStages tiles;
//  * S^T[token][row] = K Q^T: A = the K tile (K-major), B = the unit's Q rows
//    (16 rows x 128, K-major, in shared memory), D in TMEM (lane = token);
//  * the softmax runs over the tokens (TMEM lanes) of each row: per tile the
//    row maxima of the four warps (redux.sync on order-preserving integers)
//    are exchanged in shared memory, then probabilities in fp32 (base 2),
//    rounded to bf16 once for both the product and the running sum;
//  * O^T[d][row] = V^T P^T: A = the V tile read MN-major (the layout TMA gave
//    it), B = P^T written by the softmax threads to shared memory, D into a
//    fresh TMEM tile (lane = d) that the same threads fold into their
//    registers one tile later (O = O * 2^(m_old - m_new) + P V);
//  * warp-specialised and persistent: warp 8 takes units from a global
//    counter, loads each unit's Q rows and gathers its tiles; warp 9 issues
//    the MMAs (S of the next tile before P V of this one, across units); two
//    softmax warpgroups (warps 0-3 and 4-7) take a unit's tiles in turn, each
//    with its own running softmax state, and at the unit's end the second
//    hands its state to the first, which merges them with the group prefix's
//    partial states and stores the bf16 rows.  The rings run across units,
//    so a unit's start and end hide under the next one's gathers;
//  * a unit (sub-group, kv head) reads the sub-group's shared keys past its
//    group prefix once for all members' rows, then each member's own keys,
//    masked for the other members' rows;
//  * every wait is bounded (mbarriers only, no named barriers); a timeout
//    sets PA_DEVERR_TIMEOUT and every role leaves.
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

constexpr int kWD = 128;              // head_dim
constexpr int kWTok = 128;            // tokens per key tile: the MMA M side of S^T
constexpr int kWRows = 16;            // query rows of a unit: the MMA N side
constexpr int kWStages = 3;           // key tiles in flight per CTA
constexpr int kWThreads = 320;        // warps 0-7 two softmax warpgroups, 8 producer, 9 MMA issuer
constexpr int kWHalf = 16384;         // one 64-column half of a 128 x 128 bf16 tile
constexpr int kWTile = 32768;         // 128 x 128 bf16
constexpr int kWRowTile = 4096;       // 16 rows x 128 bf16: two 64-column halves of 2 KB
constexpr uint32_t kWTmemCols = 128;  // warpgroup g: S^T at 64g + [0, 32) (two buffers), P V at 64g + [32, 64)

struct WideArgs {
  const __nv_bfloat16 *q;
  const int32_t *bt;
  const int32_t *ctx;
  __nv_bfloat16 *out;
  const int32_t *sub_start;  // null: every sequence is a unit of one member
  const int32_t *sub_shared;
  int nsg;
  const int32_t *grp_start;
  const int32_t *grp_prefix;
  int ngroups;
  const float *pre_o;  // [npre][S][Hq][D]
  const float *pre_ml; // [npre][S][Hq][2]
  int npre;
  unsigned int *ctr;   // units handed out (zeroed before the launch)
  int32_t *err;
  int S, Hq, Hkv, G, rows, num_blocks, max_blocks, max_ctx;
  float scale_log2;
};

// Barriers (one mbarrier each): K/V tile landed / free; per softmax
// warpgroup: S^T ready / read, P^T written / read, P V tile ready / read,
// tile maxima and row sums exchanged among its 128 threads; Q rows loaded /
// done with; unit descriptor posted / done with; the second warpgroup's
// state handed over / taken; the first warpgroup's fold weights; every MMA
// complete.
enum {
  WB_FULL = 0,
  WB_EMPTY = WB_FULL + kWStages,
  WB_SFULL = WB_EMPTY + kWStages,  // [g][2]
  WB_SEMPTY = WB_SFULL + 4,        // [g][2]
  WB_PFULL = WB_SEMPTY + 4,        // [g]
  WB_PEMPTY = WB_PFULL + 2,        // [g]
  WB_OFULL = WB_PEMPTY + 2,        // [g][2]
  WB_OEMPTY = WB_OFULL + 4,        // [g][2]
  WB_MAX = WB_OEMPTY + 4,          // [g][2]
  WB_RED = WB_MAX + 4,             // [g][2]
  WB_QFULL = WB_RED + 4,
  WB_QEMPTY = WB_QFULL + 2,
  WB_UFULL = WB_QEMPTY + 2,
  WB_UEMPTY = WB_UFULL + 2,
  WB_XCH = WB_UEMPTY + 2,
  WB_XDONE = WB_XCH + 1,
  WB_WTS = WB_XDONE + 1,
  WB_DONE = WB_WTS + 1,
  WB_COUNT = WB_DONE + 1
};

template <int B>
struct WideSmem {
  static constexpr int kPages = kWTok / B;
  static constexpr int kStage = 2 * kWTile;                            // K tile then V tile
  static constexpr int kOffQ = kWStages * kStage;                      // [2] Q^T tiles
  static constexpr int kOffP = kOffQ + 2 * kWRowTile;                  // [g] P^T tiles
  static constexpr int kOffX = kOffP + 2 * kWRowTile;                  // [16][128] fp32: warpgroup 1's O
  static constexpr int kOffMeta = kOffX + kWRows * kWD * 4;            // [stage][page] first token, owner, bound
  static constexpr int kOffUnit = kOffMeta + kWStages * kPages * 3 * 4;  // [2][16] unit descriptors
  static constexpr int kOffMax = kOffUnit + 2 * 16 * 4;                // [g][2][4 warps][16] tile maxima
  static constexpr int kOffRed = kOffMax + 2 * 2 * 4 * 16 * 4;         // [g][2][4 warps][16] row sums
  static constexpr int kOffXml = kOffRed + 2 * 2 * 4 * 16 * 4;         // [16] m, [16] l of warpgroup 1
  static constexpr int kOffWts = kOffXml + 2 * 16 * 4;                 // [16][2 + kMaxPrefixParts] weights
  static constexpr int kOffBar = (kOffWts + 16 * (2 + kMaxPrefixParts) * 4 + 7) & ~7;
  static constexpr int kOffMisc = kOffBar + WB_COUNT * 8;  // TMEM address, dead flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// float <-> int with the same order (for redux.sync.max over scores)
__device__ __forceinline__ int ord_of(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float float_of_ord(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

constexpr uint32_t kIdS = umma_idesc_bf16(128, kWRows, false, false);   // K tile x Q^T, both K-major
constexpr uint32_t kIdPV = umma_idesc_bf16(128, kWRows, true, false);   // V^T (MN-major) x P^T

template <int B>
__global__ void __launch_bounds__(kWThreads, 1)
    decode_wide_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const WideArgs a) {
  using L = WideSmem<B>;
  constexpr int P = L::kPages;
  constexpr int kW = 2 + kMaxPrefixParts;  // fold weights of a row: own two states, then the prefix's ranges
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *dead = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  int *meta = reinterpret_cast<int *>(smem + L::kOffMeta);
  int *udesc = reinterpret_cast<int *>(smem + L::kOffUnit);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(&bars[WB_FULL + i], 1);
      mbar_init(&bars[WB_EMPTY + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[WB_SFULL + i], 1);
      mbar_init(&bars[WB_SEMPTY + i], 128);
      mbar_init(&bars[WB_OFULL + i], 1);
      mbar_init(&bars[WB_OEMPTY + i], 128);
      mbar_init(&bars[WB_MAX + i], 128);
      mbar_init(&bars[WB_RED + i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[WB_PFULL + i], 128);
      mbar_init(&bars[WB_PEMPTY + i], 1);
      mbar_init(&bars[WB_QFULL + i], 1);
      mbar_init(&bars[WB_QEMPTY + i], 1);
      mbar_init(&bars[WB_UFULL + i], 1);
      mbar_init(&bars[WB_UEMPTY + i], 257);
    }
    mbar_init(&bars[WB_XCH], 128);
    mbar_init(&bars[WB_XDONE], 128);
    mbar_init(&bars[WB_WTS], 128);
    mbar_init(&bars[WB_DONE], 1);
    *dead = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tslot, kWTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto fail = [&]() {
    *dead = 1;
    if (a.err) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  };
  // bounded wait, uniform over the warp (warp collectives follow the waits)
  auto wait_warp = [&](int b, uint32_t parity) -> bool {
    bool r = !*dead;
    if (r && !mbar_wait(&bars[b], parity)) {
      fail();
      r = false;
    }
    return __all_sync(0xffffffffu, r);
  };
  const int G = a.G;
  const int nunits = a.nsg * a.Hkv;
  const UnitShape us{a.S, a.G, a.rows, a.max_blocks, a.max_ctx, a.ngroups};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int u = 0, j = 0;
    bool ok = true;
    while (ok) {
      int t = 0;
      if (lane == 0) t = (int)atomicAdd(a.ctr, 1u);
      t = __shfl_sync(0xffffffffu, t, 0);
      const int ub = u & 1;
      if (u >= 2 && !wait_warp(WB_UEMPTY + ub, (uint32_t)(((u >> 1) - 1) & 1))) break;
      int *ud = udesc + ub * 16;
      if (t >= nunits) {  // nothing left: tell the other roles
        if (lane == 0) {
          ud[0] = 1;
          mbar_arrive(&bars[WB_UFULL + ub]);
        }
        break;
      }
      const int sg = t / a.Hkv, kvh = t - sg * a.Hkv;
      int s0, nm, kstart, kshared;
      const int n = subgroup_plan_warp(us, B, sg, a.sub_start, a.sub_shared, a.grp_start, a.grp_prefix, a.ctx, &s0,
                                       &nm, &kstart, &kshared);
      const int ntiles = n < 0 ? 0 : (n + P - 1) / P;
      const int ncols = n < 0 ? 0 : nm * G;
      // the unit's Q rows (member g / G, head g % G), rows past the unit zero
      const int qb = u & 1;
      if (u >= 2 && !wait_warp(WB_QEMPTY + qb, (uint32_t)(((u >> 1) - 1) & 1))) break;
      uint8_t *qd = smem + L::kOffQ + qb * kWRowTile;
#pragma unroll
      for (int k = 0; k < kWRows * 16 / 32; ++k) {
        const int i = k * 32 + lane, r = i >> 4, c = i & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < ncols)
          v = __ldg(reinterpret_cast<const uint4 *>(a.q + ((size_t)(s0 + r / G) * a.Hq + (size_t)kvh * G + r % G) * kWD) +
                    c);
        *reinterpret_cast<uint4 *>(qd + (c >> 3) * 2048 + sw128(r, c & 7)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ud[0] = 0;
        ud[1] = sg;
        ud[2] = kvh;
        ud[3] = s0;
        ud[4] = nm;
        ud[5] = kstart;
        ud[6] = kshared;
        ud[7] = n;
        ud[8] = ntiles;
        mbar_arrive(&bars[WB_QFULL + qb]);
        mbar_arrive(&bars[WB_UFULL + ub]);
      }
      // members' contexts and the end of each member's own pages (after the shared ones)
      const int c = (n >= 0 && lane < nm) ? __ldg(a.ctx + s0 + lane) : 0;
      const int own = (n >= 0 && lane < nm) ? (c + B - 1) / B - kshared / B : 0;
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int shared_pages = n >= 0 ? (kshared - kstart) / B : 0;
      for (int tt = 0; tt < ntiles; ++tt, ++j) {
        const int stage = j % kWStages;
        if (j >= kWStages && !wait_warp(WB_EMPTY + stage, (uint32_t)(((j / kWStages) - 1) & 1))) {
          ok = false;
          break;
        }
        // page `lane` of the tile: its id, first token, owner and the context bounding its keys
        const int i = tt * P + lane;
        int m = -1, lb = kstart / B + i;
        for (int mm = 0; mm < nm; ++mm) {
          const int e = __shfl_sync(0xffffffffu, incl, mm), o = __shfl_sync(0xffffffffu, own, mm);
          if (i >= shared_pages && m < 0 && i < shared_pages + e) {
            m = mm;
            lb = kshared / B + (i - (shared_pages + e - o));
          }
        }
        const int cm = __shfl_sync(0xffffffffu, c, max(m, 0));
        int pg = -1;
        if (lane < P && i < n) {
          pg = __ldg(a.bt + (size_t)(s0 + max(m, 0)) * a.max_blocks + lb);
          if (pg < 0 || pg >= a.num_blocks) {
            if (a.err) atomicOr(a.err, PA_DEVERR_PAGE);
            pg = -1;
          }
        }
        if (lane < P) {
          int *mt = meta + (stage * P + lane) * 3;
          mt[0] = lb * B;
          mt[1] = m;
          mt[2] = pg >= 0 ? (m >= 0 ? cm : kshared) : -1;  // no tokens of a missing page count
        }
        const unsigned have = __ballot_sync(0xffffffffu, pg >= 0);
        __syncwarp();
        if (lane == 0) {
          if (have)
            mbar_arrive_expect_tx(&bars[WB_FULL + stage], (uint32_t)__popc(have) * 2u * B * 256u);
          else
            mbar_arrive(&bars[WB_FULL + stage]);
        }
        __syncwarp();
        if (pg >= 0) {
          uint8_t *kd = smem + stage * L::kStage + lane * B * 128;
          const int row = (pg * a.Hkv + kvh) * B;
          tma_load_2d_hint(kd, &tmK, 0, row, &bars[WB_FULL + stage], pol);
          tma_load_2d_hint(kd + kWHalf, &tmK, 64, row, &bars[WB_FULL + stage], pol);
          tma_load_2d_hint(kd + kWTile, &tmV, 0, row, &bars[WB_FULL + stage], pol);
          tma_load_2d_hint(kd + kWTile + kWHalf, &tmV, 64, row, &bars[WB_FULL + stage], pol);
        }
      }
      ++u;
    }
    // copies still in flight land before the CTA leaves
    for (int jj = j - kWStages < 0 ? 0 : j - kWStages; jj < j; ++jj)
      mbar_wait(&bars[WB_FULL + jj % kWStages], (uint32_t)((jj / kWStages) & 1));
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto wait = [&](int b, uint32_t parity) -> bool {
        if (*dead) return false;
        if (mbar_wait(&bars[b], parity)) return true;
        fail();
        return false;
      };
      int u = 0, j = 0, jg0 = 0, jg1 = 0;  // tiles so far: all, and of each softmax warpgroup
      bool ok = true;
      while (ok) {
        const int ub = u & 1;
        if (!wait(WB_UFULL + ub, (uint32_t)((u >> 1) & 1))) break;
        const int *ud = udesc + ub * 16;
        if (ud[0] == 1) break;
        const int ntiles = ud[8];
        const int qb = u & 1;
        if (!wait(WB_QFULL + qb, (uint32_t)((u >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t qaddr = smem_u32(smem + L::kOffQ + qb * kWRowTile);
        // S^T of the unit's tile tt (global tile jj) into its warpgroup's buffer
        auto issue_s = [&](int tt, int jj) -> bool {
          const int g = tt & 1, lj = (g ? jg1 : jg0) + (tt >> 1), sb = lj & 1, stage = jj % kWStages;
          if (!wait(WB_FULL + stage, (uint32_t)((jj / kWStages) & 1))) return false;
          if (lj >= 2 && !wait(WB_SEMPTY + 2 * g + sb, (uint32_t)(((lj >> 1) - 1) & 1))) return false;
          tc_fence_after();
          const uint32_t kb = smem_u32(smem + stage * L::kStage);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * kWHalf + (kk & 3) * 32, qoff = (kk >> 2) * 2048 + (kk & 3) * 32;
            umma_bf16(tmem + 64 * g + sb * kWRows, umma_desc_sw128(kb + koff, 16, 1024),
                      umma_desc_sw128(qaddr + qoff, 16, 1024), kIdS, kk > 0);
          }
          umma_commit(&bars[WB_SFULL + 2 * g + sb]);
          return true;
        };
        if (ntiles > 0) ok = issue_s(0, j);
        for (int tt = 0; ok && tt < ntiles; ++tt) {
          if (tt + 1 < ntiles && !(ok = issue_s(tt + 1, j + tt + 1))) break;
          const int g = tt & 1, lj = (g ? jg1 : jg0) + (tt >> 1), ob = lj & 1, stage = (j + tt) % kWStages;
          if (!wait(WB_PFULL + g, (uint32_t)(lj & 1)) ||
              (lj >= 2 && !wait(WB_OEMPTY + 2 * g + ob, (uint32_t)(((lj >> 1) - 1) & 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = smem_u32(smem + stage * L::kStage + kWTile);
          const uint32_t pb = smem_u32(smem + L::kOffP + g * kWRowTile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(tmem + 64 * g + 2 * kWRows + ob * kWRows, umma_desc_sw128(vb + kk * 2048, kWHalf, 1024),
                      umma_desc_sw128(pb + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024), kIdPV, kk > 0);
          umma_commit(&bars[WB_EMPTY + stage]);
          umma_commit(&bars[WB_PEMPTY + g]);
          umma_commit(&bars[WB_OFULL + 2 * g + ob]);
        }
        if (!ok) break;
        j += ntiles;
        jg0 += (ntiles + 1) >> 1;
        jg1 += ntiles >> 1;
        umma_commit(&bars[WB_QEMPTY + qb]);
        mbar_arrive(&bars[WB_UEMPTY + ub]);
        ++u;
      }
      umma_commit(&bars[WB_DONE]);
      mbar_wait(&bars[WB_DONE], 0);  // every MMA complete before TMEM is freed
    }
  } else {
    // ------------------------------ softmax warpgroups, fold and units' ends
    const int g = warp >> 2, wq = warp & 3;  // warpgroup, its warp (TMEM lane quarter)
    const int t = tid & 127;                 // token of a key tile; d of the P V tiles
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16) + 64 * g;
    float *smax = reinterpret_cast<float *>(smem + L::kOffMax) + g * 128;
    float *sred_g = reinterpret_cast<float *>(smem + L::kOffRed) + g * 128;
    float *xo = reinterpret_cast<float *>(smem + L::kOffX);
    float *xml = reinterpret_cast<float *>(smem + L::kOffXml);
    float *wts = reinterpret_cast<float *>(smem + L::kOffWts);
    uint8_t *pbase = smem + L::kOffP + g * kWRowTile + (t >> 6) * 2048 + (t & 7) * 2;
    const size_t slab = (size_t)a.S * a.Hq;
    bool prefix_visible = false;
    int u = 0, j = 0, lj = 0;  // units, tiles of the CTA, tiles of this warpgroup
    bool ok = true;
    while (ok) {
      const int ub = u & 1;
      if (!wait_warp(WB_UFULL + ub, (uint32_t)((u >> 1) & 1))) break;
      const int *ud = udesc + ub * 16;
      if (ud[0] == 1) break;
      const int kvh = ud[2], s0 = ud[3], nm = ud[4], kstart = ud[5], n = ud[7], ntiles = ud[8];
      const int ncols = n < 0 ? 0 : nm * G;
      const unsigned colmask = (1u << ncols) - 1u;
      float mrun[kWRows], lsum[kWRows], oreg[kWRows], aprev[kWRows];
#pragma unroll
      for (int r = 0; r < kWRows; ++r) {
        mrun[r] = -INFINITY;
        lsum[r] = 0.f;
        oreg[r] = 0.f;
        aprev[r] = 1.f;
      }
      // O = O 2^(m_old - m_new) + P V of this warpgroup's tile lt (its factors in aprev)
      auto fold = [&](int lt) -> bool {
        const int ob = lt & 1;
        if (!wait_warp(WB_OFULL + 2 * g + ob, (uint32_t)((lt >> 1) & 1))) return false;
        tc_fence_after();
        uint32_t ov[kWRows];
        tmem_ld16(lane_base + 2 * kWRows + ob * kWRows, ov);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[WB_OEMPTY + 2 * g + ob]);
#pragma unroll
        for (int r = 0; r < kWRows; ++r) oreg[r] = oreg[r] * aprev[r] + __uint_as_float(ov[r]);
        return true;
      };
      int mine = 0;  // tiles of this unit taken by this warpgroup
      for (int tt = g; tt < ntiles; tt += 2, ++lj, ++mine) {
        const int jj = j + tt, stage = jj % kWStages, sb = lj & 1;
        if (!wait_warp(WB_FULL + stage, (uint32_t)((jj / kWStages) & 1)) ||
            !wait_warp(WB_SFULL + 2 * g + sb, (uint32_t)((lj >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[kWRows];
        tmem_ld16(lane_base + sb * kWRows, sv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[WB_SEMPTY + 2 * g + sb]);
        // this thread's token: the rows it counts for (a member's own page only for that member's rows)
        const int *mt = meta + (stage * P + t / B) * 3;
        const int tok = mt[0] + t % B, owner = mt[1], octx = mt[2];
        const bool tvalid = tok < octx;
        const unsigned vmask =
            tvalid ? (owner < 0 ? colmask : (((1u << G) - 1u) << (owner * G)) & colmask) : 0u;
        float s[kWRows];
        int pick = 0;  // lane r keeps row r's warp maximum
#pragma unroll
        for (int r = 0; r < kWRows; ++r) {
          s[r] = (vmask >> r) & 1u ? __uint_as_float(sv[r]) * a.scale_log2 : -INFINITY;
          const int o = __reduce_max_sync(0xffffffffu, ord_of(s[r]));
          pick = lane == r ? o : pick;
        }
        // tile maxima of the rows over the warpgroup's four warps
        float *mx = smax + sb * 64;
        if (lane < kWRows) mx[wq * 16 + lane] = float_of_ord(pick);
        mbar_arrive(&bars[WB_MAX + 2 * g + sb]);
        if (!wait_warp(WB_MAX + 2 * g + sb, (uint32_t)((lj >> 1) & 1))) {
          ok = false;
          break;
        }
        float tmx[kWRows];
#pragma unroll
        for (int q4 = 0; q4 < kWRows / 4; ++q4) {
          const float4 a0 = reinterpret_cast<const float4 *>(mx)[q4], a1 = reinterpret_cast<const float4 *>(mx + 16)[q4];
          const float4 a2 = reinterpret_cast<const float4 *>(mx + 32)[q4], a3 = reinterpret_cast<const float4 *>(mx + 48)[q4];
          tmx[4 * q4] = fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x));
          tmx[4 * q4 + 1] = fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y));
          tmx[4 * q4 + 2] = fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z));
          tmx[4 * q4 + 3] = fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w));
        }
        float alpha[kWRows];
        uint32_t pbits[kWRows];
#pragma unroll
        for (int r = 0; r < kWRows; ++r) {
          const float mn = fmaxf(mrun[r], tmx[r]);
          alpha[r] = mn == -INFINITY ? 1.f : ex2_ftz(mrun[r] - mn);
          const __nv_bfloat16 pb = __float2bfloat16((vmask >> r) & 1u ? ex2_ftz(s[r] - mn) : 0.f);
          lsum[r] = lsum[r] * alpha[r] + __bfloat162float(pb);
          pbits[r] = (uint32_t)__bfloat16_as_ushort(pb);
          mrun[r] = mn;
        }
        // value rows of tokens that count for no row may hold any bits
        // (NaN included) and would meet a zero probability: clear them
        if (!tvalid) {
          uint8_t *vd = smem + stage * L::kStage + kWTile + t * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4 *>(vd + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(vd + kWHalf + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        // P^T tile: row r, token t (K-major, 128-byte swizzle)
        if (lj >= 1 && !wait_warp(WB_PEMPTY + g, (uint32_t)((lj - 1) & 1))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int r = 0; r < kWRows; ++r)
          *reinterpret_cast<uint16_t *>(pbase + sw128(r, (t & 63) >> 3)) = (uint16_t)pbits[r];
        fence_proxy_async_smem();
        mbar_arrive(&bars[WB_PFULL + g]);
        if (mine > 0 && !fold(lj - 1)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int r = 0; r < kWRows; ++r) aprev[r] = alpha[r];
      }
      if (!ok) break;
      if (mine > 0 && !fold(lj - 1)) break;
      j += ntiles;

      // ---- the unit's end: this warpgroup's row sums over its 128 token lanes
#pragma unroll
      for (int r = 0; r < kWRows; ++r) {
        float v = lsum[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        lsum[r] = v;
      }
      float *sred = sred_g + (u & 1) * 64;
      if (lane < kWRows) {
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < kWRows; ++r) v = lane == r ? lsum[r] : v;
        sred[wq * 16 + lane] = v;
      }
      mbar_arrive(&bars[WB_RED + 2 * g + (u & 1)]);
      if (!wait_warp(WB_RED + 2 * g + (u & 1), (uint32_t)((u >> 1) & 1))) break;
      float lrow[kWRows];
#pragma unroll
      for (int r = 0; r < kWRows; ++r) lrow[r] = sred[r] + sred[16 + r] + sred[32 + r] + sred[48 + r];
      if (g == 1) {
        // hand this warpgroup's state to the first: its O (d = t) and the rows' m and l
        if (u >= 1 && !wait_warp(WB_XDONE, (uint32_t)((u - 1) & 1))) break;
#pragma unroll
        for (int r = 0; r < kWRows; ++r) xo[r * kWD + t] = oreg[r];
        if (t < kWRows) {
          float mv = 0.f, lv = 0.f;
#pragma unroll
          for (int r = 0; r < kWRows; ++r) {
            mv = t == r ? mrun[r] : mv;
            lv = t == r ? lrow[r] : lv;
          }
          xml[t] = mv;
          xml[16 + t] = lv;
        }
        mbar_arrive(&bars[WB_XCH]);
      } else {
        if (!wait_warp(WB_XCH, (uint32_t)(u & 1))) break;
        const int npre = (kstart > 0 && n >= 0) ? a.npre : 0;
        if (npre > 0 && !prefix_visible) {
          asm volatile("griddepcontrol.wait;" ::: "memory");  // the prefix pass (this grid's predecessor) is complete
          prefix_visible = true;
        }
        if (t < ncols) {  // thread r: the weights of row r's states (this warpgroup's, the second's, the prefix's)
          const int r = t;
          const size_t row = (size_t)(s0 + r / G) * a.Hq + (size_t)kvh * G + r % G;
          float m0 = -INFINITY, l0 = 0.f;
#pragma unroll
          for (int k = 0; k < kWRows; ++k) {
            m0 = k == r ? mrun[k] : m0;
            l0 = k == r ? lrow[k] : l0;
          }
          const float m1 = xml[r], l1 = xml[16 + r];
          float M = fmaxf(l0 > 0.f ? m0 : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
          for (int p = 0; p < npre; ++p) {
            const float2 ml = __ldg(reinterpret_cast<const float2 *>(a.pre_ml) + p * slab + row);
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
          }
          const float c0 = l0 > 0.f ? ex2_ftz(m0 - M) : 0.f, c1 = l1 > 0.f ? ex2_ftz(m1 - M) : 0.f;
          float den = c0 * l0 + c1 * l1;
          for (int p = 0; p < npre; ++p) {
            const float2 ml = __ldg(reinterpret_cast<const float2 *>(a.pre_ml) + p * slab + row);
            const float w = ml.y > 0.f ? ml.y * ex2_ftz(ml.x - M) : 0.f;
            wts[r * kW + 2 + p] = w;
            den += w;
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          wts[r * kW] = c0 * inv;
          wts[r * kW + 1] = c1 * inv;
          for (int p = 0; p < npre; ++p) wts[r * kW + 2 + p] *= inv;
        }
        mbar_arrive(&bars[WB_WTS]);
        if (!wait_warp(WB_WTS, (uint32_t)(u & 1))) break;
        if (n < 0) {  // refused unit: zero rows (in range), report
          if (s0 >= 0 && nm > 0 && s0 + nm <= a.S)
            for (int r = 0; r < nm * G; ++r)
              a.out[((size_t)(s0 + r / G) * a.Hq + (size_t)kvh * G + r % G) * kWD + t] = __float2bfloat16(0.f);
          if (t == 0 && a.err) atomicOr(a.err, PA_DEVERR_CTX);
        } else {
#pragma unroll
          for (int r = 0; r < kWRows; ++r) {
            if (r < ncols) {
              const size_t row = (size_t)(s0 + r / G) * a.Hq + (size_t)kvh * G + r % G;
              float res = wts[r * kW] * oreg[r] + wts[r * kW + 1] * xo[r * kWD + t];
              for (int p = 0; p < npre; ++p) res += wts[r * kW + 2 + p] * __ldg(a.pre_o + (p * slab + row) * kWD + t);
              a.out[row * kWD + t] = __float2bfloat16(res);
            }
          }
        }
        mbar_arrive(&bars[WB_XDONE]);
      }
      mbar_arrive(&bars[WB_UEMPTY + ub]);
      ++u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kWTmemCols);
  }
  // a programmatic dependent of the prefix pass: complete only after it
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int B>
int launch_wide(const CUtensorMap &tk, const CUtensorMap &tv, const WideArgs &a, int sms, cudaStream_t st) {
  using L = WideSmem<B>;
  static_assert(L::kAlloc <= 227 * 1024, "wide decode shared memory over the per-CTA limit");
  auto kern = decode_wide_kernel<B>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
    return PA_ERR_CUDA;
  const long long nunits = (long long)a.nsg * a.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nunits < sms ? nunits : sms));
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

bool wide_supported(const pa_decode_desc *d, int nsg, int rows) {
  return d->head_dim == kWD && (d->block_size == 16 || d->block_size == 32) && nsg > 0 && nsg <= kTaskMaxSub &&
         nsg <= d->num_seqs && rows > 0 && rows <= kWRows && (long long)nsg * d->num_kv_heads < (1ll << 31);
}

int decode_wide_launch(const pa_decode_desc *d, const void *q, const void *k_pool, const void *v_pool,
                       const int32_t *block_tables, const int32_t *context_lens, const DecodePrefix &pre, int rows,
                       void *out, unsigned int *counter, int32_t *err_flag, void *stream) {
  const int sms = current_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const uint64_t nrows = (uint64_t)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tk, tv;
  if (!encode_2d_bf16(&tk, k_pool, nrows, kWD, d->block_size, 64, true) ||
      !encode_2d_bf16(&tv, v_pool, nrows, kWD, d->block_size, 64, true))
    return PA_ERR_CUDA;
  WideArgs a{};
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
  a.ctr = counter;
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d->block_size == 16 ? launch_wide<16>(tk, tv, a, sms, s) : launch_wide<32>(tk, tv, a, sms, s);
}

}  // namespace pa
