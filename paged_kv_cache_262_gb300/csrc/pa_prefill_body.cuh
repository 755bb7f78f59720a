// The chunked-prefill tile of libpagedattn (sm_103a): argument block, shared
// memory and TMEM plan, and the per-CTA device code, included by the prefill
// kernel (pa_prefill.cu) and the mixed-step kernel (pa_mixed.cu).  The design
// notes are at the top of pa_prefill.cu.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {
namespace {

struct PrefillArgs {
  const __nv_bfloat16 *q;
  const int32_t *cu_q;
  const int32_t *bt;
  const int32_t *ctx;
  __nv_bfloat16 *out;
  int32_t *err;
  int R, Hq, Hkv, num_blocks, max_blocks, max_ctx, total_q;
  float scale_log2;
  int causal;       // 0: every row sees all ctx keys (shared-prefix pass)
  float *part_o;    // non-null: write fp32 o/l [kparts][total_q][Hq][128] ...
  float *part_ml;   // ... and (m, l) [kparts][total_q][Hq][2] instead of bf16 out
  int kparts;       // non-causal: keys split into kparts ranges of kpart_len
  int kpart_len;    // (a multiple of 128), one partial state per range
};

constexpr int kD = 128;         // head_dim
constexpr int kBM = 128;        // MMA rows per query tile (two tiles per CTA)
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kHalf = 16384;    // one 64-column half of a 128 x 128 bf16 tile
constexpr int kTile = 32768;    // 128 x 128 bf16
#ifndef PA_PREFILL_KST
#define PA_PREFILL_KST 2
#endif
constexpr int KST = PA_PREFILL_KST;       // K ring depth
constexpr int VST = 2;                    // V ring depth
constexpr int kOffQ = 0;                  // tiles A, B
constexpr int kOffK = kOffQ + 2 * kTile;
constexpr int kOffV = kOffK + KST * kTile;
constexpr int kOffBar = kOffV + VST * kTile;
constexpr int kSmem = kOffBar + 256 + 1024;
constexpr int kTmemCols = 512;  // S/P of A [0,128), of B [128,256); O of A [256,384), of B [384,512)
constexpr int kThreads = 384;  // three warpgroups
#ifndef PA_PREFILL_LPT_MAX
#define PA_PREFILL_LPT_MAX 256
#endif
constexpr int kLptMaxSeqs = PA_PREFILL_LPT_MAX;  // longest-first chunk order up to this many chunks
// Register split (setmaxnreg): the two softmax warpgroups hold a 128-column
// row of scores each and take kRegsSoftmax per thread; the third warpgroup
// (producer, MMA issuer, two idle warps) gives its registers back.  The sum
// equals the launch allocation of kThreads x kRegsLaunch, which the host
// checks before every launch (a larger sum would wait forever).
constexpr int kRegsLaunch = 168, kRegsSoftmax = 216, kRegsOther = 72;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split");

// Barriers: Q rows stored (both tiles); K and V stage full / free (one per
// ring slot); S of tile A / B ready; P of tile A / B written; all MMAs done.
enum {
  BAR_Q = 0, BAR_K_FULL = 1, BAR_K_EMPTY = BAR_K_FULL + KST, BAR_V_FULL = BAR_K_EMPTY + KST,
  BAR_V_EMPTY = BAR_V_FULL + VST, BAR_S_FULL = BAR_V_EMPTY + VST, BAR_P_FULL = BAR_S_FULL + 2,
  BAR_O_DONE = BAR_P_FULL + 2, NBARS = BAR_O_DONE + 1
};
static_assert(NBARS * 8 + 8 <= 256, "barrier area");
static_assert(kOffBar + 256 + 1024 <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t pack2(float a, float b) { return pack_bf16(a, b); }

// P of one row: 2^(s * scale_log2 - m) for the 128 scores, packed to bf16
// pairs into TMEM columns [col, col + 64); the row sum adds the unrounded
// fp32 probabilities in four packed chains (acc).
__device__ __forceinline__ void probabilities(const float (&s)[kBN], float2 sc2, float2 nm2, uint32_t col,
                                              float2 (&acc)[4]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int k = c * 64 + 2 * e;
      const float2 t = fma2(make_float2(s[k], s[k + 1]), sc2, nm2);
      const float2 p = make_float2(ex2_ftz(t.x), ex2_ftz(t.y));
      w[e] = pack2(p.x, p.y);
      acc[e & 3] = add2(acc[e & 3], p);
    }
    tmem_st32(col + c * 32, w);
  }
}

// One prefill CTA's work: the pair of query tiles (bx of gx, counted from the
// last), kv head by, chunk / key range bz, on all kThreads threads of the CTA
// with its shared memory at `smem` (1024-aligned, kSmem - 1024 bytes).  The
// prefill kernel runs one per CTA; the mixed-step kernel gives some CTAs this
// role and others decode units.
template <int B, int G, bool PARTIAL>
__device__ __forceinline__ void prefill_tile(const CUtensorMap *tmK, const CUtensorMap *tmV, const PrefillArgs &a,
                                             int bx, int by, int bz, int gx, uint8_t *smem) {
  constexpr int TP = kBM / G;        // positions per query tile
  constexpr int PAGES = kBN / B;     // pages per key tile
  // 8 pages a tile (16-token pages): one producer lane per page, so the
  // tile's 32 loads leave together (1035 -> 1309 TFLOP/s on the mixed step
  // with 16-token pages); 4 pages: one lane issues them all (0.7% faster).
  constexpr bool kLanePerPage = PAGES > 4;
  constexpr uint32_t kIdS = umma_idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdPV = umma_idesc_bf16(128, 128, false, true);

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffBar + NBARS * 8);
  volatile int *dead = reinterpret_cast<volatile int *>(smem + kOffBar + NBARS * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = gx - 1 - bx;  // later tiles see more keys: start them first
  const int g = by, kpart = bz % a.kparts;
  // Chunks in order of decreasing context (the longest work first), so that
  // the last CTAs to start are short ones; ties in chunk order.
  int r = bz / a.kparts;
  if (a.R > 1 && a.R <= kLptMaxSeqs) {
    __shared__ int s_r;
    for (int i = threadIdx.x; i < a.R; i += kThreads) {
      const int ci = __ldg(a.ctx + i);
      int rank = 0;
      for (int k = 0; k < a.R; ++k) {
        const int ck = __ldg(a.ctx + k);
        rank += (ck > ci) || (ck == ci && k < i);
      }
      if (rank == r) s_r = i;
    }
    __syncthreads();
    r = s_r;
  }
  const int c0 = __ldg(a.cu_q + r), c1 = __ldg(a.cu_q + r + 1);
  const int C = c1 - c0;
  const int ctx_full = __ldg(a.ctx + r);
  // key range of this CTA: all keys, or one of the non-causal key ranges
  const int key_lo = a.kparts > 1 ? kpart * a.kpart_len : 0;
  const int ctx = a.kparts > 1 ? max(0, min(ctx_full - key_lo, a.kpart_len)) : ctx_full;
  float *part_o = a.part_o ? a.part_o + (size_t)kpart * a.total_q * a.Hq * kD : nullptr;
  float *part_ml = a.part_ml ? a.part_ml + (size_t)kpart * a.total_q * a.Hq * 2 : nullptr;
  const int q0 = qt * 2 * TP;  // first position index of tile A
  if (C <= 0 || q0 >= C) return;
  const bool empty = a.kparts > 1 && ctx_full > 0 && ctx == 0;  // range past a shorter prefix
  const bool bad = ctx_full <= 0 || (a.causal && C > ctx) || ctx_full > a.max_blocks * B || ctx_full > a.max_ctx ||
                   c0 < 0 || c1 > a.total_q;
  if (bad || empty) {  // zero this CTA's rows (an empty partial state); report bad ones
    if (c0 >= 0 && c1 <= a.total_q) {
      for (int m = threadIdx.x; m < 2 * kBM; m += kThreads) {
        const int t = q0 + m / G;
        if (t >= C) continue;
        const size_t row = (size_t)(c0 + t) * a.Hq + g * G + m % G;
        if (part_o) {
          for (int i = 0; i < kD; ++i) part_o[row * kD + i] = 0.f;
          part_ml[2 * row] = -INFINITY;
          part_ml[2 * row + 1] = 0.f;
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * kD);
          for (int i = 0; i < kD / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    if (bad && threadIdx.x == 0 && a.err) atomicOr(a.err, PA_DEVERR_CTX);
    return;
  }
  const int npages = (ctx + B - 1) / B;  // pages of this CTA's key range
  // last valid position of the CTA (non-causal rows all sit at ctx - 1)
  const int pos_hi = a.causal ? ctx - C + min(C, q0 + 2 * TP) - 1 : ctx - 1;
  const int T = pos_hi / kBN + 1;                         // key tiles

  if (threadIdx.x == 0) {
    mbar_init(&bars[BAR_Q], 256);
    for (int b = BAR_K_FULL; b < BAR_P_FULL; ++b) mbar_init(&bars[b], 1);
    mbar_init(&bars[BAR_P_FULL], 128);
    mbar_init(&bars[BAR_P_FULL + 1], 128);
    mbar_init(&bars[BAR_O_DONE], 1);
    *dead = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto wait = [&](int b, uint32_t parity) {
    if (*dead) return false;
    if (mbar_wait(&bars[b], parity)) return true;
    *dead = 1;
    if (a.err) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    return false;
  };

  if (warp >= 8) {
    setmaxnreg_dec<kRegsOther>();
    if (warp == 8) {
      if constexpr (kLanePerPage) {
        // ----------------------------------------------------------- producer
        // lane i < PAGES gathers page i of each key tile, so the tile's loads
        // leave together rather than one after another from a single lane
        const uint64_t pol = policy_evict_first();
        const int32_t *bt_row = a.bt + (size_t)r * a.max_blocks + key_lo / B;
        auto page_id = [&](int j) {  // validated page of this lane in key tile j, -1 = none
          const int pi = j * PAGES + lane;
          int pg = -1;
          if (lane < PAGES && pi < npages) {
            pg = __ldg(bt_row + pi);
            if (pg < 0 || pg >= a.num_blocks) {
              if (a.err) atomicOr(a.err, PA_DEVERR_PAGE);
              pg = -1;
            }
          }
          return pg;
        };
        auto load = [&](int pg, uint64_t *bar, uint8_t *dst, const CUtensorMap *map) {
          const unsigned have = __ballot_sync(0xffffffffu, pg >= 0);
          if (lane == 0) {
            if (have == 0)
              mbar_arrive(bar);
            else
              mbar_arrive_expect_tx(bar, (uint32_t)__popc(have) * B * 256);
          }
          __syncwarp();
          if (pg >= 0) {
            const int row = (pg * a.Hkv + g) * B;
            tma_load_2d_hint(dst + lane * B * 128, map, 0, row, bar, pol);
            tma_load_2d_hint(dst + kHalf + lane * B * 128, map, 64, row, bar, pol);
          }
        };
        auto wait_all = [&](int b, uint32_t parity) { return __all_sync(0xffffffffu, wait(b, parity)); };
        int cur = page_id(0);
        for (int j = 0; j < T; ++j) {
          const int ks = j % KST, vs = j % VST;
          const int nxt = j + 1 < T ? page_id(j + 1) : -1;  // table reads of the next tile overlap this one
          if (j >= KST && !wait_all(BAR_K_EMPTY + ks, (uint32_t)((j / KST - 1) & 1))) break;
          load(cur, &bars[BAR_K_FULL + ks], smem + kOffK + ks * kTile, tmK);
          if (j >= VST && !wait_all(BAR_V_EMPTY + vs, (uint32_t)((j / VST - 1) & 1))) break;
          load(cur, &bars[BAR_V_FULL + vs], smem + kOffV + vs * kTile, tmV);
          cur = nxt;
        }
      } else if (lane == 0) {
        // ----------------------------------------------------------- producer
        const uint64_t pol = policy_evict_first();
        const int32_t *bt_row = a.bt + (size_t)r * a.max_blocks + key_lo / B;
        auto page_ids = [&](int j, int (&pages)[PAGES]) {  // validated ids of tile j, -1 = none
  #pragma unroll
          for (int i = 0; i < PAGES; ++i) {
            const int pi = j * PAGES + i;
            int pg = -1;
            if (pi < npages) {
              pg = __ldg(bt_row + pi);
              if (pg < 0 || pg >= a.num_blocks) {
                if (a.err) atomicOr(a.err, PA_DEVERR_PAGE);
                pg = -1;
              }
            }
            pages[i] = pg;
          }
        };
        auto load = [&](const int (&pages)[PAGES], uint64_t *bar, uint8_t *dst, const CUtensorMap *map) {
          int n = 0;
  #pragma unroll
          for (int i = 0; i < PAGES; ++i) n += pages[i] >= 0;
          if (n == 0) {
            mbar_arrive(bar);
            return;
          }
          mbar_arrive_expect_tx(bar, (uint32_t)n * B * 256);
  #pragma unroll
          for (int i = 0; i < PAGES; ++i) {
            if (pages[i] < 0) continue;
            const int row = (pages[i] * a.Hkv + g) * B;
            tma_load_2d_hint(dst + i * B * 128, map, 0, row, bar, pol);
            tma_load_2d_hint(dst + kHalf + i * B * 128, map, 64, row, bar, pol);
          }
        };
        int cur[PAGES], nxt[PAGES];
        page_ids(0, cur);
        for (int j = 0; j < T; ++j) {
          const int ks = j % KST, vs = j % VST;
          if (j + 1 < T) page_ids(j + 1, nxt);  // table reads of the next tile overlap this one
          if (j >= KST && !wait(BAR_K_EMPTY + ks, (uint32_t)((j / KST - 1) & 1))) break;
          load(cur, &bars[BAR_K_FULL + ks], smem + kOffK + ks * kTile, tmK);
          if (j >= VST && !wait(BAR_V_EMPTY + vs, (uint32_t)((j / VST - 1) & 1))) break;
          load(cur, &bars[BAR_V_FULL + vs], smem + kOffV + vs * kTile, tmV);
  #pragma unroll
          for (int i = 0; i < PAGES; ++i) cur[i] = nxt[i];
        }
      }
    } else if (warp == 9 && lane == 0) {
      // --------------------------------------------------------- MMA issuer
      const uint32_t sq = smem_u32(smem + kOffQ), sk = smem_u32(smem + kOffK);
      const uint32_t sv = smem_u32(smem + kOffV);
      auto issue_s = [&](int x, int j) {  // S of tile x (0 = A, 1 = B) against K tile j
        const uint32_t kb = sk + (j % KST) * kTile, qb = sq + x * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + x * 128, umma_desc_sw128(qb + off, 16, 1024), umma_desc_sw128(kb + off, 16, 1024),
                    kIdS, kk > 0);
        }
        umma_commit(&bars[BAR_S_FULL + x]);
      };
      auto issue_pv = [&](int x, int j) {  // O_x += P_x V_j, P_x from TMEM
        const uint32_t vb = sv + (j % VST) * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16_ts(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, umma_desc_sw128(vb + kk * 2048, kHalf, 1024),
                       kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = wait(BAR_Q, 0) && wait(BAR_K_FULL, 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit(&bars[BAR_K_EMPTY]);
      }
      for (int j = 0; ok && j < T; ++j) {
        const bool more = j + 1 < T;
        const uint32_t par = (uint32_t)(j & 1);
        if (!wait(BAR_V_FULL + j % VST, (uint32_t)((j / VST) & 1))) break;
        if (!wait(BAR_P_FULL, par)) break;
        tc_fence_after();
        issue_pv(0, j);
        if (more) {
          if (!wait(BAR_K_FULL + (j + 1) % KST, (uint32_t)(((j + 1) / KST) & 1))) break;
          tc_fence_after();
          issue_s(0, j + 1);
        }
        if (!wait(BAR_P_FULL + 1, par)) break;
        tc_fence_after();
        issue_pv(1, j);
        umma_commit(&bars[BAR_V_EMPTY + j % VST]);
        if (more) {
          issue_s(1, j + 1);
          umma_commit(&bars[BAR_K_EMPTY + (j + 1) % KST]);
        }
      }
      umma_commit(&bars[BAR_O_DONE]);
    }
  } else {
    // ------------------------------------- softmax: tile x, row m = TMEM lane
    setmaxnreg_inc<kRegsSoftmax>();
    const int x = warp >> 2;
    const int m = (warp & 3) * 32 + lane;
    const int tloc = q0 + x * TP + m / G;  // position index within the chunk
    const bool row_valid = tloc < C;
    const int pos = (row_valid && a.causal) ? ctx - C + tloc : ctx - 1;
    const int pos_lo = a.causal ? ctx - C + q0 + x * TP : ctx - 1;  // first position of this tile
    const int head = g * G + m % G;
    {  // the tile's Q rows -> shared memory (128-byte swizzle, two 64-column
       // halves); a warp loads two whole rows per instruction (16-byte chunk
       // per lane), rows past the chunk as zeros
      uint8_t *qd = smem + kOffQ + x * kTile;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int k = i * 128 + m, mr = k >> 4, c = k & 15;  // row and chunk of the tile
        const int t = q0 + x * TP + mr / G;
        const uint4 v = t < C ? __ldg(reinterpret_cast<const uint4 *>(
                                    a.q + ((size_t)(c0 + t) * a.Hq + g * G + mr % G) * kD) + c)
                              : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(qd + (c >> 3) * kHalf + sw128(mr, c & 7)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[BAR_Q]);
    }
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = x * 128, o_col = 256 + x * 128;
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < T; ++j) {
      if (!wait(BAR_S_FULL + x, (uint32_t)(j & 1))) break;
      tc_fence_after();
      float s[kBN];
      {
        uint32_t v[4][32];  // four loads in flight, one wait
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[c][i]);
      }
      const int key0 = j * kBN;
      const bool masked = key0 + kBN - 1 > pos_lo;  // some key past some row's position
      if (masked) {
#pragma unroll
        for (int i = 0; i < kBN; ++i) s[i] = (key0 + i <= pos) ? s[i] : -INFINITY;
      }
      float mx;  // max of the raw scores (scale > 0 keeps the order), 8 independent chains
      {
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = s[u];
#pragma unroll
        for (int i = 8; i < kBN; i += 2) pm[(i >> 1) & 7] = max3f(pm[(i >> 1) & 7], s[i], s[i + 1]);
        mx = max3f(max3f(pm[0], pm[1], pm[2]), max3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      }
      const float m_new = fmaxf(m_run, mx * a.scale_log2);
      const bool rescale = m_new > m_run + 8.f;
      const float m_use = rescale ? m_new : m_run;
      const float alpha = rescale ? exp2f(m_run - m_new) : 1.f;
      // value rows of keys past the context must not carry NaNs into 0 * v
      // (tile A's PV runs first, so tile A's threads clear them)
      if (x == 0 && key0 + kBN > ctx) {
        if (!wait(BAR_V_FULL + j % VST, (uint32_t)((j / VST) & 1))) break;
        if (key0 + m >= ctx) {
          uint8_t *vd = smem + kOffV + (j % VST) * kTile;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4 *>(vd + m * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(vd + kHalf + m * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      // P (bf16 pairs) over the first 64 columns of this tile's S
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      probabilities(s, make_float2(a.scale_log2, a.scale_log2), make_float2(-m_use, -m_use), lane_base + s_col, acc);
      const float2 acc2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
      const float lsum = acc2.x + acc2.y;
      if (rescale && j >= 1) {  // the previous PV of this tile is done (S of tile j followed it)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + o_col + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(lane_base + o_col + c * 32, v);
        }
      }
      tmem_wait_st();
      l_run = l_run * alpha + lsum;
      m_run = m_use;
      tc_fence_before();
      mbar_arrive(&bars[BAR_P_FULL + x]);
    }
    if (wait(BAR_O_DONE, 0)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      if constexpr (PARTIAL) {
        // Partial states (fp32, 512-byte rows): the warp stages its 32 rows in
        // shared memory (free now: every MMA is done), 16-byte chunks
        // XOR-swizzled by row, then writes whole rows per instruction.
        uint8_t *stage = smem + warp * (32 * 512);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + o_col + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(stage + lane * 512 + (((c * 8 + i) ^ lane) & 31) * 16) =
                make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                            __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
        }
        __syncwarp();
#pragma unroll 4
        for (int r = 0; r < 32; ++r) {
          const int mr = (warp & 3) * 32 + r;
          const int t = q0 + x * TP + mr / G;
          if (t >= C) continue;
          const size_t orow = (size_t)(c0 + t) * a.Hq + g * G + mr % G;
          reinterpret_cast<uint4 *>(part_o + orow * kD)[lane] =
              *reinterpret_cast<const uint4 *>(stage + r * 512 + ((lane ^ r) & 31) * 16);
        }
      } else {
        uint8_t *stage = smem + warp * (32 * 256);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + o_col + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = pack2(__uint_as_float(v[8 * i + 0]) * inv, __uint_as_float(v[8 * i + 1]) * inv);
            o.y = pack2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv);
            o.z = pack2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv);
            o.w = pack2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv);
            *reinterpret_cast<uint4 *>(stage + lane * 256 + (((c * 4 + i) ^ lane) & 15) * 16) = o;
          }
        }
        __syncwarp();
#pragma unroll 4
        for (int r0 = 0; r0 < 32; r0 += 2) {
          const int r = r0 + (lane >> 4), ch = lane & 15;
          const int mr = (warp & 3) * 32 + r;
          const int t = q0 + x * TP + mr / G;
          if (t >= C) continue;
          const size_t orow = (size_t)(c0 + t) * a.Hq + g * G + mr % G;
          reinterpret_cast<uint4 *>(a.out + orow * kD)[ch] =
              *reinterpret_cast<const uint4 *>(stage + r * 256 + ((ch ^ r) & 15) * 16);
        }
      }
      if constexpr (PARTIAL) {
        if (row_valid) {
          const size_t row = (size_t)(c0 + tloc) * a.Hq + head;
          part_ml[2 * row] = m_run;
          part_ml[2 * row + 1] = l_run;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Host: validates a prefill call and fills its argument block and grid (one
// CTA per pair of query tiles, kv head and chunk x key range).  grid.x == 0
// with PA_OK means there is nothing to launch.
inline int prepare_prefill(const pa_decode_desc *d, const void *q, const int32_t *cu_q, int max_q_len, int total_q,
                           const void *k_pool, const void *v_pool, const int32_t *block_tables,
                           const int32_t *context_lens, void *out, float *part_o, float *part_ml, int causal,
                           int kparts, int kpart_len, int32_t *err_flag, PrefillArgs *a, dim3 *grid) {
  *grid = dim3(0, 0, 0);
  int st = validate_decode_desc(d);
  if (st != PA_OK) return st;
  if (d->head_dim != kD) return PA_ERR_UNSUPPORTED;
  const int G = d->num_q_heads / d->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PA_ERR_UNSUPPORTED;
  if (max_q_len < 0 || total_q < 0) return PA_ERR_INVALID;
  if (d->num_seqs == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
  if (!q || !cu_q || !k_pool || !v_pool || !block_tables || !context_lens || (!out && !part_o))
    return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || (out && !aligned16(out)) ||
      (part_o && (!aligned16(part_o) || !part_ml)))
    return PA_ERR_INVALID;
  if (kparts < 1 || (kparts > 1 && (causal || !part_o || kpart_len <= 0 || kpart_len % 128 != 0)))
    return PA_ERR_INVALID;
  if ((long long)d->num_seqs * kparts > 65535 || d->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  const long long tiles = ((long long)max_q_len * G + 2 * kBM - 1) / (2 * kBM);
  if (tiles > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  a->q = static_cast<const __nv_bfloat16 *>(q);
  a->cu_q = cu_q;
  a->bt = block_tables;
  a->ctx = context_lens;
  a->out = static_cast<__nv_bfloat16 *>(out);
  a->err = err_flag;
  a->R = d->num_seqs;
  a->Hq = d->num_q_heads;
  a->Hkv = d->num_kv_heads;
  a->num_blocks = d->num_blocks;
  a->max_blocks = d->max_blocks_per_seq;
  a->max_ctx = d->max_context_len;
  a->total_q = total_q;
  a->scale_log2 = d->scale * 1.4426950408889634f;
  a->causal = causal;
  a->part_o = part_o;
  a->part_ml = part_ml;
  a->kparts = kparts;
  a->kpart_len = kpart_len;
  *grid = dim3((unsigned)tiles, d->num_kv_heads, d->num_seqs * kparts);
  return PA_OK;
}

}  // namespace
}  // namespace pa
