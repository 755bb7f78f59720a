// Shared-memory plan of libpagedattn's fused launches (sm_103a): the mixed
// step (pa_mixed.cu) and shared-prefix decode (pa_shared_prefix.cu) run one
// grid of 384-thread CTAs in which each CTA either runs one prefill tile pair
// (pa_prefill_body.cuh) or kUnitsPerCta decode units of four warps
// (pa_decode_body.cuh), each unit with its own shared memory and named
// barrier 1 + its index.  Three units fit in the prefill CTA's footprint, so
// an SM holds one CTA of either kind.
#pragma once

#include "pa_decode_body.cuh"
#include "pa_prefill_body.cuh"

namespace pa {
namespace {

constexpr int kUnitsPerCta = kThreads / 128;  // decode units (4 warps each) in one fused CTA

template <int B>
struct FusedSmem {
  // 16-token pages: two ring slots a warp (three units must fit one CTA);
  // 32-token pages: one, as in the decode kernel.
  static constexpr int kDecodeStages = B == 16 ? 2 : 1;
  using L = DecodeSmem<128, B, 4, kDecodeStages>;
  static constexpr int kUnitStride = (L::kBytes + 1023) & ~1023;
  static constexpr int kDecodeBytes = kUnitsPerCta * kUnitStride + 1024;  // + alignment slack
  static constexpr int kBytes = kDecodeBytes > kSmem ? kDecodeBytes : kSmem;
  static_assert(kBytes <= 227 * 1024, "fused shared memory over the per-CTA limit");
};

}  // namespace
}  // namespace pa
