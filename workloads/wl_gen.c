/* Fast path of the seeded input generator (same definition as the numpy code in
 * workloads/__init__.py: SplitMix64 counter stream, Box-Muller pairs in fp64,
 * fp64 -> fp32 -> bf16 round-to-nearest-even).  Holds no attention arithmetic.
 * Built by workloads/build.py; used through ctypes. */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t wl_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Uniform double in [0,1) from draw number idx (1-based counter) of a stream. */
static inline double wl_uniform(uint64_t base, uint64_t idx) {
  uint64_t z = wl_mix64(base + idx * WL_GAMMA);
  return (double)(z >> 11) * 0x1.0p-53;
}

static inline uint16_t wl_f64_to_bf16(double x) {
  float f = (float)x; /* RNE under the default rounding mode */
  uint32_t b;
  memcpy(&b, &f, 4);
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

/* n bf16 normals; the first uniform consumed is draw number pos+1.  Element e
 * uses the pair of draws (pos + 2*(e/2) + 1, pos + 2*(e/2) + 2): cos for even e,
 * sin for odd e.  Consumes 2*ceil(n/2) draws. */
void wl_normal_bf16(uint64_t base, uint64_t pos, int64_t n, uint16_t *out) {
  int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npair; ++p) {
    double u1 = wl_uniform(base, pos + 2 * (uint64_t)p + 1);
    double u2 = wl_uniform(base, pos + 2 * (uint64_t)p + 2);
    double r = sqrt(-2.0 * log1p(-u1));
    double t = (2.0 * M_PI) * u2;
    out[2 * p] = wl_f64_to_bf16(r * cos(t));
    if (2 * p + 1 < n) out[2 * p + 1] = wl_f64_to_bf16(r * sin(t));
  }
}

/* n raw draws starting at draw number pos+1. */
void wl_draw(uint64_t base, uint64_t pos, int64_t n, uint64_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = wl_mix64(base + (pos + (uint64_t)i + 1) * WL_GAMMA);
}
