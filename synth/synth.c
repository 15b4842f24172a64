/*
 * Seeded synthetic inputs for the FC2 workloads (shared by the CUDA tests,
 * the oracle checks and the benchmark; holds none of the NVFP4 arithmetic).
 *
 * Element i of stream `stream` under `seed`:
 *   key   = mix(seed * 0x9E3779B97F4A7C15 + stream + 1)
 *   w(j)  = mix(key + (j + 1) * 0x9E3779B97F4A7C15)          (splitmix64)
 *   u1,u2,u3 = top 53 bits of w(3i), w(3i+1), w(3i+2) scaled to [0, 1)
 *   z     = sqrt(-2 ln(1 - u1)) * cos(2 pi u2)                (Box-Muller)
 *   z    *= 20 if u3 < outlier_p                               (outliers)
 *   value = RNE_bf16(z * sigma)
 * The workloads draw activations as N(0,1) with 0.1% of entries x20 and
 * weights as N(0, sigma = K^-1/2) without outliers.
 * Build with -ffp-contract=off: the same bytes on x86-64 and AArch64 up to
 * libm's last-ulp differences, which the BF16 rounding absorbs.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Fill out[0..n) with elements [first, first+n) of the stream. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, int64_t n,
                       double sigma, double outlier_p, double outlier_scale, uint16_t* out) {
  const uint64_t golden = 0x9E3779B97F4A7C15ull;
  const uint64_t key = mix(seed * golden + stream + 1ull);
  const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) {
    uint64_t i = first + (uint64_t)t;
    double u1 = (double)(mix(key + (3 * i + 1) * golden) >> 11) * 0x1p-53;
    double u2 = (double)(mix(key + (3 * i + 2) * golden) >> 11) * 0x1p-53;
    double u3 = (double)(mix(key + (3 * i + 3) * golden) >> 11) * 0x1p-53;
    double z = sqrt(-2.0 * log(1.0 - u1)) * cos(two_pi * u2);
    if (u3 < outlier_p) z *= outlier_scale;
    out[t] = to_bf16((float)(z * sigma));
  }
}
