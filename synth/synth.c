/* Seeded synthetic inputs: host implementation.
 *
 * This file draws the random tensors that both the CUDA path and the CPU
 * oracle consume.  It holds none of the mixture-of-experts arithmetic.
 *
 * Definition (identical to synth/__init__.py, which evaluates the same
 * sequence of IEEE-754 float64 operations with torch on any device):
 *
 *   word(seed, tid, i) = fmix64(key(seed, tid) + (i + 1) * G)      (mod 2^64)
 *   key(seed, tid)     = fmix64(seed * G + tid)
 *   fmix64             = the SplitMix64 output finaliser (Steele, Lea, Flood 2014)
 *   u1 = ((word >> 40) + 0.5) * 2^-24          in (0, 1)
 *   u2 = ((word >> 16) & 0xFFFFFF) * 2^-24     in [0, 1)
 *   n  = sqrt(-2 * ln u1) * cos(2 pi u2)       (Box & Muller 1958)
 *   value = bf16_rne(f32_rne(n * std))
 *
 * ln and cos are evaluated with polynomials whose coefficients the caller
 * passes in (so both implementations use the same float64 constants), with
 * only +, -, *, / and sqrt, which IEEE-754 rounds correctly everywhere.
 * Build with -ffp-contract=off so no multiply-add is fused.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define G_GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t fmix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_word(uint64_t seed, uint64_t tid, uint64_t i) {
  uint64_t key = fmix64(seed * G_GOLDEN + tid);
  return fmix64(key + (i + 1) * G_GOLDEN);
}

/* ln(u) for u in (0, 1): u = m * 2^e, m folded into [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(s) with s = (m-1)/(m+1), series in s^2 by Horner. */
static double synth_ln(double u, const double* c, int nc, double ln2, double sqrt_half) {
  uint64_t bits;
  memcpy(&bits, &u, 8);
  int64_t e = (int64_t)((bits >> 52) & 0x7FF) - 1022;
  bits = (bits & 0x800FFFFFFFFFFFFFULL) | (1022ULL << 52);
  double m;
  memcpy(&m, &bits, 8);
  if (m < sqrt_half) { m = m * 2.0; e = e - 1; }
  double s = (m - 1.0) / (m + 1.0);
  double z = s * s;
  double p = c[nc - 1];
  for (int k = nc - 2; k >= 0; --k) p = p * z + c[k];
  return 2.0 * s * p + (double)e * ln2;
}

/* cos(2 pi v) for v in [0, 1): fold to w in [0, 1/4] exactly, Taylor series in theta^2. */
static double synth_cos2pi(double v, const double* c, int nc, double two_pi) {
  double w = v;
  if (w > 0.5) w = 1.0 - w;
  double sign = 1.0;
  if (w > 0.25) { w = 0.5 - w; sign = -1.0; }
  double th = w * two_pi;
  double t2 = th * th;
  double p = c[nc - 1];
  for (int k = nc - 2; k >= 0; --k) p = p * t2 + c[k];
  return sign * p;
}

static uint16_t synth_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u = u + 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Draw out[0..n) = values for counters start .. start+n-1. */
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, int64_t n, double std,
                       const double* ln_coef, int n_ln, const double* cos_coef, int n_cos,
                       const double* consts /* ln2, sqrt_half, two_pi */, uint16_t* out) {
  const double ln2 = consts[0], sqrt_half = consts[1], two_pi = consts[2];
  const double inv24 = 1.0 / 16777216.0;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t w = synth_word(seed, tid, start + (uint64_t)i);
    double u1 = ((double)(w >> 40) + 0.5) * inv24;
    double u2 = (double)((w >> 16) & 0xFFFFFFULL) * inv24;
    double r = sqrt(-2.0 * synth_ln(u1, ln_coef, n_ln, ln2, sqrt_half));
    double v = r * synth_cos2pi(u2, cos_coef, n_cos, two_pi);
    out[i] = synth_f32_to_bf16((float)(v * std));
  }
}
