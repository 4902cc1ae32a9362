/* CPU oracle for the mixture-of-experts layer - TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this code.  It shares nothing with the CUDA library: its own bf16
 * conversion, its own routing, sort and matrix loops.
 *
 * What it computes - the MoE layer of "X-Stage: An Overlooked Pipeline Stage
 * for Communication-Computation Overlap in DiT Inference", MegaMoE background
 * paragraph: a router selects top-k experts per token; Dispatch sends each
 * token to its experts; each expert applies Linear-1 (hidden -> intermediate),
 * a SwiGLU activation (Shazeer 2020, "GLU Variants Improve Transformer") and
 * Linear-2 (intermediate -> hidden); Combine returns the outputs to the token
 * and sums the top-k results weighted by the router weights.  On one GPU
 * Dispatch/Combine are local permutations, so the oracle is the unfused
 * textbook computation, step by step, in plain loops:
 *
 *   1. logits[t,e] = sum_h x[t,h] * Wr[h,e] (+ bias[e])        fp32, canonical order
 *   2. top-k by logit (descending, ties -> lower expert id, NaN below -inf),
 *      w_j = softmax over the k selected logits (= full softmax renormalised)
 *   3. Dispatch: stable counting sort of the (t, j) pairs by expert id
 *   4. Linear-1: g = x W1[e][:, 0:I], u = x W1[e][:, I:2I]     fp32 accumulate
 *      SwiGLU:   a = bf16_rne(silu(g) * u)                    (act = 0)
 *      bilinear: a = bf16_rne(g * u)                          (act = 1, the
 *                GLU variant of the same paper; used as an exactness test)
 *   5. Linear-2: o = a W2[e]                                   fp32 accumulate
 *   6. Combine: y[t] = bf16_rne(sum_j fl(w_j * o_j)), slot order j = 0..k-1
 *
 * Precision: bf16 inputs, fp32 accumulation with one rounding per step
 * (fmaf), intermediate a rounded to bf16, output y rounded to bf16; softmax
 * weights in fp64, rounded to fp32.
 *
 * Canonical router order (the page does not fix a summation order; top-k is
 * a discrete decision, so both implementations must take it on identical
 * fp32 values): 32 partial sums, partial j accumulating h = j, j+32, j+64,
 * ... in ascending h with fmaf; then pairwise tree additions
 * p[j] += p[j+16] (j<16), p[j] += p[j+8] (j<8), ..., p[0] += p[1];
 * logit = p[0], plus bias[e] (one fp32 add) when a bias is given.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp (no fused multiply-adds other than
 * the explicit fmaf calls).  OpenMP only splits independent tokens.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */
static float o_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even fp32 -> bf16; NaN stays NaN (quiet bit set). */
static uint16_t o_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u = u + 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16_array(int64_t n, const float* in, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = o_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------- 1. router logits */
void oracle_router_logits(int64_t T, int H, int E, const uint16_t* x, const uint16_t* Wr,
                          const float* bias, float* logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      float p[32];
      for (int j = 0; j < 32; ++j) {
        p[j] = 0.0f;
        for (int h = j; h < H; h += 32)
          p[j] = fmaf(o_bf16_to_f32(x[t * H + h]), o_bf16_to_f32(Wr[(int64_t)h * E + e]), p[j]);
      }
      for (int off = 16; off >= 1; off >>= 1)
        for (int j = 0; j < off; ++j) p[j] = p[j] + p[j + off];
      logits[t * E + e] = bias ? p[0] + bias[e] : p[0];
    }
  }
}

/* ---------------------------------------------------- 2. top-k + weights */
/* Does expert a (logit la) rank strictly before expert b (logit lb)?
 * Higher logit first; NaN ranks below every number including -inf; equal
 * logits (and NaN vs NaN) rank by lower expert id. */
static int o_ranks_before(float la, int a, float lb, int b) {
  int na = isnan(la), nb = isnan(lb);
  if (na != nb) return nb;          /* the non-NaN one first */
  if (!na && la != lb) return la > lb;
  return a < b;
}

void oracle_topk(int64_t T, int E, int k, const float* logits, int32_t* ids, float* w) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    unsigned char taken[1024];
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {          /* selection: k passes over E */
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || o_ranks_before(l[e], e, l[best], best)) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    double m = (double)l[ids[t * k]];
    float ex[64];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      ex[j] = (float)exp((double)l[ids[t * k + j]] - m);
      sum += (double)ex[j];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = (float)((double)ex[j] / sum);
  }
}

/* ------------------------------------------------- 3. Dispatch (counting sort) */
/* counts[e] = #pairs routed to e; offsets = exclusive prefix (E+1 entries);
 * rows of expert e are offsets[e] .. offsets[e+1]-1 in ascending pair order
 * f = t*k + j; row_pair[row] = f; row_of[f] = row. */
void oracle_dispatch(int64_t T, int E, int k, const int32_t* ids, int32_t* counts,
                     int32_t* offsets, int32_t* row_pair, int32_t* row_of) {
  int64_t R = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t f = 0; f < R; ++f) counts[ids[f]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t f = 0; f < R; ++f) {
    int32_t row = cursor[ids[f]]++;
    row_pair[row] = (int32_t)f;
    row_of[f] = row;
  }
  free(cursor);
}

/* ------------------------------------------- 4-5. one expert on one token */
/* W1e: [H][2I] (columns 0..I-1 gate, I..2I-1 up); W2e: [I][H].
 * a_out[I] (bf16 bits), o_out[H] fp32; scratch >= 2I floats. */
void oracle_expert_ffn(int H, int I, const uint16_t* xrow, const uint16_t* W1e, const uint16_t* W2e,
                       int act, uint16_t* a_out, float* o_out, float* scratch) {
  float* acc = scratch;
  for (int n = 0; n < 2 * I; ++n) acc[n] = 0.0f;
  for (int h = 0; h < H; ++h) {             /* each acc[n] sums over h in ascending order */
    float xv = o_bf16_to_f32(xrow[h]);
    const uint16_t* wrow = W1e + (int64_t)h * 2 * I;
    for (int n = 0; n < 2 * I; ++n) acc[n] = fmaf(xv, o_bf16_to_f32(wrow[n]), acc[n]);
  }
  for (int n = 0; n < I; ++n) {
    float g = acc[n], u = acc[I + n], v;
    if (act == 0) {
      float s = g / (1.0f + expf(-g));      /* SiLU(g) = g * sigmoid(g) */
      v = s * u;
    } else {
      v = g * u;
    }
    a_out[n] = o_f32_to_bf16(v);
  }
  for (int m = 0; m < H; ++m) o_out[m] = 0.0f;
  for (int n = 0; n < I; ++n) {             /* each o[m] sums over n in ascending order */
    float an = o_bf16_to_f32(a_out[n]);
    const uint16_t* wrow = W2e + (int64_t)n * H;
    for (int m = 0; m < H; ++m) o_out[m] = fmaf(an, o_bf16_to_f32(wrow[m]), o_out[m]);
  }
}

/* ------------------------------------------------ 4-6. sampled tokens */
/* For each sampled token t = tokens[s]: run its k experts and combine.
 * W1p[e] / W2p[e]: per-expert pointers (only the experts the sample uses
 * need to be non-NULL).  y_out [ns][H] bf16 bits; a_out [ns][k][I] and
 * o_out [ns][k][H] optional (NULL to skip).  Returns 0, or -1 if a needed
 * expert pointer is NULL. */
int oracle_forward_tokens(int H, int I, int E, int k, int act, const uint16_t* x,
                          const uint16_t* const* W1p, const uint16_t* const* W2p,
                          const int32_t* ids, const float* w, int64_t ns, const int64_t* tokens,
                          uint16_t* y_out, uint16_t* a_out, float* o_out) {
  for (int64_t s = 0; s < ns; ++s)
    for (int j = 0; j < k; ++j) {
      int e = ids[tokens[s] * k + j];
      if (e < 0 || e >= E || !W1p[e] || !W2p[e]) return -1;
    }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t s = 0; s < ns; ++s) {
    int64_t t = tokens[s];
    float* scratch = (float*)malloc(sizeof(float) * (size_t)(2 * I));
    float* o = (float*)malloc(sizeof(float) * (size_t)H * (size_t)k);
    uint16_t* a = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    if (!scratch || !o || !a) { bad = 1; }
    else {
      for (int j = 0; j < k; ++j) {
        int e = ids[t * k + j];
        oracle_expert_ffn(H, I, x + t * H, W1p[e], W2p[e], act, a, o + (int64_t)j * H, scratch);
        if (a_out) memcpy(a_out + (s * k + j) * I, a, sizeof(uint16_t) * (size_t)I);
        if (o_out) memcpy(o_out + (s * k + j) * H, o + (int64_t)j * H, sizeof(float) * (size_t)H);
      }
      for (int m = 0; m < H; ++m) {          /* 6. Combine, slot order */
        float acc = w[t * k] * o[m];
        for (int j = 1; j < k; ++j) acc = acc + w[t * k + j] * o[(int64_t)j * H + m];
        y_out[s * H + m] = o_f32_to_bf16(acc);
      }
    }
    free(scratch);
    free(o);
    free(a);
  }
  return bad ? -2 : 0;
}

/* ============================================================================
 * Rounding flags of the intermediate and the interval of y they allow.
 *
 * Why: the intermediate a = bf16(silu(g) * u) is a discrete decision taken on
 * fp32 accumulations g, u.  An implementation that accumulates in another
 * order (the page fixes none) gets g, u that differ in the last bits, and
 * where silu(g) * u lies that close to a bf16 rounding boundary it rounds to
 * the neighbouring bf16 value.  The oracle reports, for every element, the
 * bf16 values a_lo <= a <= a_hi that such an accumulation can produce, and
 * carries them through Linear-2 and Combine as an interval of y.
 *
 * Stated bound.  g* = sum_h x_h W_hn, the exact value, is taken as the double
 * sum of the exact products (each bf16 x bf16 product is exact in double; the
 * double sum errs by at most H 2^-53 sum_h |x_h W_hn|, added to the radius).
 * The implementation under test accumulates in ascending h in steps of
 * O_STEP products (the tensor-core instruction depth for bf16), each step
 * D_s = D_{s-1} + (its products) rounded with an error of at most
 * O_STEP_ULPS units in the last place of the larger of |D_{s-1}| and the
 * step's sum of |products|; so its fp32 result lies within
 *     r = O_STEP_ULPS 2^-23 (sum_s |D_{s-1}| + sum_h |x_h W_hn|)
 * of g*.  (A sum rounded to nearest once per product, in any order, is
 * covered whenever the step error dominates; the oracle's own fmaf sum is
 * not assumed to lie in the range - its a is added to it explicitly.)
 * silu and the product are evaluated over [g* - r, g* + r] x [u* - r_u,
 * u* + r_u] in double, widened by (|g| + r + 8) 2^-22 relative for the
 * evaluation of exp, the division and the product on either side, and the
 * extremes rounded outward to bf16.
 * ========================================================================== */
#define O_STEP 16
#define O_STEP_ULPS 2.0
#define O_SILU_XMIN (-1.2784645427610738)       /* the minimum of x / (1 + e^-x) */

static double o_silu_d(double g) { return g / (1.0 + exp(-g)); }

/* bf16 value (bits) at or below v / at or above v: v to float rounded outward, then RNE. */
static uint16_t o_bf16_at_or_below(double v) {
  float f = (float)v;
  if ((double)f > v) f = nextafterf(f, -INFINITY);
  return o_f32_to_bf16(f);
}
static uint16_t o_bf16_at_or_above(double v) {
  float f = (float)v;
  if ((double)f < v) f = nextafterf(f, INFINITY);
  return o_f32_to_bf16(f);
}

/* For one token and one expert: a_lo[n], a_hi[n] (bf16 bits), the extreme bf16 values the
 * intermediate can take under the stated bound (always bracketing the oracle's own a);
 * g_out [2I] / rad_out [2I] (optional): the exact g (n < I) and u (n >= I) as doubles and
 * their radius r. */
void oracle_expert_h_range(int H, int I, const uint16_t* xrow, const uint16_t* W1e, int act,
                           uint16_t* a_lo, uint16_t* a_hi, double* g_out, double* rad_out) {
  double* acc = (double*)malloc(sizeof(double) * (size_t)(2 * I));
  double* sd = (double*)malloc(sizeof(double) * (size_t)(2 * I));    /* sum_s |D_{s-1}| */
  double* sp = (double*)malloc(sizeof(double) * (size_t)(2 * I));    /* sum_h |products| */
  float* facc = (float*)malloc(sizeof(float) * (size_t)(2 * I));     /* the oracle's own fp32 sums */
  for (int n = 0; n < 2 * I; ++n) { acc[n] = sd[n] = sp[n] = 0.0; facc[n] = 0.0f; }
  for (int h = 0; h < H; ++h) {
    if (h % O_STEP == 0)
      for (int n = 0; n < 2 * I; ++n) sd[n] += fabs(acc[n]);
    float xv = o_bf16_to_f32(xrow[h]);
    const uint16_t* wrow = W1e + (int64_t)h * 2 * I;
    for (int n = 0; n < 2 * I; ++n) {
      float wv = o_bf16_to_f32(wrow[n]);
      double p = (double)xv * (double)wv;
      acc[n] += p;
      sp[n] += fabs(p);
      facc[n] = fmaf(xv, wv, facc[n]);       /* the same steps as oracle_expert_ffn */
    }
  }
  for (int n = 0; n < 2 * I; ++n) {
    double r = O_STEP_ULPS * 0x1p-23 * (sd[n] + sp[n]) + (double)H * 0x1p-53 * sp[n];
    if (g_out) g_out[n] = acc[n];
    if (rad_out) rad_out[n] = r;
    sd[n] = r;
  }
  for (int n = 0; n < I; ++n) {
    float gf = facc[n], uf = facc[I + n];
    float v = (act == 0) ? (gf / (1.0f + expf(-gf))) * uf : gf * uf;   /* exactly the oracle's a */
    uint16_t a = o_f32_to_bf16(v);
    a_lo[n] = a_hi[n] = a;
    double g = acc[n], u = acc[I + n], rg = sd[n], ru = sd[I + n];
    if (!isfinite(g) || !isfinite(u) || !isfinite(v)) continue;
    double glo = g - rg, ghi = g + rg, ulo = u - ru, uhi = u + ru;
    double smin, smax, slack;
    if (act == 0) {
      double s1 = o_silu_d(glo), s2 = o_silu_d(ghi);
      smin = s1 < s2 ? s1 : s2;
      smax = s1 < s2 ? s2 : s1;
      if (glo < O_SILU_XMIN && O_SILU_XMIN < ghi) smin = o_silu_d(O_SILU_XMIN);
      slack = (fabs(g) + rg + 8.0) * 0x1p-22;
    } else {
      smin = glo;
      smax = ghi;
      slack = 0x1p-22;
    }
    double pr[4] = {smin * ulo, smin * uhi, smax * ulo, smax * uhi};
    double vlo = pr[0], vhi = pr[0];
    for (int i = 1; i < 4; ++i) {
      if (pr[i] < vlo) vlo = pr[i];
      if (pr[i] > vhi) vhi = pr[i];
    }
    double mag = fabs(vlo) > fabs(vhi) ? fabs(vlo) : fabs(vhi);
    vlo -= slack * mag;
    vhi += slack * mag;
    uint16_t lo = o_bf16_at_or_below(vlo), hi = o_bf16_at_or_above(vhi);
    if (o_bf16_to_f32(lo) < o_bf16_to_f32(a)) a_lo[n] = lo;
    if (o_bf16_to_f32(hi) > o_bf16_to_f32(a)) a_hi[n] = hi;
  }
  free(acc);
  free(sd);
  free(sp);
  free(facc);
}

/* Rows of several (token, expert) pairs, each with its own expert's weights: row i is token
 * toks[i] through expert W1p[i] / W2p[i] (oracle_expert_ffn: a_out [n][I] bf16 bits, o_out
 * [n][H] fp32).  With dlo/dhi [n][H] (double, may be NULL): the change of o that the flagged
 * intermediates can cause - for each flagged element, (a_lo - a) and (a_hi - a) times its
 * row of W2, the smaller and the larger summed separately; nflag[i] counts row i's flagged
 * elements, and a_lo_out / a_hi_out [n][I] (may be NULL) receive the ranges themselves. */
void oracle_expert_rows(int H, int I, int act, const uint16_t* x, int64_t n, const int64_t* toks,
                        const uint16_t* const* W1p, const uint16_t* const* W2p, uint16_t* a_out,
                        float* o_out, double* dlo, double* dhi, int32_t* nflag, uint16_t* a_lo_out,
                        uint16_t* a_hi_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    const uint16_t* xrow = x + toks[i] * H;
    float* scratch = (float*)malloc(sizeof(float) * (size_t)(2 * I));
    oracle_expert_ffn(H, I, xrow, W1p[i], W2p[i], act, a_out + i * I, o_out + i * H, scratch);
    free(scratch);
    if (!dlo) continue;
    uint16_t* lo = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    uint16_t* hi = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    oracle_expert_h_range(H, I, xrow, W1p[i], act, lo, hi, NULL, NULL);
    if (a_lo_out) memcpy(a_lo_out + i * I, lo, sizeof(uint16_t) * (size_t)I);
    if (a_hi_out) memcpy(a_hi_out + i * I, hi, sizeof(uint16_t) * (size_t)I);
    double* dl = dlo + i * H;
    double* dh = dhi + i * H;
    for (int m = 0; m < H; ++m) dl[m] = dh[m] = 0.0;
    int32_t cnt = 0;
    const uint16_t* a = a_out + i * I;
    for (int nn = 0; nn < I; ++nn) {
      if (lo[nn] == a[nn] && hi[nn] == a[nn]) continue;
      ++cnt;
      double d1 = (double)o_bf16_to_f32(lo[nn]) - (double)o_bf16_to_f32(a[nn]);
      double d2 = (double)o_bf16_to_f32(hi[nn]) - (double)o_bf16_to_f32(a[nn]);
      const uint16_t* wrow = W2p[i] + (int64_t)nn * H;
      for (int m = 0; m < H; ++m) {
        double wv = (double)o_bf16_to_f32(wrow[m]);
        double c1 = d1 * wv, c2 = d2 * wv;
        dl[m] += c1 < c2 ? c1 : c2;
        dh[m] += c1 < c2 ? c2 : c1;
      }
    }
    if (nflag) nflag[i] = cnt;
    free(lo);
    free(hi);
  }
}

/* Combine of ns tokens from their k slot outputs o [ns][k][H] and weights w [ns][k]: the same
 * fp32 slot-order sum as oracle_forward_tokens; y [ns][H] bf16 bits and y32 (the sum before
 * rounding).  With dlo/dhi [ns][k][H]: ylo/yhi = y32 + the smallest / largest change the
 * flagged intermediates of the k slots can cause, in double. */
void oracle_combine(int H, int k, int64_t ns, const float* w, const float* o, const double* dlo,
                    const double* dhi, uint16_t* y, float* y32, double* ylo, double* yhi) {
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < ns; ++s) {
    const float* os = o + s * k * H;
    const float* ws = w + s * k;
    for (int m = 0; m < H; ++m) {
      float acc = ws[0] * os[m];
      for (int j = 1; j < k; ++j) acc = acc + ws[j] * os[(int64_t)j * H + m];
      y[s * H + m] = o_f32_to_bf16(acc);
      if (y32) y32[s * H + m] = acc;
      if (dlo) {
        double lo = (double)acc, hi = (double)acc;
        for (int j = 0; j < k; ++j) {
          double wj = (double)ws[j];
          double c1 = wj * dlo[(s * k + j) * H + m], c2 = wj * dhi[(s * k + j) * H + m];
          lo += c1 < c2 ? c1 : c2;
          hi += c1 < c2 ? c2 : c1;
        }
        ylo[s * H + m] = lo;
        yhi[s * H + m] = hi;
      }
    }
  }
}
