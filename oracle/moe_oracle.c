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
