// Warp-level pieces of the top-k selection shared by the router kernels:
// order-preserving logit keys, the k-round warp arg-max, and the renormalised
// softmax weights of the selected logits.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace moe {

// Order-preserving key of a logit: higher logit -> larger key; -0 == +0; NaN -> 0
// (below -inf, whose key is 0x007FFFFF).
__device__ __forceinline__ uint32_t logit_key(float l) {
  if (l != l) return 0u;
  if (l == 0.0f) l = 0.0f;
  const uint32_t u = __float_as_uint(l);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selection key of expert e: (logit key, 0xFFFF - e), so the maximum is the highest
// logit and, among equal logits, the lowest id.  Key 0 never wins over a real key.
__device__ __forceinline__ uint64_t select_key(float l, int e) {
  return ((uint64_t)logit_key(l) << 32) | (uint64_t)(0xFFFFu - (uint32_t)e);
}

// k rounds of warp arg-max over key[] (lane holds experts lane + 32 i): lane j < k
// receives the expert of rank j.  Selected keys are cleared.
template <int NK>
__device__ __forceinline__ int warp_select_topk(uint64_t (&key)[NK], int k, int lane) {
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < NK; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
      best = o > best ? o : best;
    }
#pragma unroll
    for (int i = 0; i < NK; ++i)
      if (key[i] == best) key[i] = 0ull;
    if (lane == j) my_e = (int)(0xFFFFu - (uint32_t)(best & 0xFFFFu));
  }
  return my_e;
}

// The k-th largest key over the warp (k >= 1), in every lane; the k largest are cleared.
template <int NK>
__device__ __forceinline__ uint64_t warp_kth_key(uint64_t (&key)[NK], int k) {
  uint64_t best = 0;
  for (int j = 0; j < k; ++j) {
    best = 0;
#pragma unroll
    for (int i = 0; i < NK; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
      best = o > best ? o : best;
    }
#pragma unroll
    for (int i = 0; i < NK; ++i)
      if (key[i] == best) key[i] = 0ull;
  }
  return best;
}

// Inverse of logit_key for non-NaN logits (-0 comes back as +0).
__device__ __forceinline__ float key_logit(uint32_t kk) {
  return __uint_as_float((kk & 0x80000000u) ? (kk & 0x7FFFFFFFu) : ~kk);
}

// Exact a - b as hi + lo (Knuth's two-sum); lo = 0 when hi is not finite.
__device__ __forceinline__ float two_diff(float a, float b, float* lo) {
  const float hi = __fsub_rn(a, b);
  if (!isfinite(hi)) {
    *lo = 0.0f;
    return hi;
  }
  const float bb = __fsub_rn(hi, a);
  *lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(-b, bb));
  return hi;
}

// Weight of this lane's slot (lanes 0..k-1 hold the selected logits in rank
// order): softmax over the k selected logits, relative to the first.  fp32, with
// the argument l_j - l_0 kept exact as a two-term sum (exp(hi + lo) =
// exp(hi)(1 + lo) to first order, lo <= half an ulp of hi) and the slot-order sum
// compensated (Neumaier), so each weight is within a few 1e-7 relative of the
// exactly rounded softmax without fp64 (whose rate on this GPU is a small
// fraction of fp32).
__device__ __forceinline__ float warp_softmax_weight(float my_l, int k, int lane) {
  const float m = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  float lo;
  const float hi = two_diff(my_l, m, &lo);
  const float eh = expf(hi);
  const float ex = (lane < k) ? __fmaf_rn(eh, lo, eh) : 0.0f;
  float sum = 0.0f, comp = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float v = __shfl_sync(0xFFFFFFFFu, ex, j);
    const float s2 = __fadd_rn(sum, v);
    comp = __fadd_rn(comp, fabsf(sum) >= fabsf(v) ? __fadd_rn(__fsub_rn(sum, s2), v)
                                                 : __fadd_rn(__fsub_rn(v, s2), sum));
    sum = s2;
  }
  if (isfinite(sum)) sum = __fadd_rn(sum, comp);
  return __fdiv_rn(ex, sum);
}

}  // namespace moe
