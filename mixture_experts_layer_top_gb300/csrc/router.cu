// Router: logits in the canonical fp32 order, then top-k selection with
// softmax weights, and the per-expert row histogram.
//
// The layer is the MoE layer of the X-Stage paper's MegaMoE background
// paragraph: "a router selects one or more experts for each token" and
// Combine weights the top-k results by "the router weights".  The selection
// is a discrete decision, so the logits must be bitwise identical to an
// independent CPU evaluation; the library fixes one summation order:
//   partial j (j = 0..31) accumulates h = j, j+32, ... with fmaf in ascending h,
//   then the partials are added pairwise (j, j+16), (j, j+8), ..., (j, j+1).
// fp32 addition is commutative, so a warp xor-butterfly gives exactly that tree.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int RT_TOK = 32;    // tokens per CTA
constexpr int RT_EXP = 32;    // experts per CTA
constexpr int RT_HC = 128;    // h per staged chunk (4 x 32)
constexpr int RT_ROW = 40;    // bf16 elements per smem row (32 + 8 pad = 80 bytes, conflict-free 16 B reads)
constexpr int RT_THREADS = 512;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// One reduce-scatter step of the butterfly: lanes pair with lane ^ 2^S, each
// keeps half of its 2^(S+2) values and adds its partner's copy of that half.
// The pairs added are exactly (j, j ^ 2^S), i.e. the canonical tree level.
template <int S>
__device__ __forceinline__ void rs_step(float (&acc)[64], int lane) {
  constexpr int off = 1 << S;
  constexpr int half = 1 << (S + 1);
  const bool upper = (lane >> S) & 1;
#pragma unroll
  for (int i = 0; i < half; ++i) {
    const float send = upper ? acc[i] : acc[half + i];
    const float keep = upper ? acc[half + i] : acc[i];
    const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, off);
    acc[i] = keep + recv;
  }
}

// grid (ceil(T/32), ceil(E/32)), 512 threads = 16 warps; warp (tg, eg) owns
// tokens t0 + 8*tg .. +8 and experts e0 + 8*eg .. +8.  Lane L holds the
// partial sums of residue class h = L (mod 32) for all 64 of those outputs.
__global__ void __launch_bounds__(RT_THREADS, 1)
router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wr,
                     const float* __restrict__ bias, float* __restrict__ logits, int T, int H, int E) {
  __shared__ __align__(16) uint16_t xs[2][RT_HC][RT_ROW];   // x transposed: [h][token]
  __shared__ __align__(16) uint16_t ws[2][RT_HC][RT_ROW];   // Wr: [h][expert]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * RT_TOK, e0 = blockIdx.y * RT_EXP;
  const int tg = warp >> 2, eg = warp & 3;

  // staging roles: x: token = tid & 31, 8-element h chunk = tid >> 5 (16 chunks of 8 = 128)
  //                Wr: row = tid >> 2 (128 rows), 8-expert part = tid & 3
  const int xs_tok = tid & 31, xs_c = tid >> 5;
  const int ws_row = tid >> 2, ws_part = tid & 3;
  const bool x_ok = (t0 + xs_tok) < T;
  const int we = e0 + ws_part * 8;
  const bool w_full = (we + 8) <= E;
  const bool e_vec = (E % 8) == 0;

  auto load_x = [&](int h0) -> uint4 {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (x_ok) v = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + xs_tok) * H + h0 + xs_c * 8);
    return v;
  };
  auto load_w = [&](int h0) -> uint4 {
    uint4 v = make_uint4(0, 0, 0, 0);
    const uint16_t* src = Wr + (size_t)(h0 + ws_row) * E + we;
    if (w_full && e_vec) {
      v = *reinterpret_cast<const uint4*>(src);
    } else {
      uint16_t tmp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) tmp[i] = (we + i < E) ? src[i] : (uint16_t)0;
      v.x = tmp[0] | ((uint32_t)tmp[1] << 16);
      v.y = tmp[2] | ((uint32_t)tmp[3] << 16);
      v.z = tmp[4] | ((uint32_t)tmp[5] << 16);
      v.w = tmp[6] | ((uint32_t)tmp[7] << 16);
    }
    return v;
  };
  auto store_stage = [&](int buf, const uint4& xv, const uint4& wv) {
    const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xs[buf][xs_c * 8 + 2 * i][xs_tok] = (uint16_t)(u[i] & 0xFFFFu);
      xs[buf][xs_c * 8 + 2 * i + 1][xs_tok] = (uint16_t)(u[i] >> 16);
    }
    *reinterpret_cast<uint4*>(&ws[buf][ws_row][ws_part * 8]) = wv;
  };

  float acc[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.0f;

  const int nchunk = H / RT_HC;   // H is a multiple of 256
  uint4 xv = load_x(0), wv = load_w(0);
  store_stage(0, xv, wv);
  __syncthreads();
  for (int c = 0; c < nchunk; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunk) {
      xv = load_x((c + 1) * RT_HC);
      wv = load_w((c + 1) * RT_HC);
    }
#pragma unroll
    for (int i = 0; i < RT_HC / 32; ++i) {
      const int hr = i * 32 + lane;   // global h = c*128 + 32*i + lane  ==  lane (mod 32)
      float xf[8], wf[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(&xs[buf][hr][tg * 8]), xf);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(&ws[buf][hr][eg * 8]), wf);
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a * 8 + b] = __fmaf_rn(xf[a], wf[b], acc[a * 8 + b]);
    }
    if (c + 1 < nchunk) store_stage(buf ^ 1, xv, wv);
    __syncthreads();
  }

  // Reduce-scatter butterfly (see rs_step); lane L ends with outputs 2L, 2L+1.
  rs_step<4>(acc, lane);
  rs_step<3>(acc, lane);
  rs_step<2>(acc, lane);
  rs_step<1>(acc, lane);
  rs_step<0>(acc, lane);
  const int o = 2 * lane;
  const int t = t0 + tg * 8 + (o >> 3);
  const int e = e0 + eg * 8 + (o & 7);
  if (t < T) {
    float v0 = acc[0], v1 = acc[1];
    if (e < E) logits[(size_t)t * E + e] = bias ? v0 + bias[e] : v0;
    if (e + 1 < E) logits[(size_t)t * E + e + 1] = bias ? v1 + bias[e + 1] : v1;
  }
}

// Order-preserving key of a logit: higher logit -> larger key; -0 == +0; NaN -> 0
// (below -inf, whose key is 0x007FFFFF).
__device__ __forceinline__ uint32_t logit_key(float l) {
  if (l != l) return 0u;
  if (l == 0.0f) l = 0.0f;
  const uint32_t u = __float_as_uint(l);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per token.  Keys combine (logit key, 0xFFFF - expert) so the
// maximum is the highest logit and, among equal logits, the lowest id.
__global__ void __launch_bounds__(256)
topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
            float* __restrict__ w, int32_t* __restrict__ counts) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  uint64_t key[MAX_E / 32];
#pragma unroll
  for (int i = 0; i < MAX_E / 32; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? (((uint64_t)logit_key(l[e]) << 32) | (uint64_t)(0xFFFFu - (uint32_t)e)) : 0ull;
  }
  int my_e = 0;
  float my_l = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
      best = o > best ? o : best;
    }
    const int e = (int)(0xFFFFu - (uint32_t)(best & 0xFFFFu));
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i)
      if (key[i] == best) key[i] = 0ull;
    if (lane == j) {
      my_e = e;
      my_l = l[e];
    }
  }
  // weights: softmax over the k selected logits, exponentials and sum in fp64
  const double m = (double)__shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float ex = (lane < k) ? (float)exp((double)my_l - m) : 0.0f;
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += (double)__shfl_sync(0xFFFFFFFFu, ex, j);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_e;
    w[(size_t)t * k + lane] = (float)((double)ex / sum);
    atomicAdd(&counts[my_e], 1);
  }
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* Wr, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t st) {
  dim3 grid((T + RT_TOK - 1) / RT_TOK, (E + RT_EXP - 1) / RT_EXP);
  router_logits_kernel<<<grid, RT_THREADS, 0, st>>>(x, Wr, bias, logits, T, H, E);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                        cudaStream_t st) {
  topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, E, k, ids, w, counts);
  return cudaGetLastError();
}

}  // namespace moe
