// Router: logits in the canonical fp32 order, then top-k selection with
// softmax weights, and the per-expert row histogram.
//
// The layer is the MoE layer of the X-Stage paper's MegaMoE paragraph
// (introduction): each token is routed to its top-k experts, and Combine weights
// their outputs by the router's weights for that token.  The selection
// is a discrete decision, so the logits must be bitwise identical to an
// independent CPU evaluation; the library fixes one summation order:
//   partial j (j = 0..31) accumulates h = j, j+32, ... with fmaf in ascending h,
//   then the partials are added pairwise (j, j+16), (j, j+8), ..., (j, j+1).
// fp32 addition is commutative, so a warp xor-butterfly gives exactly that tree.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {

namespace {

constexpr int RT_TOK = 32;      // tokens per CTA
constexpr int RT_EXP = 32;      // experts per CTA
constexpr int RT_HC = 256;      // h per pipeline stage (8 x 32); the last stage of an H that is not a
                                // multiple of 256 holds zeros past H (a fused multiply-add of 0 * 0
                                // leaves a partial sum unchanged, so the canonical value is the same)
constexpr int RT_NS = 4;        // pipeline stages
constexpr int RT_XROW = RT_HC + 8;   // bf16 per staged x row (528 B; 16-B multiple, conflict-free reads)
constexpr int RT_WROW = RT_EXP + 8;  // bf16 per staged Wr row (80 B; conflict-free 16-B reads)
constexpr int RT_STAGE_X = RT_TOK * RT_XROW;   // elements
constexpr int RT_STAGE_W = RT_HC * RT_WROW;
constexpr int RT_SMEM = RT_NS * (RT_STAGE_X + RT_STAGE_W) * 2;
constexpr int RT_THREADS = 512;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
// partial sums of residue class h = L (mod 32) for all 64 of those outputs,
// each accumulated with one rounded fused multiply-add per h in ascending h
// (two outputs per packed f32x2 FMA).  x and Wr chunks of 256 h stream through
// a 4-stage cp.async ring in shared memory.
__global__ void __launch_bounds__(RT_THREADS, 1)
router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wr,
                     const float* __restrict__ bias, float* __restrict__ logits, int T, int H, int E) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  extern __shared__ __align__(16) uint16_t rsm[];
  uint16_t* xs = rsm;                               // [NS][32 tok][XROW]
  uint16_t* ws = rsm + RT_NS * RT_STAGE_X;          // [NS][HC][WROW]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * RT_TOK, e0 = blockIdx.y * RT_EXP;
  const int tg = warp >> 2, eg = warp & 3;

  // copy roles, RT_HC / 128 rounds per stage: x chunk q = tid + 512 j is token q / XCH,
  // 8-element chunk q % XCH; Wr chunk q is row q / 4, 8-expert part q % 4
  constexpr int XCH = RT_HC / 8;
  const int we_base = e0;
  const bool w_vec = (E % 8) == 0;

  auto issue = [&](int chunk) {
    const int st = chunk % RT_NS;
    const int h0 = chunk * RT_HC;
#pragma unroll
    for (int j = 0; j < RT_HC / 128; ++j) {
      const int q = tid + RT_THREADS * j;
      const int tok = q / XCH, c = q % XCH;
      const bool x_ok = (t0 + tok) < T && h0 + c * 8 < H;
      cp_async16(xs + st * RT_STAGE_X + tok * RT_XROW + c * 8, x_ok ? x + (size_t)(t0 + tok) * H + h0 + c * 8 : x,
                 x_ok);
      const int row = q >> 2, part = q & 3;
      const int we = we_base + part * 8;
      uint16_t* wdst = ws + st * RT_STAGE_W + row * RT_WROW + part * 8;
      const bool h_ok = h0 + row < H;
      const uint16_t* wsrc = Wr + (size_t)(h_ok ? h0 + row : 0) * E + we;
      if (w_vec) {
        cp_async16(wdst, (we < E && h_ok) ? wsrc : Wr, we < E && h_ok);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) wdst[i] = (we + i < E && h_ok) ? wsrc[i] : (uint16_t)0;
      }
    }
  };

  float2 acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.0f, 0.0f);

  const int nchunk = (H + RT_HC - 1) / RT_HC;
#pragma unroll
  for (int c = 0; c < RT_NS - 1; ++c) {
    if (c < nchunk) issue(c);
    cp_async_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    if (c + RT_NS - 1 < nchunk) issue(c + RT_NS - 1);
    cp_async_commit();
    cp_async_wait<RT_NS - 1>();
    __syncthreads();
    const uint16_t* xb = xs + (c % RT_NS) * RT_STAGE_X + (tg * 8) * RT_XROW;
    const uint16_t* wb = ws + (c % RT_NS) * RT_STAGE_W + eg * 8;
#pragma unroll
    for (int i = 0; i < RT_HC / 32; ++i) {
      const int hr = i * 32 + lane;   // global h = c*RT_HC + 32*i + lane == lane (mod 32)
      const uint4 wv = *reinterpret_cast<const uint4*>(wb + hr * RT_WROW);
      const float2 w01 = make_float2(__uint_as_float(wv.x << 16), __uint_as_float(wv.x & 0xFFFF0000u));
      const float2 w23 = make_float2(__uint_as_float(wv.y << 16), __uint_as_float(wv.y & 0xFFFF0000u));
      const float2 w45 = make_float2(__uint_as_float(wv.z << 16), __uint_as_float(wv.z & 0xFFFF0000u));
      const float2 w67 = make_float2(__uint_as_float(wv.w << 16), __uint_as_float(wv.w & 0xFFFF0000u));
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float xf = __uint_as_float((uint32_t)xb[a * RT_XROW + hr] << 16);
        const float2 xx = make_float2(xf, xf);
        acc[a * 4 + 0] = __ffma2_rn(xx, w01, acc[a * 4 + 0]);
        acc[a * 4 + 1] = __ffma2_rn(xx, w23, acc[a * 4 + 1]);
        acc[a * 4 + 2] = __ffma2_rn(xx, w45, acc[a * 4 + 2]);
        acc[a * 4 + 3] = __ffma2_rn(xx, w67, acc[a * 4 + 3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  float f[64];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    f[2 * i] = acc[i].x;
    f[2 * i + 1] = acc[i].y;
  }
  // Reduce-scatter butterfly (see rs_step); lane L ends with outputs 2L, 2L+1
  // (output o = 8 * token + expert within the warp's 8 x 8 tile).
  rs_step<4>(f, lane);
  rs_step<3>(f, lane);
  rs_step<2>(f, lane);
  rs_step<1>(f, lane);
  rs_step<0>(f, lane);
  const int o = 2 * lane;
  const int t = t0 + tg * 8 + (o >> 3);
  const int e = e0 + eg * 8 + (o & 7);
  if (t < T) {
    const float v0 = f[0], v1 = f[1];
    if (e < E) logits[(size_t)t * E + e] = bias ? v0 + bias[e] : v0;
    if (e + 1 < E) logits[(size_t)t * E + e + 1] = bias ? v1 + bias[e + 1] : v1;
  }
}

constexpr int TK_WARPS = 8;
constexpr int TK_MAX_TOK_PER_WARP = 8;
static_assert(TK_WARPS * TK_MAX_TOK_PER_WARP <= DS_CHUNK_TOK, "a block's tokens span two chunks at most");

// Top-k over caller-given (or canonical) logits: one warp per token, tpw tokens
// per warp in turn; selection and weights as in routing.cuh.  Expert counts go
// through a shared-memory histogram, one global atomic per (block, expert).
__global__ void __launch_bounds__(TK_WARPS * 32)
topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
            float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ chist, int tpw) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  __shared__ int32_t hist[2][MAX_E];   // expert counts of the block's tokens in its first / second chunk
  for (int i = threadIdx.x; i < 2 * MAX_E; i += blockDim.x) hist[i / MAX_E][i % MAX_E] = 0;
  __syncthreads();
  const int c_first = (blockIdx.x * tpw * TK_WARPS) / DS_CHUNK_TOK;   // tpw * TK_WARPS <= DS_CHUNK_TOK
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nkey = (E + 31) >> 5;
  for (int it = 0; it < tpw; ++it) {
    const int t = (blockIdx.x * tpw + it) * TK_WARPS + warp;
    if (t >= T) break;
    const float* l = logits + (size_t)t * E;
    uint64_t key[MAX_E / 32];
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int e = lane + 32 * i;
      key[i] = (i < nkey && e < E) ? select_key(l[e], e) : 0ull;
    }
    const int my_e = warp_select_topk(key, k, lane);
    const float my_l = (lane < k) ? l[my_e] : 0.0f;
    const float wt = warp_softmax_weight(my_l, k, lane);
    if (lane < k) {
      ids[(size_t)t * k + lane] = my_e;
      w[(size_t)t * k + lane] = wt;
      atomicAdd(&hist[t / DS_CHUNK_TOK - c_first][my_e], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int h0 = hist[0][i], h1 = hist[1][i];
    if (h0 + h1) atomicAdd(&counts[i], h0 + h1);
    if (h0) atomicAdd(&chist[(size_t)c_first * E + i], h0);
    if (h1) atomicAdd(&chist[(size_t)(c_first + 1) * E + i], h1);
  }
}

}  // namespace

cudaError_t router_prepare() {
  return cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RT_SMEM);
}

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* Wr, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t st) {
  dim3 grid((T + RT_TOK - 1) / RT_TOK, (E + RT_EXP - 1) / RT_EXP);
  return launch_pdl(router_logits_kernel, grid, dim3(RT_THREADS), RT_SMEM, st, x, Wr, bias, logits, T, H, E);
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                        int32_t* chist, int num_sms, cudaStream_t st) {
  // tokens per warp: enough blocks for two per SM, up to TK_MAX_TOK_PER_WARP tokens each
  int tpw = (T + 2 * num_sms * TK_WARPS - 1) / (2 * num_sms * TK_WARPS);
  tpw = tpw < 1 ? 1 : (tpw > TK_MAX_TOK_PER_WARP ? TK_MAX_TOK_PER_WARP : tpw);
  const int per_block = tpw * TK_WARPS;
  return launch_pdl(topk_kernel, dim3((T + per_block - 1) / per_block), dim3(TK_WARPS * 32), 0, st, logits, T, E, k, ids,
                    w, counts, chist, tpw);
}

}  // namespace moe
