// Router on the tensor cores with a certified, exact top-k.
//
// The MoE layer of the X-Stage paper's MegaMoE paragraph (introduction) sends
// each token to the experts its router picks; that choice is discrete,
// so this library fixes one canonical fp32 order for the logits (lane-strided
// partial sums, then a pairwise tree; router.cu) and routes on exactly those
// values.  Evaluating every logit that way costs T*H*E FMAs on the CUDA cores.
// This path gets the same routing from far fewer of them:
//
//  1. router_prep_kernel: WrT = Wr^T (expert-major rows, for K-major tensor-core
//     tiles and coalesced per-expert reads).
//  2. router_tc_kernel: estimates L~[t,e] = sum_h x[t,h] Wr[h,e] with tcgen05
//     (bf16 products are exact in fp32; accumulation in TMEM).  The K blocks are
//     dealt round-robin to A independent TMEM accumulators (chains) per CTA and K
//     is split over S CTAs; the epilogue adds its A chains and the S partial sums
//     are added by the select kernel, both in a fixed order.  Its epilogue warps,
//     idle during the mainloop, write upper bounds nw[e] >= ||Wr[:,e]||_2.
//  3. router_select_kernel (one warp per token): nx >= ||x[t,:]||_2 and, for every
//     expert, a bound d[e] >= |L~[t,e] - L[t,e]| where L is the canonical logit:
//        d[e] = cH * nx * nw[e] + 2^-20 (|L~[t,e]| + |bias[e]|),
//        cH = (n + 1) 2^-17 + (A S + H/32 + 8) 2^-22,  n = MMA steps of the longest chain.
//     Model: one 16-deep MMA step D' = D + sum of 16 exact products errs by at most
//     2^-17 (|D| + sum |products|) (several times the error of an adder that aligns
//     the 17 addends to the largest and keeps 24 bits of each).  Along a chain |D|
//     never exceeds the chain's sum of |products| S_c, so a chain of n steps errs by
//     at most (n + 1) 2^-17 S_c; over all chains that is (n + 1) 2^-17 sum_h |x_h w_h|.
//     The A S - 1 fp32 additions of chain values, the canonical order's own
//     rounding (H/32 fused multiply-adds per partial, 5 tree additions) and slack
//     make the second term; sum_h |x_h w_h| <= ||x|| ||w|| (Cauchy-Schwarz), and
//     2^-20 (...) covers the bias additions.  Short chains keep the bound tight,
//     so few experts need the canonical evaluation.
//     With theta = the k-th largest of L~ - d, an expert with L~[e] + d[e] < theta
//     has k experts certainly above it and cannot be selected; every other
//     expert (the candidates, at least k of them) gets its canonical logit
//     recomputed (same order as router.cu), and the top-k, ties and weights are
//     taken on those exact values.  A token whose estimates or bounds are not
//     finite (NaN/Inf in x, Wr or the bias) recomputes all E logits.
//     The logits row written out holds the canonical value for every candidate
//     (so for every selected expert) and the estimate L~ + bias elsewhere.
#include <cuda.h>
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {

namespace {

// ------------------------------------------------------------------ 1. prep
constexpr int RP_H = 64;    // h rows per block

// grid (ceil(E/32), H/64), 256 threads: WrT[e0 .. e0+31][h0 .. h0+63] = Wr[h0.., e0..]^T.
__global__ void __launch_bounds__(256)
router_prep_kernel(const uint16_t* __restrict__ Wr, int H, int E, uint16_t* __restrict__ WrT) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  __shared__ __align__(16) uint16_t tile[32][RP_H + 8];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int e0 = blockIdx.x * 32, h0 = blockIdx.y * RP_H;
  const int e = e0 + tx;
#pragma unroll
  for (int r = ty; r < RP_H; r += 8) tile[tx][r] = (e < E) ? Wr[(size_t)(h0 + r) * E + e] : (uint16_t)0;
  __syncthreads();
  const int i = threadIdx.x >> 3, c = threadIdx.x & 7;   // expert row i, 8-element chunk c
  if (e0 + i < E)
    *reinterpret_cast<uint4*>(WrT + (size_t)(e0 + i) * H + h0 + c * 8) =
        *reinterpret_cast<const uint4*>(&tile[i][c * 8]);
}

// ------------------------------------------------------------------ 2. tensor-core estimate
constexpr int RTC_BM = 128;                  // tokens per CTA
constexpr int RTC_BK = 64;                   // K per stage (one 128-byte swizzle row)
constexpr int RTC_NST = 4;
constexpr int RTC_A_BYTES = RTC_BM * RTC_BK * 2;          // 16 KB
constexpr int RTC_B_MAX = 256 * RTC_BK * 2;               // 32 KB (N <= 256 experts)
constexpr int RTC_STAGE = RTC_A_BYTES + RTC_B_MAX;
constexpr int RTC_THREADS = 192;             // producer, MMA, 4 epilogue warps
constexpr int RTC_TMEM_COLS = 512;          // A chains x (128 or 256) columns

struct RtcCtl {
  uint64_t full[RTC_NST];
  uint64_t empty[RTC_NST];
  uint64_t acc;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int RTC_CTL_OFF = RTC_NST * RTC_STAGE;
constexpr int RTC_SMEM = RTC_CTL_OFF + 256 + 1024;
static_assert(sizeof(RtcCtl) <= 256, "control block exceeds its reservation");
static_assert(RTC_SMEM <= 232448, "shared memory per CTA exceeded");

// grid (ceil(T/128), S).  CTA (m, s): tokens [128 m, +128) x all experts (N = n_pad
// columns), K blocks [s*kb_per, min(kb_total, (s+1)*kb_per)), the j-th of them
// accumulated into chain j mod n_chain (TMEM columns [chain * cstride, + n_pad)).
// A = x tile (K-major), B = WrT tile (K-major, rows beyond E zero-filled by TMA).
// The epilogue warps (one token row per thread) add the chains in order and write
// part[s][t][e].
__global__ void __launch_bounds__(RTC_THREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const uint16_t* __restrict__ WrT, int T, int H, int E, int n_pad, int kb_total, int kb_per,
                 int n_chain, float* __restrict__ part, float* __restrict__ nw, uint32_t* __restrict__ err,
                 int64_t tmo) {
  extern __shared__ uint8_t rtc_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rtc_raw) + 1023) & ~(uintptr_t)1023);
  RtcCtl* ctl = reinterpret_cast<RtcCtl*>(smem + RTC_CTL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * RTC_BM, s = blockIdx.y;
  const int kb0 = s * kb_per;
  const int kb1 = min(kb_total, kb0 + kb_per);
  const uint32_t b_bytes = (uint32_t)n_pad * RTC_BK * 2;
  const uint32_t cstride = n_pad <= 128 ? 128u : 256u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RTC_NST; ++i) {
      ptx::mbar_init(&ctl->full[i], 1);
      ptx::mbar_init(&ctl->empty[i], 1);
    }
    ptx::mbar_init(&ctl->acc, 1);
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmX);
    ptx::tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    ptx::tmem_alloc<RTC_TMEM_COLS>(&ctl->tmem_base);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;
  ptx::grid_dep_wait();   // the transposed router weight is visible from here on

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, tmo, abort_flag)) {
          atomicOr(err, ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* sa = smem + stage * RTC_STAGE;
        ptx::mbar_arrive_expect_tx(&ctl->full[stage], RTC_A_BYTES + b_bytes);
        ptx::tma_load_2d(&tmX, &ctl->full[stage], sa, kb * RTC_BK, m0, pol);
        ptx::tma_load_2d(&tmW, &ctl->full[stage], sa + RTC_A_BYTES, kb * RTC_BK, 0, pol);
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == RTC_NST) { stage = 0; phase ^= 1u; }
      }
      // no copy may still be landing when the CTA exits
      int dummy = 0;
      for (int i = 0; i < RTC_NST; ++i)
        if (issued & (1u << i)) ptx::mbar_wait(&ctl->full[i], (last_par >> i) & 1u, tmo, &dummy);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(RTC_BM, (uint32_t)n_pad, false);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait(&ctl->full[stage], phase, tmo, abort_flag)) {
          atomicOr(err, ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(smem + stage * RTC_STAGE);
        const uint32_t b0 = a0 + RTC_A_BYTES;
#pragma unroll
        for (int kk = 0; kk < RTC_BK / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
          const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 32, 16, 1024);
          const int j = kb - kb0;
          ptx::mma_bf16(tmem_base + (uint32_t)(j % n_chain) * cstride, ad, bd, idesc,
                        (j >= n_chain || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&ctl->empty[stage]);
        if (++stage == RTC_NST) { stage = 0; phase ^= 1u; }
      }
      ptx::mma_commit(&ctl->acc);   // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    {
      // while the mainloop runs: nw[e] >= ||Wr[:,e]||_2 for experts e = cta + n_cta * (q + 4 i),
      // one warp per expert (lane-strided sums of squares, then the xor tree), rounded up by
      // more than the relative error of the additions and of the square root
      const int n_cta = (int)(gridDim.x * gridDim.y), cta = (int)(blockIdx.y * gridDim.x + blockIdx.x);
      const float up = 1.0f + (float)H * 0x1p-21f;
      for (int e = cta + n_cta * (warp - 2); e < E; e += 4 * n_cta) {
        const uint16_t* wr = WrT + (size_t)e * H;
        float ss = 0.0f;
#pragma unroll 4
        for (int h = lane * 8; h < H; h += 256) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(wr + h));
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(u[j] << 16), hi = __uint_as_float(u[j] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
        if (lane == 0) nw[e] = sqrtf(ss) * up;
      }
    }
    const bool ok = ptx::mbar_wait(&ctl->acc, 0, tmo, abort_flag);
    if (!ok) {
      atomicOr(err, ERR_TIMEOUT);
      *abort_flag = 1;
    }
    ptx::tc_fence_after();
    const bool write = ok && !*abort_flag;
    const int t = m0 + q * 32 + lane;
    float* prow = part + ((size_t)s * T + t) * E;
    const bool vec = (E & 3) == 0;
    const int used = min(n_chain, kb1 - kb0);   // chains that received at least one K block
    for (int c = 0; c < n_pad; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
      ptx::tmem_ld_wait();
      for (int a = 1; a < used; ++a) {
        uint32_t u[32];
        ptx::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + a * cstride + (uint32_t)c, u);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(u[j]));
      }
      if (!write || t >= T) continue;
      if (vec && c + 32 <= E) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          reinterpret_cast<float4*>(prow + c)[j] =
              make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                          __uint_as_float(v[4 * j + 3]));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < E) prow[c + j] = __uint_as_float(v[j]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<RTC_TMEM_COLS>(tmem_base);
  }
}

// ------------------------------------------------------------------ 3. certified selection
constexpr int SEL_WARPS = 8;
static_assert(SEL_WARPS <= DS_CHUNK_TOK, "a block's tokens span two chunks at most");

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// p_lo = fma(x_lo, w_lo, p_lo), p_hi = fma(x_hi, w_hi, p_hi) on the two bf16 halves
// of x and w, each with one rounding to fp32 (the product of two bf16 values is
// exact, so this is fmaf on the widened values).
__device__ __forceinline__ void fma_bf16x2(uint32_t x, uint32_t w, float& p_lo, float& p_hi) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "mov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
      "fma.rn.f32.bf16 %1, xh, wh, %1;\n\t}"
      : "+f"(p_lo), "+f"(p_hi)
      : "r"(x), "r"(w));
}

// Canonical logit of (token row xr, expert row wr) computed by the 4 lanes of a
// group: lane `sub` holds partials 8 sub .. 8 sub + 7 (partial j sums h = j (mod 32)
// in ascending h with one fused multiply-add each); the tree then adds partial
// pairs (j, j+16), (j, j+8), (j, j+4), (j, j+2), (j, j+1) - lanes sub^2 and sub^1
// for the first two levels, inside the lane for the rest.  Every lane of the
// group returns the same value.
template <bool H_TAIL>
__device__ __forceinline__ float canonical_dot(const uint16_t* __restrict__ xr, const uint16_t* __restrict__ wr,
                                               int H, int sub) {
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = 0.0f;
  // trips of four 32-wide steps, two trips per iteration over the first H256 = H - H mod 256 h,
  // the next trip's loads issued before this trip's fused multiply-adds; then (H_TAIL: H not a
  // multiple of 256, a separate instance so the measured loop above keeps its registers) the
  // remaining 32-wide steps, still in ascending h
  const int H256 = H_TAIL ? (H & ~255) : H;
  uint4 xa[4], wa[4], xb[4], wb[4];
  auto load = [&](uint4 (&xv)[4], uint4 (&wv)[4], int h) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      xv[u] = __ldg(reinterpret_cast<const uint4*>(xr + h + 32 * u));
      wv[u] = __ldg(reinterpret_cast<const uint4*>(wr + h + 32 * u));
    }
  };
  auto fma_trip = [&](const uint4 (&xv)[4], const uint4 (&wv)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      fma_bf16x2(xv[u].x, wv[u].x, p[0], p[1]);
      fma_bf16x2(xv[u].y, wv[u].y, p[2], p[3]);
      fma_bf16x2(xv[u].z, wv[u].z, p[4], p[5]);
      fma_bf16x2(xv[u].w, wv[u].w, p[6], p[7]);
    }
  };
  if (!H_TAIL || H256 > 0) {
    load(xa, wa, 8 * sub);
    for (int h = 8 * sub; h < H256; h += 256) {
      load(xb, wb, h + 128);
      fma_trip(xa, wa);
      if (h + 256 < H256) load(xa, wa, h + 256);
      fma_trip(xb, wb);
    }
  }
  if (H_TAIL) {
    for (int h = H256 + 8 * sub; h < H; h += 32) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + h));
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wr + h));
      fma_bf16x2(xv.x, wv.x, p[0], p[1]);
      fma_bf16x2(xv.y, wv.y, p[2], p[3]);
      fma_bf16x2(xv.z, wv.z, p[4], p[5]);
      fma_bf16x2(xv.w, wv.w, p[6], p[7]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = __fadd_rn(p[j], __shfl_xor_sync(0xFFFFFFFFu, p[j], 2));
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = __fadd_rn(p[j], __shfl_xor_sync(0xFFFFFFFFu, p[j], 1));
#pragma unroll
  for (int j = 0; j < 4; ++j) p[j] = __fadd_rn(p[j], p[j + 4]);
#pragma unroll
  for (int j = 0; j < 2; ++j) p[j] = __fadd_rn(p[j], p[j + 2]);
  return __fadd_rn(p[0], p[1]);
}

// Block of SEL_WARPS warps, tokens [tb * ntok, +ntok) (ntok <= SEL_WARPS), warp w
// owning token w: (1) bounds and candidates per token (the row's loads all in flight
// at once); (2) the block's warps evaluate every (token, candidate) pair together,
// 8 pairs per warp at a time; (3) each warp ranks its token's candidates on the
// exact values (one pass over them when there are at most 32, k rounds of warp
// arg-max over all experts otherwise).  E <= 32 NK.
// Resident blocks per SM: the kernel is latency-bound (memory waits on the canonical
// re-evaluation's loads), so occupancy helps where the registers allow it: 4 blocks (64
// registers) for E <= 128 measured faster than 3 (80 registers) - fine workload 68 -> 64 us -
// while for E = 256 the 64-register build spills in the hot loop and 3 blocks stay faster
// (large layer 121-128 vs 136-144 us).
template <int NK, bool H_TAIL>
__global__ void __launch_bounds__(SEL_WARPS * 32, (NK <= 4) ? 4 : 3)
router_select_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ WrT, const float* __restrict__ part,
                     int S, const float* __restrict__ nw, const float* __restrict__ bias, int T, int H, int E, int k,
                     float cH, int ntok, float* __restrict__ logits, int32_t* __restrict__ ids,
                     float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ chist) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  __shared__ int32_t hist[2][NK * 32];   // expert counts of the block's tokens in its first / second chunk
  __shared__ float lg[SEL_WARPS][NK * 32];
  __shared__ int16_t cl[SEL_WARPS][NK * 32];
  __shared__ int32_t top[SEL_WARPS][MAX_K];
  __shared__ int pref[SEL_WARPS + 1];
  for (int i = threadIdx.x; i < 2 * NK * 32; i += blockDim.x) hist[i / (NK * 32)][i % (NK * 32)] = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * ntok + warp;
  const int c_first = (blockIdx.x * ntok) / DS_CHUNK_TOK;   // ntok <= DS_CHUNK_TOK: two chunks at most
  const bool has_tok = warp < ntok && t < T;
  float* my_lg = lg[warp];
  int16_t* my_cl = cl[warp];
  bool cand[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i) cand[i] = false;
  int ncand = 0;
  if (has_tok) {
    // nx >= ||x_t||_2, 8 loads in flight per lane (they also bring the row into L1 for (2))
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int n16 = H / 8;
    float ss = 0.0f;
    for (int m0 = lane; m0 < n16; m0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (m0 + 32 * u < n16) v[u] = __ldg(xr + m0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (m0 + 32 * u < n16) {
          const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ss = fmaf(bf16_lo(q[j]), bf16_lo(q[j]), ss);
            ss = fmaf(bf16_hi(q[j]), bf16_hi(q[j]), ss);
          }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    const float nx = sqrtf(ss) * (1.0f + (float)H * 0x1p-21f);
    // estimates and their bounds
    float lo_b[NK], hi_b[NK], vs[NK];
    bool bad = !isfinite(nx);
#pragma unroll
    for (int i = 0; i < NK; ++i) vs[i] = 0.0f;
#pragma unroll 4
    for (int sp = 0; sp < S; ++sp) {   // split partials in a fixed order, many loads in flight
      const float* pp = part + ((size_t)sp * T + t) * E;
#pragma unroll
      for (int i = 0; i < NK; ++i)
        if (lane + 32 * i < E) vs[i] += __ldcs(pp + lane + 32 * i);
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int e = lane + 32 * i;
      lo_b[i] = 0.0f;
      hi_b[i] = 0.0f;
      if (e < E) {
        const float v = vs[i];
        const float b = bias ? bias[e] : 0.0f;
        const float est = bias ? v + b : v;
        const float d = cH * nx * nw[e] + 0x1p-20f * (fabsf(v) + fabsf(b)) + 0x1p-120f;
        bad = bad || !isfinite(est) || !isfinite(d);
        lo_b[i] = est - d;
        hi_b[i] = est + d;
        my_lg[e] = est;
      }
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    // candidates: every expert not certainly beaten by k others
    if (!bad) {
      uint64_t key[NK];
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        const int e = lane + 32 * i;
        key[i] = (e < E) ? select_key(lo_b[i], e) : 0ull;
      }
      const float theta = key_logit((uint32_t)(warp_kth_key(key, k) >> 32));
#pragma unroll
      for (int i = 0; i < NK; ++i) cand[i] = (lane + 32 * i < E) && hi_b[i] >= theta;
    } else {
#pragma unroll
      for (int i = 0; i < NK; ++i) cand[i] = (lane + 32 * i < E);
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, cand[i]);
      if (cand[i]) my_cl[ncand + __popc(m & ((1u << lane) - 1u))] = (int16_t)(lane + 32 * i);
      ncand += __popc(m);
    }
  }
  if (lane == 0) pref[warp + 1] = ncand;
  __syncthreads();
  if (threadIdx.x == 0) {
    pref[0] = 0;
    for (int i = 1; i <= SEL_WARPS; ++i) pref[i] += pref[i - 1];
  }
  __syncthreads();
  // canonical logits of every (token, candidate) pair of the block, 8 per warp at a time
  const int total = pref[SEL_WARPS];
  const int grp = lane >> 2, sub = lane & 3;
  for (int base = warp * 8; base < total; base += SEL_WARPS * 8) {
    const int pi = base + grp;
    const int q = pi < total ? pi : base;   // idle lanes repeat a real pair (result unused)
    int slot = 0;
#pragma unroll
    for (int i = 1; i < SEL_WARPS; ++i) slot += (q >= pref[i]) ? 1 : 0;
    const int e = cl[slot][q - pref[slot]];
    const int tt = blockIdx.x * ntok + slot;
    float l = canonical_dot<H_TAIL>(x + (size_t)tt * H, WrT + (size_t)e * H, H, sub);
    if (bias) l = __fadd_rn(l, bias[e]);
    if (pi < total && sub == 0) lg[slot][e] = l;
  }
  __syncthreads();
  if (has_tok) {
    // exact top-k among the candidates (keys are distinct: the expert id is part of them)
    int my_e = 0;
    if (ncand <= 32) {
      const bool act = lane < ncand;
      const int e = act ? my_cl[lane] : 0;
      const uint64_t key = act ? select_key(my_lg[e], e) : 0ull;
      int rank = 0;
      for (int j = 0; j < ncand; ++j) rank += (__shfl_sync(0xFFFFFFFFu, key, j) > key) ? 1 : 0;
      if (act && rank < k) top[warp][rank] = e;
      __syncwarp();
      if (lane < k) my_e = top[warp][lane];
    } else {
      uint64_t key[NK];
#pragma unroll
      for (int i = 0; i < NK; ++i) key[i] = cand[i] ? select_key(my_lg[lane + 32 * i], lane + 32 * i) : 0ull;
      my_e = warp_select_topk(key, k, lane);
    }
    const float my_l = (lane < k) ? my_lg[my_e] : 0.0f;
    const float wt = warp_softmax_weight(my_l, k, lane);
    if (lane < k) {
      ids[(size_t)t * k + lane] = my_e;
      w[(size_t)t * k + lane] = wt;
      atomicAdd(&hist[t / DS_CHUNK_TOK - c_first][my_e], 1);
    }
    for (int e = lane; e < E; e += 32) logits[(size_t)t * E + e] = my_lg[e];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int h0 = hist[0][i], h1 = hist[1][i];
    if (h0 + h1) atomicAdd(&counts[i], h0 + h1);
    if (h0) atomicAdd(&chist[(size_t)c_first * E + i], h0);
    if (h1) atomicAdd(&chist[(size_t)(c_first + 1) * E + i], h1);
  }
}

template <int NK>
cudaError_t launch_select(dim3 grid, cudaStream_t st, const uint16_t* x, const RouterWs& rw, int S,
                          const float* bias, int T, int H, int E, int k, float cH, int ntok, float* logits,
                          int32_t* ids, float* w, int32_t* counts, int32_t* chist) {
  auto kern = (H % 256 == 0) ? router_select_kernel<NK, false> : router_select_kernel<NK, true>;
  return launch_pdl(kern, grid, dim3(SEL_WARPS * 32), 0, st, x, rw.WrT, rw.part, S, rw.nw, bias,
                    T, H, E, k, cH, ntok, logits, ids, w, counts, chist);
}

}  // namespace

cudaError_t router_tc_prepare() {
  return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RTC_SMEM);
}

RouterSplit router_split(int T, int H, int E, int num_sms) {
  RouterSplit r;
  const int m_tiles = (T + RTC_BM - 1) / RTC_BM;
  const int kb_total = H / RTC_BK;
  int s = (num_sms < 256 ? num_sms : 256) / (m_tiles > 0 ? m_tiles : 1);
  const int s_max = kb_total / 2 > 0 ? kb_total / 2 : 1;
  s = s < 1 ? 1 : (s > ROUTER_MAX_SPLITS ? ROUTER_MAX_SPLITS : s);
  s = s > s_max ? s_max : s;
  r.kb_total = kb_total;
  r.kb_per = (kb_total + s - 1) / s;
  r.splits = (kb_total + r.kb_per - 1) / r.kb_per;   // no empty split
  r.m_tiles = m_tiles;
  const int n_pad = ((E + 15) / 16) * 16;
  r.n_chain = n_pad <= 128 ? 4 : 2;                  // chains x (128 | 256) columns = all of TMEM
  r.chain_steps = ((r.kb_per + r.n_chain - 1) / r.n_chain) * (RTC_BK / 16);
  return r;
}

float router_bound_coef(int H, const RouterSplit& r) {
  return (float)(r.chain_steps + 1) * 0x1p-17f + (float)(r.n_chain * r.splits + H / 32 + 8) * 0x1p-22f;
}

cudaError_t launch_router_prep(const uint16_t* Wr, int H, int E, const RouterWs& rw, cudaStream_t st) {
  return launch_pdl(router_prep_kernel, dim3((E + 31) / 32, H / RP_H), dim3(256), 0, st, Wr, H, E, rw.WrT);
}

cudaError_t launch_router_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, const uint16_t* x, const float* bias,
                             const RouterWs& rw, const RouterSplit& sp, int T, int H, int E, int k, int num_sms,
                             float* logits, int32_t* ids, float* w, int32_t* counts, int32_t* chist,
                             uint32_t* err, int64_t timeout_ns, cudaStream_t st) {
  const int n_pad = ((E + 15) / 16) * 16;
  const int m_tiles = (T + RTC_BM - 1) / RTC_BM;
  cudaError_t e = launch_pdl(router_tc_kernel, dim3(m_tiles, sp.splits), dim3(RTC_THREADS), RTC_SMEM, st, tmX, tmW,
                             rw.WrT, T, H, E, n_pad, sp.kb_total, sp.kb_per, sp.n_chain, rw.part, rw.nw, err,
                             timeout_ns);
  if (e != cudaSuccess) return e;
  // tokens per block: chosen so that a block's (token, candidate) pairs mostly fit one round
  // of SEL_WARPS * 8 four-lane groups (a few more pairs would cost a whole second round).
  // Long rows mean longer accumulation chains, a larger bound coefficient and more
  // candidates per token: measured best 7 tokens for H = 2048 (fine, skewed workloads) and
  // 5 for H = 7168.  Fewer when T is small, so that every SM gets a block.
  const int per_block = (H >= 4096) ? 5 : 7;
  int ntok = (T + num_sms - 1) / num_sms;
  ntok = ntok < 1 ? 1 : (ntok > per_block ? per_block : ntok);
  const dim3 grid((T + ntok - 1) / ntok);
  const float cH = router_bound_coef(H, sp);
  if (E <= 32) return launch_select<1>(grid, st, x, rw, sp.splits, bias, T, H, E, k, cH, ntok, logits, ids, w, counts, chist);
  if (E <= 64) return launch_select<2>(grid, st, x, rw, sp.splits, bias, T, H, E, k, cH, ntok, logits, ids, w, counts, chist);
  if (E <= 128) return launch_select<4>(grid, st, x, rw, sp.splits, bias, T, H, E, k, cH, ntok, logits, ids, w, counts, chist);
  return launch_select<8>(grid, st, x, rw, sp.splits, bias, T, H, E, k, cH, ntok, logits, ids, w, counts, chist);
}

}  // namespace moe
