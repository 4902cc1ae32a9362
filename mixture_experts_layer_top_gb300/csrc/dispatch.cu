// Dispatch on one GPU: a stable counting sort of the (token, slot) pairs into
// expert-contiguous rows, the tile schedule of the grouped GEMMs, and the row
// gather x_pad[padded row] = x[token(row)].
//
// In the X-Stage paper's MegaMoE paragraph (introduction), Dispatch moves every
// token to the rank that holds each of its experts; with every expert on this
// GPU that becomes a permutation: rows of expert e occupy offsets[e] .. offsets[e+1]-1, in
// ascending token order (each token routes to an expert at most once).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int DS_THREADS = 1024;
constexpr int DS_PER_THREAD = 16;

// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = sh_warp[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, si, off);
      if (lane >= off) si += o;
    }
    sh_warp[lane] = si - s;   // exclusive prefix of warp totals
    if (lane == 31) sh_warp[32] = si;
  }
  __syncthreads();
  const int res = sh_warp[warp] + inc - v;
  *total = sh_warp[32];
  __syncthreads();   // sh_warp reusable afterwards
  return res;
}

// CTAs 0..E-1: compaction of expert e's pairs in ascending pair order f = t*k+j
// (compact rows, plus the padded row of each pair and the weight of that row).
// CTA E: offsets, tile schedule, zeroed readiness counters.
__global__ void __launch_bounds__(DS_THREADS)
dispatch_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, const int32_t* __restrict__ counts,
                int T, int E, int k, int nL1, int nL2, int num_sms, int mode, int wave_experts, int lead,
                int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair, int32_t* __restrict__ row_of,
                int32_t* __restrict__ prow_of, float* __restrict__ prow_w, int32_t* __restrict__ tiles,
                int32_t* __restrict__ sched, int32_t* __restrict__ ready) {
  const int R = T * k;
  if ((int)blockIdx.x < E) {
    __shared__ int sh_warp[33];
    __shared__ int s_base, s_pbase;
    const int e = blockIdx.x;
    if (threadIdx.x < 32) {
      int s = 0, u = 0;
      for (int i = threadIdx.x; i < e; i += 32) {
        const int c = counts[i];
        s += c;
        u += (c + UNIT_ROWS - 1) / UNIT_ROWS;
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, off);
      }
      if (threadIdx.x == 0) {
        s_base = s;
        s_pbase = u * UNIT_ROWS;   // padded rows of expert e start here
      }
    }
    __syncthreads();
    if (counts[e] == 0) return;
    int running = s_base;
    const int pdelta = s_pbase - s_base;   // padded row = compact row + pdelta
    const bool vec_ok = (R % 4) == 0;
    for (int base = 0; base < R; base += DS_THREADS * DS_PER_THREAD) {
      const int f0 = base + threadIdx.x * DS_PER_THREAD;
      int v[DS_PER_THREAD];
      if (vec_ok && f0 + DS_PER_THREAD <= R) {
#pragma unroll
        for (int q = 0; q < DS_PER_THREAD / 4; ++q) {
          const int4 p = *reinterpret_cast<const int4*>(ids + f0 + 4 * q);
          v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < DS_PER_THREAD; ++q) v[q] = (f0 + q < R) ? ids[f0 + q] : -1;
      }
      int c = 0;
#pragma unroll
      for (int q = 0; q < DS_PER_THREAD; ++q) c += (v[q] == e);
      int total;
      int pos = running + block_exclusive_scan(c, sh_warp, &total);
#pragma unroll
      for (int q = 0; q < DS_PER_THREAD; ++q) {
        if (v[q] == e) {
          const int f = f0 + q;
          row_pair[pos] = f;
          row_of[f] = pos;
          prow_of[f] = pos + pdelta;
          prow_w[pos + pdelta] = w[f];
          ++pos;
        }
      }
      running += total;
    }
    return;
  }

  // ---- schedule CTA
  __shared__ SchedTables s;
  __shared__ int s_counts[MAX_E];
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_counts[i] = counts[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    sched_build(s, s_counts, E, nL1, nL2, num_sms, mode, wave_experts, lead);
    int o = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = o;
      o += s_counts[e];
    }
    offsets[E] = o;
    sched[0] = s.n1_total;
    sched[1] = s.total;
    sched[2] = s.total_mt;
    sched[3] = o;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < s.total_mt; g += blockDim.x) {
    sched_emit_mtile(s, g, tiles);
    ready[g] = 0;
  }
}

// One warp per dispatch row: x_pad[padded row, :] = x[token, :] (16-byte copies).
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row_pair,
                   const int32_t* __restrict__ prow_of, int R, int H, int k, uint16_t* __restrict__ x_pad) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  const int f = row_pair[row];
  const int t = f / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(x_pad + (size_t)prow_of[f] * H);
  for (int i = lane; i < H / 8; i += 32) dst[i] = src[i];
}

// Debug copy of the intermediates into caller order: h[compact row] and P[t*k+j]
// (P as fp32: the stored fp16 value times its block's power-of-two scale, exact).
__global__ void __launch_bounds__(256)
compact_intermediates_kernel(const int32_t* __restrict__ row_pair, const int32_t* __restrict__ prow_of, int R,
                             int H, int I, const uint16_t* __restrict__ h_pad, const uint16_t* __restrict__ P_pad,
                             const float* __restrict__ S_pad, uint16_t* __restrict__ h, float* __restrict__ P) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  const int f = row_pair[row];
  const size_t pr = (size_t)prow_of[f];
  if (h)
    for (int i = lane; i < I / 8; i += 32)
      reinterpret_cast<uint4*>(h + (size_t)row * I)[i] = reinterpret_cast<const uint4*>(h_pad + pr * I)[i];
  if (P)
    for (int c = lane; c < H; c += 32)
      P[(size_t)f * H + c] = __half2float(__ushort_as_half(P_pad[pr * H + c])) * S_pad[pr * (H / L2_COLS) + c / L2_COLS];
}

}  // namespace

cudaError_t launch_dispatch(const Workspace& ws, int T, int E, int k, int H, int I, int num_sms, int mode,
                            int wave_experts, int lead, cudaStream_t st) {
  dispatch_kernel<<<E + 1, DS_THREADS, 0, st>>>(ws.ids, ws.w, ws.counts, T, E, k, I / L1_COLS, H / L2_COLS,
                                                num_sms, mode, wave_experts, lead, ws.offsets, ws.row_pair,
                                                ws.row_of, ws.prow_of, ws.prow_w, ws.tiles, ws.sched, ws.ready);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* row_pair, const int32_t* prow_of, int R, int H, int k,
                          uint16_t* x_pad, cudaStream_t st) {
  gather_rows_kernel<<<(R + 7) / 8, 256, 0, st>>>(x, row_pair, prow_of, R, H, k, x_pad);
  return cudaGetLastError();
}

cudaError_t launch_compact_intermediates(const int32_t* row_pair, const int32_t* prow_of, int R, int H, int I,
                                         const uint16_t* h_pad, const uint16_t* P_pad, const float* S_pad,
                                         uint16_t* h, float* P, cudaStream_t st) {
  compact_intermediates_kernel<<<(R + 7) / 8, 256, 0, st>>>(row_pair, prow_of, R, H, I, h_pad, P_pad, S_pad, h, P);
  return cudaGetLastError();
}

}  // namespace moe
