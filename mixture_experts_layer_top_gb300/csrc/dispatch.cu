// Dispatch on one GPU: a stable counting sort of the (token, slot) pairs into
// expert-contiguous rows, the tile schedule of the grouped GEMMs, and the row
// gather x_pad[padded row of (t, j)] = x[t].
//
// In the X-Stage paper's MegaMoE paragraph (introduction), Dispatch moves every
// token to the rank that holds each of its experts; with every expert on this
// GPU that becomes a permutation: rows of expert e occupy offsets[e] .. offsets[e+1]-1, in
// ascending token order (each token routes to an expert at most once).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int DS_THREADS = 512;
constexpr int DS_PER_THREAD = 16;
constexpr int DS_SPLIT = 8;              // at most this many CTAs share one expert's compaction
constexpr int DS_ROWS_PER_PART = 256;    // an expert gets one CTA per this many of its rows

// Block-wide exclusive scan of one int per thread (DS_THREADS threads); returns the
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
    int s = (lane < DS_THREADS / 32) ? sh_warp[lane] : 0;
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

// Grid E * DS_SPLIT: CTA b works for expert e = b % E, part p = b / E.  The CTAs of
// part 0 build the schedule tables of sched_build in their shared memory (in
// parallel; identical values) and each writes its slice of the tile list.  Expert
// e's compaction - its pairs in ascending pair order f = t*k+j, giving compact rows,
// the padded row of each pair and the weight of that row - is split over
// P_e = ceil(count_e / DS_ROWS_PER_PART) <= DS_SPLIT parts of the pair range; part p
// first counts e's pairs before its range, so the order stays stable.
__global__ void __launch_bounds__(DS_THREADS)
dispatch_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, const int32_t* __restrict__ counts,
                int T, int E, int k, int nL1, int nL2, int workers, int mode, int wave_experts, int lead,
                int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair, int32_t* __restrict__ row_of,
                int32_t* __restrict__ prow_of, float* __restrict__ prow_w, int32_t* __restrict__ tiles,
                int32_t* __restrict__ sched, int32_t* __restrict__ ready) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int R = T * k;
  const int e = blockIdx.x % E, part = blockIdx.x / E;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cnt_e = counts[e];
  const int n_parts = min(DS_SPLIT, max(1, (cnt_e + DS_ROWS_PER_PART - 1) / DS_ROWS_PER_PART));
  if (part > 0 && part >= n_parts) return;
  __shared__ SchedTables s;
  __shared__ int s_cum[MAX_E];          // Linear-1 tiles of experts 0..e (inclusive)
  __shared__ int s_wstart[MAX_E + 1];   // first expert of each wave
  __shared__ int s_W;
  __shared__ int sh_warp[33];
  if (part == 0) {
  if (tid == 0) {
    s.E = E;
    s.nL1 = nL1;
    s.nL2 = nL2;
    s.mode = mode;
  }
  // units per expert and their exclusive prefix: warp 0, lane l owning experts 8l .. 8l+7
  if (tid < 32) {
    int m[MAX_E / 32], loc = 0;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int x = lane * (MAX_E / 32) + i;
      m[i] = (x < E) ? (counts[x] + UNIT_ROWS - 1) / UNIT_ROWS : 0;
      loc += m[i];
    }
    int inc = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
      if (lane >= off) inc += o;
    }
    int run = inc - loc;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int x = lane * (MAX_E / 32) + i;
      if (x < E) {
        s.cnt[x] = counts[x];
        s.mt[x] = m[i];
        s.mtb[x] = run;
        s_cum[x] = (run + m[i]) * nL1;
      }
      run += m[i];
    }
    if (lane == 31) {
      s.mtb[E] = inc;
      s.total_mt = inc;
    }
  }
  __syncthreads();
  // waves: the greedy rule of sched_build (a wave that starts at expert x closes at
  // the first expert y in [x, E-2] whose Linear-1 tiles since x reach `workers`, else
  // at E-1).  nxt[x] = y + 1 for every x in parallel, then one short pointer chase.
  __shared__ int s_nxt[MAX_E];
  if (mode != MOE_SCHED_PHASED && wave_experts <= 0) {
    for (int x = tid; x < E; x += blockDim.x) {
      const int base = x > 0 ? s_cum[x - 1] : 0;
      int lo = x, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_cum[mid] - base >= workers) hi = mid; else lo = mid + 1;
      }
      s_nxt[x] = lo + 1;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int W = 0;
    if (mode == MOE_SCHED_PHASED) {
      s_wstart[W++] = 0;
    } else if (wave_experts > 0) {
      for (int x = 0; x < E; x += wave_experts) s_wstart[W++] = x;
    } else {
      for (int x = 0; x < E; x = s_nxt[x]) s_wstart[W++] = x;
    }
    s_wstart[W] = E;
    s.W = W;
    s_W = W;
  }
  __syncthreads();
  const int W = s_W;
  for (int x = tid; x < E; x += blockDim.x) {
    int lo = 0, hi = W - 1;   // last wave whose first expert is <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_wstart[mid] <= x) lo = mid; else hi = mid - 1;
    }
    s.wave_of[x] = lo;
  }
  for (int v = tid; v <= W; v += blockDim.x) s.w_first_mt[v] = (v < W) ? s.mtb[s_wstart[v]] : s.mtb[E];
  __syncthreads();
  // segment starts (the values of sched_segments) by warp scans over the waves
  if (tid < 32) {
    const int D = (mode == MOE_SCHED_INTERLEAVED) ? min(max(lead, 1), W) : 0;
    auto nmt = [&](int v) { return s.w_first_mt[v + 1] - s.w_first_mt[v]; };
    // interleaved: pre-segments a[0..D-1] (Linear-1 of the first D waves), then merged
    // segments b[w] = Linear-2(w) + Linear-1(w + D); otherwise a[w] = L1(w), b[w] = a[w] + L1(w)
    int carry = 0;
    if (mode == MOE_SCHED_INTERLEAVED) {
      for (int c0 = 0; c0 < D; c0 += 32) {
        const int v = c0 + lane;
        const int len = v < D ? nmt(v) * nL1 : 0;
        int inc = len;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
          if (lane >= off) inc += o;
        }
        if (v < D) s.seg_a[v] = carry + inc - len;
        carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
      }
    }
    for (int c0 = 0; c0 < W; c0 += 32) {
      const int v = c0 + lane;
      int len = 0;
      if (v < W) {
        len = (mode == MOE_SCHED_INTERLEAVED)
                  ? nmt(v) * nL2 + (v + D < W ? nmt(v + D) * nL1 : 0)
                  : nmt(v) * (nL1 + nL2);
      }
      int inc = len;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
        if (lane >= off) inc += o;
      }
      if (v < W) {
        if (mode == MOE_SCHED_INTERLEAVED) {
          s.seg_b[v] = carry + inc - len;
        } else {
          s.seg_a[v] = carry + inc - len;
          s.seg_b[v] = carry + inc - len + nmt(v) * nL1;
        }
      }
      carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
    if (lane == 0) {
      s.lead = D;
      s.n1_total = s.total_mt * nL1;
      s.total = carry;
    }
  }
  __syncthreads();

  // ---- this CTA's slice of the tile list and readiness counters
  const int per_unit = nL1 + nL2;
  const int n_pairs = s.total_mt * per_unit;
  for (int q = e * DS_THREADS + tid; q < n_pairs; q += E * DS_THREADS) {
    const int g = q / per_unit, j = q - g * per_unit;
    sched_emit_tile(s, g, sched_expert_of(s, g), j, tiles);
  }
  for (int g = e * DS_THREADS + tid; g < s.total_mt; g += E * DS_THREADS) ready[g] = 0;
  }  // part == 0

  // ---- compaction of expert e (rows offsets[e] .. offsets[e] + counts[e] - 1), part p:
  // pairs [f_lo, f_hi) (boundaries on multiples of 16)
  const int span = ((R + n_parts - 1) / n_parts + 15) & ~15;
  const int f_lo = min(R, part * span), f_hi = min(R, f_lo + span);
  __shared__ int c_base, c_off, s_pbase;
  if (tid < 32) {
    int acc = 0, u = 0;
    for (int i = lane; i < e; i += 32) {
      const int c = counts[i];
      acc += c;
      u += (c + UNIT_ROWS - 1) / UNIT_ROWS;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      u += __shfl_xor_sync(0xFFFFFFFFu, u, off);
    }
    if (lane == 0) {
      c_base = acc;
      c_off = acc;              // first compact row of e
      s_pbase = u * UNIT_ROWS;  // first padded row of e
      if (part == 0) {
        offsets[e] = acc;
        if (e == E - 1) {
          offsets[E] = acc + cnt_e;
          sched[0] = s.n1_total;
          sched[1] = s.total;
          sched[2] = s.total_mt;
          sched[3] = acc + cnt_e;
        }
      }
    }
  }
  __syncthreads();
  if (cnt_e == 0) return;
  if (f_lo > 0) {   // e's pairs before this part's range (read and count only)
    int c = 0;
    for (int f = tid * 4; f < f_lo; f += DS_THREADS * 4) {
      if ((R % 4) == 0 && f + 4 <= f_lo) {
        const int4 q4 = *reinterpret_cast<const int4*>(ids + f);
        c += (q4.x == e) + (q4.y == e) + (q4.z == e) + (q4.w == e);
      } else {
        for (int q = f; q < min(f + 4, f_lo); ++q) c += (ids[q] == e);
      }
    }
    int total;
    block_exclusive_scan(c, sh_warp, &total);
    if (tid == 0) c_base += total;
    __syncthreads();
  }
  int running = c_base;
  const int pdelta = s_pbase - c_off;   // padded row = compact row + pdelta
  const bool vec_ok = (R % 4) == 0;
  // this thread's DS_PER_THREAD ids of the chunk starting at `base` (-1 past f_hi)
  auto load_ids = [&](int base, int (&v)[DS_PER_THREAD]) {
    const int f0 = base + tid * DS_PER_THREAD;
    if (vec_ok && f0 + DS_PER_THREAD <= f_hi) {
#pragma unroll
      for (int q = 0; q < DS_PER_THREAD / 4; ++q) {
        const int4 p = *reinterpret_cast<const int4*>(ids + f0 + 4 * q);
        v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < DS_PER_THREAD; ++q) v[q] = (f0 + q < f_hi) ? ids[f0 + q] : -1;
    }
  };
  constexpr int CHUNK = DS_THREADS * DS_PER_THREAD;
  int v[DS_PER_THREAD], vn[DS_PER_THREAD];
  load_ids(f_lo, v);
  for (int base = f_lo; base < f_hi; base += CHUNK) {
    if (base + CHUNK < f_hi) load_ids(base + CHUNK, vn);   // next chunk in flight during this one
    const int f0 = base + tid * DS_PER_THREAD;
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
#pragma unroll
    for (int q = 0; q < DS_PER_THREAD; ++q) v[q] = vn[q];
  }
}

// One warp per (token, 2 KB column chunk): x[t, chunk] is read once and written to
// the padded rows of the token's k (token, slot) pairs, x_pad[prow_of[t*k+j], :] =
// x[t, :]; four independent 16-byte loads per lane in flight, streaming stores (the
// rows are read back by the grouped GEMM long after this kernel).  Token order keeps
// every x row a single DRAM read.
constexpr int GA_CHUNK = 128;   // 16-byte units per warp task (2 KB)
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ prow_of, int T, int H, int k,
                   uint16_t* __restrict__ x_pad) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int n = H / 8;                                  // 16-byte units per row, a multiple of 32
  const int nch = (n + GA_CHUNK - 1) / GA_CHUNK;
  const int task = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (task >= T * nch) return;
  const int t = task / nch, c0 = (task - t * nch) * GA_CHUNK;
  const int c1 = min(n, c0 + GA_CHUNK);
  uint4* dst[MAX_K];
#pragma unroll
  for (int j = 0; j < MAX_K; ++j)
    dst[j] = (j < k) ? reinterpret_cast<uint4*>(x_pad + (size_t)prow_of[(size_t)t * k + j] * H) : nullptr;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  int i = c0 + lane;
  if (c1 - c0 == GA_CHUNK) {
    const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64), d = __ldg(src + i + 96);
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
      if (j < k) {
        __stcs(dst[j] + i, a);
        __stcs(dst[j] + i + 32, b);
        __stcs(dst[j] + i + 64, c);
        __stcs(dst[j] + i + 96, d);
      }
    }
  } else {
    for (; i < c1; i += 32) {
      const uint4 a = __ldg(src + i);
#pragma unroll
      for (int j = 0; j < MAX_K; ++j)
        if (j < k) __stcs(dst[j] + i, a);
    }
  }
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
      P[(size_t)f * H + c] = __half2float(__ushort_as_half(P_pad[pr * H + c])) * S_pad[pr * (H / P_SCALE_COLS) + c / P_SCALE_COLS];
}

// Token block from page-locked host memory (mapped into this device's address space)
// into the device staging buffer, pulled by the SMs with 16-byte loads: over the
// CPU-GPU link these reach a higher rate than the copy engines do for one buffer.
__global__ void __launch_bounds__(512)
stage_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  ptx::grid_dep_wait();   // the previous forward no longer reads dst from here on
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st) {
  const int64_t n = (int64_t)(bytes / 16);
  int64_t blocks = (n + 511) / 512;
  if (blocks > num_sms) blocks = num_sms;
  if (blocks < 1) blocks = 1;
  return launch_pdl(stage_copy_kernel, dim3((unsigned)blocks), dim3(512), 0, st, static_cast<const uint4*>(src),
                    static_cast<uint4*>(dst), n);
}

cudaError_t launch_dispatch(const Workspace& ws, int T, int E, int k, int H, int I, int num_sms, int mode,
                            int wave_experts, int lead, cudaStream_t st) {
  return launch_pdl(dispatch_kernel, dim3(E * DS_SPLIT), dim3(DS_THREADS), 0, st, ws.ids, ws.w, ws.counts, T, E, k, I / L1_COLS, H / L2_COLS, num_sms, mode, wave_experts, lead, ws.offsets, ws.row_pair, ws.row_of, ws.prow_of, ws.prow_w, ws.tiles, ws.sched, ws.ready);
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* prow_of, int T, int H, int k, uint16_t* x_pad,
                          cudaStream_t st) {
  const int nch = (H / 8 + GA_CHUNK - 1) / GA_CHUNK;
  return launch_pdl(gather_rows_kernel, dim3((T * nch + 7) / 8), dim3(256), 0, st, x, prow_of, T, H, k, x_pad);
}

cudaError_t launch_compact_intermediates(const int32_t* row_pair, const int32_t* prow_of, int R, int H, int I,
                                         const uint16_t* h_pad, const uint16_t* P_pad, const float* S_pad,
                                         uint16_t* h, float* P, cudaStream_t st) {
  compact_intermediates_kernel<<<(R + 7) / 8, 256, 0, st>>>(row_pair, prow_of, R, H, I, h_pad, P_pad, S_pad, h, P);
  return cudaGetLastError();
}

}  // namespace moe
