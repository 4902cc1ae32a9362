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
constexpr int DS_WARPS = DS_THREADS / 32;
constexpr int DS_SCHED_CTAS = 8;   // CTAs that build the schedule tables and share out the tile list

// Grid DS_SCHED_CTAS + C, C = ceil(T / DS_CHUNK_TOK).
//
// CTAs 0 .. DS_SCHED_CTAS-1 build the schedule tables of sched_build in their shared
// memory (identical values) and each writes its slice of the tile list and of the
// readiness counters; CTA 0 also writes offsets[] and sched[].
//
// CTA DS_SCHED_CTAS + c sorts the pairs f = t*k + j of tokens c*DS_CHUNK_TOK ..
// +DS_CHUNK_TOK-1 (a counting sort, stable: expert e's rows hold its pairs in ascending
// f).  The first row of e in this chunk is e's first compact row plus e's pairs in
// the chunks before, read from the router's chunk histograms chist[c][e].  Within the
// chunk, pairs go in rounds of DS_THREADS consecutive pairs, one per thread: a pair's
// row is (e's running row) + (e's pairs in the earlier warps of the round) + (e's
// pairs in the earlier lanes of its warp, from __match_any_sync).
__global__ void __launch_bounds__(DS_THREADS)
dispatch_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, const int32_t* __restrict__ counts,
                const int32_t* __restrict__ chist, int T, int E, int k, int nL1, int nL2, int workers, int mode,
                int wave_experts, int lead, int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair,
                int32_t* __restrict__ row_of, int32_t* __restrict__ prow_of, float* __restrict__ prow_w,
                int32_t* __restrict__ tiles, int32_t* __restrict__ sched, int32_t* __restrict__ ready,
                uint32_t* __restrict__ err, int dead_row, int test_bad_id) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int R = T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // compact and padded first rows of every expert: warp 0, lane l owning experts 8l .. 8l+7
  __shared__ int s_crow[MAX_E + 1];   // first compact row
  __shared__ int s_units[MAX_E + 1];  // first unit (padded row / UNIT_ROWS)
  __shared__ int s_cnt[MAX_E];
  if (tid < 32) {
    int m[MAX_E / 32], c[MAX_E / 32], loc_m = 0, loc_c = 0;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int x = lane * (MAX_E / 32) + i;
      c[i] = (x < E) ? counts[x] : 0;
      m[i] = (c[i] + UNIT_ROWS - 1) / UNIT_ROWS;
      loc_m += m[i];
      loc_c += c[i];
    }
    int inc_m = loc_m, inc_c = loc_c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int om = __shfl_up_sync(0xFFFFFFFFu, inc_m, off);
      const int oc = __shfl_up_sync(0xFFFFFFFFu, inc_c, off);
      if (lane >= off) {
        inc_m += om;
        inc_c += oc;
      }
    }
    int run_m = inc_m - loc_m, run_c = inc_c - loc_c;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int x = lane * (MAX_E / 32) + i;
      if (x < E) {
        s_cnt[x] = c[i];
        s_units[x] = run_m;
        s_crow[x] = run_c;
      }
      run_m += m[i];
      run_c += c[i];
    }
    if (lane == 31) {
      s_units[E] = inc_m;
      s_crow[E] = inc_c;
    }
  }

  if (blockIdx.x < DS_SCHED_CTAS) {
    // ---------------------------------------------------------------- schedule tables
    __shared__ SchedTables s;
    __shared__ int s_cum[MAX_E];          // Linear-1 tiles of experts 0..e (inclusive)
    __shared__ int s_wstart[MAX_E + 1];   // first expert of each wave
    __shared__ int s_W;
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {
      s.cnt[x] = s_cnt[x];
      s.mt[x] = s_units[x + 1] - s_units[x];
      s.mtb[x] = s_units[x];
      s_cum[x] = s_units[x + 1] * nL1;
    }
    if (tid == 0) {
      s.E = E;
      s.nL1 = nL1;
      s.nL2 = nL2;
      s.mode = mode;
      s.mtb[E] = s_units[E];
      s.total_mt = s_units[E];
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
    // this CTA's slice of the tile list and readiness counters
    const int per_unit = nL1 + nL2;
    const int n_pairs = s.total_mt * per_unit;
    const int b = blockIdx.x;
    for (int q = b * DS_THREADS + tid; q < n_pairs; q += DS_SCHED_CTAS * DS_THREADS) {
      const int g = q / per_unit, j = q - g * per_unit;
      sched_emit_tile(s, g, sched_expert_of(s, g), j, tiles);
    }
    for (int g = b * DS_THREADS + tid; g < s.total_mt; g += DS_SCHED_CTAS * DS_THREADS) ready[g] = 0;
    if (b == 0) {
      for (int x = tid; x <= E; x += blockDim.x) offsets[x] = s_crow[x];
      if (tid == 0) {
        sched[0] = s.n1_total;
        sched[1] = s.total;
        sched[2] = s.total_mt;
        sched[3] = s_crow[E];
      }
    }
    return;
  }

  // ------------------------------------------------------------------ chunk c of the pairs
  const int c = blockIdx.x - DS_SCHED_CTAS;
  const int f_lo = c * DS_CHUNK_TOK * k, f_hi = min(R, f_lo + DS_CHUNK_TOK * k);
  __shared__ int s_part[DS_WARPS * MAX_E];   // [G][E] chunk-prefix partial sums, then [DS_WARPS][E] per-warp counts
  // e's pairs in chunks 0 .. c-1: thread (g, e) sums chunks g, g + G, ... (G groups of E threads)
  const int G = DS_THREADS / E;
  {
    const int g = tid / E, e = tid - g * E;
    if (g < G) {
      int acc = 0;
      for (int c0 = g; c0 < c; c0 += 8 * G) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = (c0 + u * G < c) ? chist[(size_t)(c0 + u * G) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += v[u];
      }
      s_part[g * E + e] = acc;
    }
  }
  __syncthreads();
  int run = 0;   // thread e < E: compact row of e's next pair
  int pdelta_own = 0;
  if (tid < E) {
    run = s_crow[tid];
    for (int g = 0; g < G; ++g) run += s_part[g * E + tid];
    pdelta_own = s_units[tid] * UNIT_ROWS - s_crow[tid];
  }
  __shared__ int s_pdelta[MAX_E];   // padded row - compact row of e
  if (tid < E) s_pdelta[tid] = pdelta_own;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = f_lo; r0 < f_hi; r0 += DS_THREADS) {
    const int f = r0 + tid;
    int e = f < f_hi ? ids[f] : -1;
    if (test_bad_id && f == 0) e = E;         // test only: one pair's expert id out of range
    if (f < f_hi && (unsigned)e >= (unsigned)E) {
      // ids come from the router and are always in range; an inconsistent one is reported,
      // and its pair gets the dead row (zero P, no tile: Combine adds nothing for it)
      atomicOr(err, ERR_CHECK);
      prow_of[f] = dead_row;
      e = -1;
    }
    const bool valid = e >= 0;
    const float wf = valid ? w[f] : 0.0f;
    __syncthreads();   // s_part free (previous round's rows read)
    for (int i = tid; i < DS_WARPS * E; i += DS_THREADS) s_part[i] = 0;
    __syncthreads();
    const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(m & lt_mask);
    if (valid && rank == 0) s_part[warp * E + e] = __popc(m);
    __syncthreads();
    if (tid < E) {   // exclusive prefix over the warps, from e's running row
      int acc = run;
#pragma unroll
      for (int q = 0; q < DS_WARPS; ++q) {
        const int t = s_part[q * E + tid];
        s_part[q * E + tid] = acc;
        acc += t;
      }
      run = acc;
    }
    __syncthreads();
    const int pos = valid ? s_part[warp * E + e] + rank : 0;
    if (valid && pos < s_crow[e + 1]) {   // rows stay in e's range even if counts and ids disagreed
      const int prow = pos + s_pdelta[e];
      row_pair[pos] = f;
      row_of[f] = pos;
      prow_of[f] = prow;
      prow_w[prow] = wf;
    } else if (valid) {                   // more pairs of e than the router counted: reported
      atomicOr(err, ERR_CHECK);
      prow_of[f] = dead_row;
    }
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
                             int R_pad, int H, int I, const uint16_t* __restrict__ h_pad,
                             const uint16_t* __restrict__ P_pad, const float* __restrict__ S_pad,
                             uint16_t* __restrict__ h, float* __restrict__ P) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  const int f = row_pair[row];
  // after inconsistent routing (reported by Dispatch) a compact row may hold no pair: zeros
  const int32_t prr = ((unsigned)f < (unsigned)R) ? prow_of[f] : -1;
  if ((unsigned)prr >= (unsigned)R_pad) {
    if (h)
      for (int i = lane; i < I / 8; i += 32) reinterpret_cast<uint4*>(h + (size_t)row * I)[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const size_t pr = (size_t)prr;
  if (h)
    for (int i = lane; i < I / 8; i += 32)
      reinterpret_cast<uint4*>(h + (size_t)row * I)[i] = reinterpret_cast<const uint4*>(h_pad + pr * I)[i];
  if (P)
    for (int c = lane; c < H; c += 32)
      P[(size_t)f * H + c] = __half2float(__ushort_as_half(P_pad[pr * H + c])) * S_pad[pr * (H / P_SCALE_COLS) + c / P_SCALE_COLS];
}

// Token block from page-locked host memory (mapped into this device's address space)
// into the device staging buffer, pulled by the SMs with 16-byte loads, four in flight
// per thread.  The CPU-GPU link, not the SMs, is the limit: 16 blocks of 512 threads
// reach its rate (measured 203 GB/s, as for 152 blocks), which leaves the other SMs
// to the router running beside the copy.
constexpr int SC_BLOCKS = 16;
__global__ void __launch_bounds__(512)
stage_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  ptx::grid_dep_wait();   // the previous forward no longer reads dst from here on
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st) {
  const int64_t n = (int64_t)(bytes / 16);
  int64_t blocks = (n + 511) / 512;
  const int64_t cap = num_sms < SC_BLOCKS ? num_sms : SC_BLOCKS;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(stage_copy_kernel, dim3((unsigned)blocks), dim3(512), 0, st, static_cast<const uint4*>(src),
                    static_cast<uint4*>(dst), n);
}

cudaError_t launch_dispatch(const Workspace& ws, int T, int E, int k, int H, int I, int num_sms, int mode,
                            int wave_experts, int lead, int dead_row, bool test_bad_id, cudaStream_t st) {
  const int chunks = (T + DS_CHUNK_TOK - 1) / DS_CHUNK_TOK;
  return launch_pdl(dispatch_kernel, dim3(DS_SCHED_CTAS + chunks), dim3(DS_THREADS), 0, st, ws.ids, ws.w, ws.counts,
                    ws.chist, T, E, k, I / L1_COLS, H / L2_COLS, num_sms, mode, wave_experts, lead, ws.offsets,
                    ws.row_pair, ws.row_of, ws.prow_of, ws.prow_w, ws.tiles, ws.sched, ws.ready, ws.err, dead_row,
                    test_bad_id ? 1 : 0);
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* prow_of, int T, int H, int k, uint16_t* x_pad,
                          cudaStream_t st) {
  const int nch = (H / 8 + GA_CHUNK - 1) / GA_CHUNK;
  return launch_pdl(gather_rows_kernel, dim3((T * nch + 7) / 8), dim3(256), 0, st, x, prow_of, T, H, k, x_pad);
}

cudaError_t launch_compact_intermediates(const int32_t* row_pair, const int32_t* prow_of, int R, int R_pad, int H,
                                         int I, const uint16_t* h_pad, const uint16_t* P_pad, const float* S_pad,
                                         uint16_t* h, float* P, cudaStream_t st) {
  compact_intermediates_kernel<<<(R + 7) / 8, 256, 0, st>>>(row_pair, prow_of, R, R_pad, H, I, h_pad, P_pad, S_pad, h,
                                                             P);
  return cudaGetLastError();
}

}  // namespace moe
