// Device pieces of the layer's data-movement steps, shared by their own launches
// (dispatch.cu, combine.cu) and the single-launch layer (fused.cu): the Dispatch sort and
// tile schedule as one "virtual block" of threads, a gather task, and a Combine item.
// Their pointer parameters carry no __restrict__: in the single launch they read data that
// earlier phases of the same kernel wrote, which the read-only (non-coherent) load path
// must not serve.  The standalone kernels keep __restrict__ on their own parameters.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int DS_SCHED_CTAS = 8;   // virtual blocks that build the schedule tables and share out the tile list
constexpr int DS_MAX_WARPS = 16;   // warps of the largest Dispatch block

// Shared memory of one Dispatch block (static in dispatch_kernel, carved from the dynamic
// shared memory of the single-launch layer).
struct DispatchSmem {
  int crow[MAX_E + 1];   // first compact row of each expert
  int units[MAX_E + 1];  // first unit of each expert
  int cnt[MAX_E];
  SchedTables s;
  int cum[MAX_E];        // Linear-1 tiles of experts 0..e (inclusive)
  int wstart[MAX_E + 1]; // first expert of each wave
  int W;
  int nxt[MAX_E];
  int pdelta[MAX_E];     // padded row - compact row of each expert
  int part[DS_MAX_WARPS * MAX_E];
};

// One virtual block vb of Dispatch (NT threads); the blocks are vb = 0 .. DS_SCHED_CTAS + C - 1,
// C = ceil(T / DS_CHUNK_TOK), run by dispatch_kernel (one CTA each) or the single-launch layer.
//
// Blocks 0 .. DS_SCHED_CTAS-1 build the schedule tables of sched_build in their shared
// memory (identical values) and each writes its slice of the tile list and of the
// readiness counters; block 0 also writes offsets[] and sched[].
//
// Block DS_SCHED_CTAS + c sorts the pairs f = t*k + j of tokens c*DS_CHUNK_TOK ..
// +DS_CHUNK_TOK-1 (a counting sort, stable: expert e's rows hold its pairs in ascending
// f).  The first row of e in this chunk is e's first compact row plus e's pairs in
// the chunks before, read from the router's chunk histograms chist[c][e].  Within the
// chunk, pairs go in rounds of NT consecutive pairs, one per thread: a pair's
// row is (e's running row) + (e's pairs in the earlier warps of the round) + (e's
// pairs in the earlier lanes of its warp, from __match_any_sync).
template <int NT>
__device__ __forceinline__ void dispatch_body(int vb, DispatchSmem& sm, const int32_t* ids, const float* w, const int32_t* counts,
                const int32_t* chist, int T, int E, int k, int nL1, int nL2, int workers, int mode,
                int wave_experts, int lead, int32_t* offsets, int32_t* row_pair,
                int32_t* row_of, int32_t* prow_of, float* prow_w,
                int32_t* tiles, int32_t* sched, int32_t* ready,
                uint32_t* err, int dead_row, int test_bad_id) {
  constexpr int NW = NT / 32;
  static_assert(NT % 32 == 0 && NT >= MAX_E && NW <= DS_MAX_WARPS, "thread count of the Dispatch body");
  const int R = T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // compact and padded first rows of every expert: warp 0, lane l owning experts 8l .. 8l+7
  int* s_crow = sm.crow;     // first compact row
  int* s_units = sm.units;   // first unit (padded row / UNIT_ROWS)
  int* s_cnt = sm.cnt;
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

  if (vb < DS_SCHED_CTAS) {
    // ---------------------------------------------------------------- schedule tables
    SchedTables& s = sm.s;
    int* s_cum = sm.cum;         // Linear-1 tiles of experts 0..e (inclusive)
    int* s_wstart = sm.wstart;   // first expert of each wave
    int& s_W = sm.W;
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
    int* s_nxt = sm.nxt;
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
    const int b = vb;
    for (int q = b * NT + tid; q < n_pairs; q += DS_SCHED_CTAS * NT) {
      const int g = q / per_unit, j = q - g * per_unit;
      sched_emit_tile(s, g, sched_expert_of(s, g), j, tiles);
    }
    for (int g = b * NT + tid; g < s.total_mt; g += DS_SCHED_CTAS * NT) ready[g] = 0;
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
  const int c = vb - DS_SCHED_CTAS;
  const int f_lo = c * DS_CHUNK_TOK * k, f_hi = min(R, f_lo + DS_CHUNK_TOK * k);
  int* s_part = sm.part;   // [G][E] chunk-prefix partial sums, then [NW][E] per-warp counts
  // e's pairs in chunks 0 .. c-1: thread (g, e) sums chunks g, g + G, ... (G groups of E threads)
  const int G = NT / E;
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
  int* s_pdelta = sm.pdelta;   // padded row - compact row of e
  if (tid < E) s_pdelta[tid] = pdelta_own;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = f_lo; r0 < f_hi; r0 += NT) {
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
    for (int i = tid; i < NW * E; i += NT) s_part[i] = 0;
    __syncthreads();
    const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(m & lt_mask);
    if (valid && rank == 0) s_part[warp * E + e] = __popc(m);
    __syncthreads();
    if (tid < E) {   // exclusive prefix over the warps, from e's running row
      int acc = run;
#pragma unroll
      for (int q = 0; q < NW; ++q) {
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
// rows are read back by the grouped GEMM long after).  Token order keeps every x row a
// single DRAM read.  Tasks are t * gather_chunks(H) + chunk.
constexpr int GA_CHUNK = 128;   // 16-byte units per warp task (2 KB)
__host__ __device__ __forceinline__ int gather_chunks(int H) { return (H / 8 + GA_CHUNK - 1) / GA_CHUNK; }

__device__ __forceinline__ void gather_task(const uint16_t* x, const int32_t* prow_of, int H,
                                            int k, uint16_t* x_pad, int task, int lane) {
  const int n = H / 8;                                  // 16-byte units per row, a multiple of 32
  const int nch = gather_chunks(H);
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

// Combine item i (one thread, 8 consecutive outputs of a token): k 16-byte loads of fp16 P
// from the slots' padded rows (found through prow_of) and their blocks' power-of-two scales,
// each widened and rescaled exactly, summed in fp32 in slot order j = 0..k-1; one 16-byte
// store.  ALL_IN_FLIGHT: the k row indices first, then all k loads at once (for small batches,
// where a resident wave of threads covers the whole output and latency decides: 128-token
// workload 12.3 -> 10.2 us); otherwise one slot after another in 32 registers, so that more
// warps stay resident (large batches are bandwidth-bound: large layer 88 vs 98 us, fine 52 vs
// 55 us with all slots in flight).  Both give the same bits.
template <bool ALL_IN_FLIGHT>
__device__ __forceinline__ void combine_item(const uint16_t* P_pad, const float* S_pad, const int32_t* prow_of, int H,
                                             int k, uint16_t* y, int64_t i) {
  const int nS = p_scale_blocks(H);
  const int64_t t = (i * 8) / H;
  const int64_t c = (i * 8) % H;
  const int32_t* pr = prow_of + t * k;
  float s[8];
  auto add = [&](int j, const uint4& v, float sc) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[q]));
      const float a = f.x * sc, b = f.y * sc;
      if (j == 0) {
        s[2 * q] = a;
        s[2 * q + 1] = b;
      } else {
        s[2 * q] = s[2 * q] + a;
        s[2 * q + 1] = s[2 * q + 1] + b;
      }
    }
  };
  if (ALL_IN_FLIGHT) {
    int64_t row[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) row[j] = (j < k) ? (int64_t)pr[j] : 0;
    uint4 v[MAX_K];
    float sc[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
      if (j < k) {
        v[j] = __ldcs(reinterpret_cast<const uint4*>(P_pad + row[j] * H + c));
        sc[j] = S_pad[row[j] * nS + c / P_SCALE_COLS];
      }
    }
#pragma unroll
    for (int j = 0; j < MAX_K; ++j)
      if (j < k) add(j, v[j], sc[j]);
  } else {
    for (int j = 0; j < k; ++j) {
      const int64_t row = pr[j];
      add(j, __ldcs(reinterpret_cast<const uint4*>(P_pad + row * H + c)), S_pad[row * nS + c / P_SCALE_COLS]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(s[2 * q], s[2 * q + 1]);
    o[q] = *reinterpret_cast<uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(y + t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moe
