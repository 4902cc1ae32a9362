// Shared definitions of the MoE layer kernels: tile shapes, workspace view,
// and the expert-wave tile scheduler (host + device, so tests can evaluate the
// exact order the GPU uses without a GPU).
#pragma once
#include <cstdint>

#include "../../include/moe_gb300.h"

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

// ------------------------------------------------------------------ tile shapes
constexpr int BM = 128;          // rows of a tile (dispatch rows of one expert)
constexpr int BK = 64;           // K per pipeline stage: 64 bf16 = one 128-byte swizzle row
constexpr int MMA_N = 256;       // tcgen05 N of both GEMMs
constexpr int L1_COLS = 128;     // intermediate columns per Linear-1 tile (gate 128 | up 128)
constexpr int L2_COLS = 256;     // output columns per Linear-2 tile
constexpr int P_SCALE_COLS = 128;  // columns of P sharing one power-of-two scale
constexpr int STAGES = 4;        // smem ring depth
constexpr int PAIR = 2;          // m-tiles per cluster tile: a 2-CTA cluster shares each B tile
constexpr int UNIT_ROWS = BM * PAIR;
constexpr int MAX_E = 256;
constexpr int MAX_K = 8;

// Shapes: H and I are multiples of 64 (one 64-column TMA box).  The last Linear-1 tile of an
// expert may hold 64 intermediate columns instead of 128, the last Linear-2 tile 64, 128 or 192
// output columns instead of 256, and the last P scale block 64 columns: the operand loads of
// the missing columns read zeros (or columns that are never stored) and their stores are skipped.
constexpr int SHAPE_ALIGN = 64;
MOE_HD int l1_blocks(int I) { return (I + L1_COLS - 1) / L1_COLS; }        // Linear-1 tiles per unit
MOE_HD int l2_blocks(int H) { return (H + L2_COLS - 1) / L2_COLS; }        // Linear-2 tiles per unit
MOE_HD int p_scale_blocks(int H) { return (H + P_SCALE_COLS - 1) / P_SCALE_COLS; }   // scales per P row

constexpr int A_STAGE_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_STAGE_BYTES = MMA_N * BK * 2;              // 32 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;                   // one 64-column box, 8 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES; // 48 KB

// device error word codes (bits)
constexpr uint32_t ERR_TIMEOUT = 1u;
constexpr uint32_t ERR_CHECK = 2u;

// ------------------------------------------------------------------ schedule
// Scheduling unit: a pair of consecutive m-tiles of one expert (UNIT_ROWS rows),
// processed by the two CTAs of a cluster (CTA rank r takes m-tile 2*unit + r).
struct SchedTables {
  int E, nL1, nL2, W, mode, lead;
  int total_mt, n1_total, total;   // total_mt: number of units
  int mt[MAX_E];           // units of expert e
  int cnt[MAX_E];          // rows of expert e
  int mtb[MAX_E + 1];      // prefix of mt
  int wave_of[MAX_E];      // wave of expert e
  int w_first_mt[MAX_E + 1];
  int seg_a[MAX_E];        // modes 0/2: first ticket of L1(w); mode 1: first ticket of pre-segment w
  int seg_b[MAX_E];        // modes 0/2: first ticket of L2(w); mode 1: first ticket of merged segment w
};

MOE_HD int sched_n_mt(const SchedTables& s, int w) { return s.w_first_mt[w + 1] - s.w_first_mt[w]; }

// Position of element i of list A (size a) when A and B (size b) are merged so
// that A[i] sits at (2i+1)/(2a) and B[j] at (2j+1)/(2b) of the segment (ties: A first).
// (Operands below 2^32 take a 32-bit division; the result is the same integer.)
MOE_HD long long div_nonneg(long long n, long long d) {
  if (n < (1ll << 32) && d < (1ll << 32)) return (long long)((unsigned)n / (unsigned)d);
  return n / d;
}
MOE_HD int merge_pos_a(int i, int a, int b) {
  if (b == 0) return i;
  long long c = div_nonneg((long long)(2 * i + 1) * b + a - 1, a);
  long long cnt = c / 2;
  return i + (int)(cnt < b ? cnt : b);
}
MOE_HD int merge_pos_b(int j, int a, int b) {
  if (a == 0) return j;
  long long f = div_nonneg((long long)(2 * j + 1) * a, b);
  long long cnt = (f + 1) / 2;
  return j + (int)(cnt < a ? cnt : a);
}

// Segment starts of the ticket list, from units and waves already in s (mt, mtb,
// wave_of, w_first_mt, W, total_mt); O(W).  Shared by the host and device builders.
MOE_HD void sched_segments(SchedTables& s, int lead) {
  const int W = s.W;
  int n1_total = 0;
  int pos = 0;
  if (s.mode == MOE_SCHED_INTERLEAVED) {
    int D = lead < 1 ? 1 : lead;
    if (D > W) D = W;
    s.lead = D;
    for (int w = 0; w < D; ++w) {
      s.seg_a[w] = pos;
      pos += sched_n_mt(s, w) * s.nL1;
    }
    for (int w = 0; w < W; ++w) {
      s.seg_b[w] = pos;
      pos += sched_n_mt(s, w) * s.nL2 + (w + D < W ? sched_n_mt(s, w + D) * s.nL1 : 0);
    }
  } else {
    s.lead = 0;
    for (int w = 0; w < W; ++w) {
      s.seg_a[w] = pos;
      pos += sched_n_mt(s, w) * s.nL1;
      s.seg_b[w] = pos;
      pos += sched_n_mt(s, w) * s.nL2;
    }
  }
  for (int w = 0; w < W; ++w) n1_total += sched_n_mt(s, w) * s.nL1;
  s.n1_total = n1_total;
  s.total = pos;
}

// Serial builder: units, waves, segment starts.  counts[E] rows per expert; workers =
// number of concurrent tile workers (2-CTA clusters); a wave is the smallest run of
// experts whose Linear-1 tiles reach it (the last expert never opens a new wave).
MOE_HD void sched_build(SchedTables& s, const int* counts, int E, int nL1, int nL2, int workers, int mode,
                        int wave_experts, int lead) {
  s.E = E;
  s.nL1 = nL1;
  s.nL2 = nL2;
  s.mode = mode;
  int tot = 0;
  for (int e = 0; e < E; ++e) {
    int m = (counts[e] + UNIT_ROWS - 1) / UNIT_ROWS;
    s.cnt[e] = counts[e];
    s.mt[e] = m;
    s.mtb[e] = tot;
    tot += m;
  }
  s.mtb[E] = tot;
  s.total_mt = tot;
  int W = 0;
  if (mode == MOE_SCHED_PHASED) {
    for (int e = 0; e < E; ++e) s.wave_of[e] = 0;
    W = 1;
  } else if (wave_experts > 0) {
    for (int e = 0; e < E; ++e) s.wave_of[e] = e / wave_experts;
    W = (E + wave_experts - 1) / wave_experts;
  } else {
    int w = 0, acc = 0;
    for (int e = 0; e < E; ++e) {
      s.wave_of[e] = w;
      acc += s.mt[e] * nL1;
      if (acc >= workers && e + 1 < E) {
        ++w;
        acc = 0;
      }
    }
    W = w + 1;
  }
  s.W = W;
  for (int e = 0; e < E; ++e)
    if (e == 0 || s.wave_of[e] != s.wave_of[e - 1]) s.w_first_mt[s.wave_of[e]] = s.mtb[e];
  s.w_first_mt[W] = tot;
  sched_segments(s, lead);
}

// Ticket of the Linear-1 tile with wave-local index j in wave w.
MOE_HD int sched_ticket_l1(const SchedTables& s, int w, int j) {
  if (s.mode != MOE_SCHED_INTERLEAVED) return s.seg_a[w] + j;
  if (w < s.lead) return s.seg_a[w] + j;
  int v = w - s.lead;
  return s.seg_b[v] + merge_pos_b(j, sched_n_mt(s, v) * s.nL2, sched_n_mt(s, w) * s.nL1);
}
// Ticket of the Linear-2 tile with wave-local index i in wave w.
MOE_HD int sched_ticket_l2(const SchedTables& s, int w, int i) {
  if (s.mode != MOE_SCHED_INTERLEAVED) return s.seg_b[w] + i;
  int b = (w + s.lead < s.W) ? sched_n_mt(s, w + s.lead) * s.nL1 : 0;
  return s.seg_b[w] + merge_pos_a(i, sched_n_mt(s, w) * s.nL2, b);
}

// Expert owning global unit g (mtb[e] <= g < mtb[e+1]).
MOE_HD int sched_expert_of(const SchedTables& s, int g) {
  int lo = 0, hi = s.E - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s.mtb[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Write tile j (0 <= j < nL1 + nL2: Linear-1 n-blocks first, then Linear-2) of global
// unit g, owned by expert e.  Tile = {phase | n << 1 | rows << 16, e, unit, g}, rows =
// the unit's valid rows (1..256).  Within a wave the tiles are ordered (expert, n-block,
// unit) with the unit fastest.
MOE_HD int min_i(int a, int b) { return a < b ? a : b; }
MOE_HD void sched_emit_tile(const SchedTables& s, int g, int e, int j, int* tiles /* 4 ints per ticket */) {
  const int m = g - s.mtb[e];
  const int w = s.wave_of[e];
  const int base = s.mtb[e] - s.w_first_mt[w];
  const int rows = min_i(UNIT_ROWS, s.cnt[e] - m * UNIT_ROWS);
  int t, x;
  if (j < s.nL1) {
    t = sched_ticket_l1(s, w, base * s.nL1 + j * s.mt[e] + m);
    x = (j << 1) | 0;
  } else {
    const int nb = j - s.nL1;
    t = sched_ticket_l2(s, w, base * s.nL2 + nb * s.mt[e] + m);
    x = (nb << 1) | 1;
  }
  tiles[4 * t + 0] = x | (rows << 16);
  tiles[4 * t + 1] = e;
  tiles[4 * t + 2] = m;
  tiles[4 * t + 3] = g;
}

// Write every tile reached from global unit g.
MOE_HD void sched_emit_mtile(const SchedTables& s, int g, int* tiles /* 4 ints per ticket */) {
  const int e = sched_expert_of(s, g);
  for (int j = 0; j < s.nL1 + s.nL2; ++j) sched_emit_tile(s, g, e, j, tiles);
}

// Upper bound of units for R routed rows over E experts.
MOE_HD long long max_mtiles(long long R, int E) { return (R + UNIT_ROWS - 1) / UNIT_ROWS + E; }

}  // namespace moe
