// Device code of the persistent grouped GEMM (both expert projections of the MoE layer):
// tile shapes, the shared-memory layout and the body that one CTA of the grid runs.  The
// design is described at the top of gemm.cu; this header is included by gemm.cu (the GEMM
// launch) and by fused.cu (the single-launch layer).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm_detail {

constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int GEMM_THREADS = 64 + EPI_THREADS;
constexpr int TMEM_COLS = 512;                         // two 256-column fp32 accumulators
constexpr int MAX_NST = 6;                             // deepest per-CTA ring compiled
constexpr int BH_BYTES = 2 * B_BOX_BYTES;              // this CTA's half of B: 16 KB
constexpr int PSTAGE_BYTES = A_STAGE_BYTES + BH_BYTES; // 32 KB
constexpr int STG_BOX_BYTES = BM * 128;                // 128 staged rows x 128 bytes (one column half): 16 KB
constexpr int ST_ROWS = 32;                            // rows per output store box (one TMEM quadrant)
constexpr int ST_BOX_BYTES = ST_ROWS * 128;            // 4 KB
constexpr int STG_BYTES = 2 * STG_BOX_BYTES;           // one staging buffer: two boxes (the two column halves)
// mbarriers and flags (SmemCtl, 152 bytes), with room to spare: with the 1 KB the GPU reserves
// per block, a small block without shared memory still fits beside a CTA of this kernel
constexpr int CTL_BYTES = 512;
// Shared-memory layout of a <NST stages, NBUF staging buffers> instance.
template <int NST, int NBUF>
struct Layout {
  static constexpr int STG_OFF = NST * PSTAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + NBUF * STG_BYTES;
  static constexpr int SMEM = BAR_OFF + CTL_BYTES + 1024;   // + slack to align the base to 1024 B
  static_assert(NST <= MAX_NST && NBUF >= 1 && NBUF <= 2, "unsupported ring split");
  static_assert(SMEM <= 232448, "shared memory per CTA exceeded");
};
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(PAIR * BM, MMA_N, true);

struct SmemCtl {
  uint64_t full[MAX_NST];   // even CTA: both CTAs' loads of the stage landed
  uint64_t empty[MAX_NST];  // both CTAs: the pair MMAs of the stage completed
  uint64_t tfull[2];        // both CTAs: accumulator ready
  uint64_t tempty[2];       // even CTA: both CTAs' epilogues drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ep_ok[2];             // epilogue go/stop decision of the waiting thread, by tile parity
};
static_assert(sizeof(SmemCtl) <= CTL_BYTES, "control block exceeds its shared-memory reservation");

__device__ __forceinline__ void set_abort(SmemCtl* ctl, uint32_t* err, uint32_t code) {
  atomicOr(err, code);
  *(volatile int*)&ctl->abort_flag = 1;
}

// Tickets of this launch: range_sel 0 the Linear-1 tiles, 1 the Linear-2 tiles, 2 all, 3 none.
__device__ __forceinline__ void tile_range(const GemmArgs& a, int& begin, int& end) {
  if (a.range_sel == 3) {
    begin = end = 0;
    return;
  }
  const int n1 = a.sched[0], tot = a.sched[1];
  begin = (a.range_sel == 1) ? n1 : 0;
  end = (a.range_sel == 0) ? n1 : tot;
}

// SwiGLU element silu(g) * u = g / (1 + exp(-g)) * u (fast exp and divide: the
// tensor-core accumulation of g and u, not these last-place errors, decides
// how often the bf16 rounding of the result differs from a host evaluation).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The whole persistent GEMM for one CTA of the grid: set-up (barriers, TMEM), the role loops
// over this cluster's tickets, tear-down.  Called by grouped_gemm_kernel and by the single-launch
// layer kernel (same grid shape: 2-CTA clusters, GEMM_THREADS threads, every cluster resident).
template <int NST, int NBUF>
__device__ __forceinline__ void grouped_gemm_body(const CUtensorMap* tmA1, const CUtensorMap* tmB1,
                                                  const CUtensorMap* tmA2, const CUtensorMap* tmB2,
                                                  const CUtensorMap* tmH, const CUtensorMap* tmP, const GemmArgs& args,
                                                  uint8_t* smem_raw) {
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  using L = Layout<NST, NBUF>;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + L::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)ptx::cluster_ctarank();
  const bool leader = rank == 0;
  constexpr uint16_t CTA_MASK = (1u << PAIR) - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);        // even CTA's producer (expect_tx for both CTAs' bytes)
      ptx::mbar_init(&ctl->empty[s], 1);       // the pair MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->tfull[b], 1);       // the pair MMA commit
      ptx::mbar_init(&ctl->tempty[b], PAIR);   // one arrival per CTA's epilogue
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(tmA1);
    ptx::tma_prefetch_desc(tmB1);
    ptx::tma_prefetch_desc(tmA2);
    ptx::tma_prefetch_desc(tmB2);
    ptx::tma_prefetch_desc(tmH);
    ptx::tma_prefetch_desc(tmP);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair<TMEM_COLS>(&ctl->tmem_base);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();     // both CTAs' barriers exist before any load or arrival crosses
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;
  const bool tracing = (args.flags & MOE_FLAG_TRACE) != 0;
  const bool tile_tracing = tracing && args.tile_trace != nullptr;
  const uint64_t t_start = ptx::globaltimer();
  uint64_t tr_a = 0, tr_b = 0;     // this thread's two wait-time counters (role specific)
  uint64_t* trp_a = tracing ? &tr_a : nullptr;
  uint64_t* trp_b = tracing ? &tr_b : nullptr;
  const int cluster = blockIdx.x / PAIR, nclusters = gridDim.x / PAIR;

  ptx::grid_dep_wait();   // Dispatch's tile list and the gathered rows are visible from here on
  int t_begin, t_end;
  tile_range(args, t_begin, t_end);
  const int64_t tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_normal();
      const uint64_t pol_a = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled_mask = 0, last_par = 0;   // per stage: filled at least once / parity of last fill
      for (int i = t_begin + cluster; i < t_end && !*abort_flag; i += nclusters) {
        const int4 tl = args.tiles[i];
        const int ph = tl.x & 1, nb = (tl.x >> 1) & 0x7FFF, e = tl.y, g = tl.w;
        const int row0 = g * UNIT_ROWS + rank * BM;     // this CTA's 128 padded rows of the unit
        if (tile_tracing) args.tile_trace[((size_t)i * PAIR + rank) * TILE_TRACE_SLOTS + TT_START] = ptx::globaltimer();
        const int nk = (ph == 0 ? args.H : args.I) / BK;
        // a unit whose valid rows all lie in the even CTA's half: the odd CTA's A rows are
        // padding, whose accumulator rows are never stored, so they are not loaded at all
        const bool a_odd_empty = (tl.x >> 16) <= BM;
        const bool load_a = !(rank == 1 && a_odd_empty);
        const uint32_t stage_tx = PAIR * PSTAGE_BYTES - (a_odd_empty ? A_STAGE_BYTES : 0);
        const CUtensorMap* tA = ph == 0 ? tmA1 : tmA2;
        const CUtensorMap* tB = ph == 0 ? tmB1 : tmB2;
        const int brow0 = e * (ph == 0 ? args.H : args.I);
        // this CTA's half of B: Linear-1 rank 0 gate / rank 1 up columns of the n-block,
        // Linear-2 columns [128 r, 128 r + 128) of the 256-column block
        const int c0 = (ph == 0) ? (rank == 0 ? nb * L1_COLS : args.I + nb * L1_COLS) : nb * L2_COLS + rank * 128;
        bool ok = true;
        // claim the next stage (bounded wait until the pair MMA released it) and set its
        // transaction count; returns the stage's operand buffers
        auto claim = [&](uint8_t*& sA, uint8_t*& sB, uint32_t& full_pair) {
          if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, tmo, abort_flag, trp_a)) return false;
          sA = smem + stage * PSTAGE_BYTES;
          sB = sA + A_STAGE_BYTES;
          full_pair = ptx::mapa_shared(&ctl->full[stage], 0);
          if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], stage_tx);
          filled_mask |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
          return true;
        };
        int kb0 = 0;   // k-blocks already claimed (B issued) before the loop below
        if (ph == 1) {
          // wait for every Linear-1 tile of this unit, from both CTAs (bounded)
          const int* rp = args.ready + g;
          const int need = PAIR * args.nL1 + ((args.flags & MOE_FLAG_TEST_STALL) ? 1 : 0);
          if (ptx::ld_acquire_gpu(rp) < need) {
            // W2 does not depend on Linear-1: the first stages' B halves are loaded while the
            // unit's Linear-1 tiles finish, their A rows (h) after the wait
            const int pre = nk < NST ? nk : NST;
            const int st0 = stage;
            for (; kb0 < pre; ++kb0) {
              uint8_t *sA, *sB;
              uint32_t full_pair;
              if (!claim(sA, sB, full_pair)) { ok = false; break; }
              ptx::tma_load_2d_pair(tB, full_pair, sB, c0, brow0 + kb0 * BK, pol_w);
              ptx::tma_load_2d_pair(tB, full_pair, sB + B_BOX_BYTES, c0 + 64, brow0 + kb0 * BK, pol_w);
            }
            if (!ok) { set_abort(ctl, args.err, ERR_TIMEOUT); break; }
            const uint64_t t0 = ptx::globaltimer();
            bool ready = false;
            while (true) {
              if (ptx::ld_acquire_gpu(rp) >= need) { ready = true; break; }
              if (*abort_flag) break;
              if ((int64_t)(ptx::globaltimer() - t0) > tmo) break;
              __nanosleep(64);
            }
            tr_b += ptx::globaltimer() - t0;
            if (!ready) { set_abort(ctl, args.err, ERR_TIMEOUT); break; }
            ptx::fence_proxy_async_global();
            if (load_a) {
              for (int q = 0; q < kb0; ++q) {
                const int sq = (st0 + q) % NST;
                uint8_t* sA = smem + sq * PSTAGE_BYTES;
                ptx::tma_load_2d_pair(tA, ptx::mapa_shared(&ctl->full[sq], 0), sA, q * BK, row0, pol_a);
              }
            }
          } else {
            ptx::fence_proxy_async_global();
          }
        }
        for (int kb = kb0; kb < nk; ++kb) {
          uint8_t *sA, *sB;
          uint32_t full_pair;
          if (!claim(sA, sB, full_pair)) { ok = false; break; }
          // the whole 128-row box even when some rows are padding: loading only the valid
          // rows' 32-row quadrants measured slower (fine workload 0.483 -> 0.512 ms), and so
          // did one 32-row box for a CTA with at most 32 valid rows (large 3.91 -> 4.03 ms)
          if (load_a) ptx::tma_load_2d_pair(tA, full_pair, sA, kb * BK, row0, pol_a);
          ptx::tma_load_2d_pair(tB, full_pair, sB, c0, brow0 + kb * BK, pol_w);
          ptx::tma_load_2d_pair(tB, full_pair, sB + B_BOX_BYTES, c0 + 64, brow0 + kb * BK, pol_w);
        }
        if (!ok) { set_abort(ctl, args.err, ERR_TIMEOUT); break; }
      }
      // Before the CTA may exit: every fill of every stage has been released by the pair
      // MMA (its commit arrives here) - which also means every copy into this CTA landed.
      int dummy = 0;
      for (int s = 0; s < NST; ++s)
        if (filled_mask & (1u << s)) ptx::mbar_wait(&ctl->empty[s], (last_par >> s) & 1u, tmo, &dummy);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool issued_any = false;
      for (int i = t_begin + cluster; i < t_end && !*abort_flag; i += nclusters, ++local) {
        const int4 tl = args.tiles[i];
        const int ph = tl.x & 1;
        const int as = local & 1;
        const uint32_t aphase = (local >> 1) & 1;
        if (!ptx::mbar_wait(&ctl->tempty[as], aphase ^ 1u, tmo, abort_flag, trp_a)) {
          set_abort(ctl, args.err, ERR_TIMEOUT);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(as * MMA_N);
        const int nk = (ph == 0 ? args.H : args.I) / BK;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(&ctl->full[stage], phase, tmo, abort_flag, trp_b)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem + stage * PSTAGE_BYTES);
          const uint32_t b0 = a0 + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 2048, B_BOX_BYTES, 1024);
            ptx::mma_bf16_pair(d, ad, bd, IDESC, (kb | kk) != 0);
          }
          issued_any = true;
          ptx::mma_commit_pair_mc(&ctl->empty[stage], CTA_MASK);   // frees the stage in both CTAs
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) { set_abort(ctl, args.err, ERR_TIMEOUT); break; }
        ptx::mma_commit_pair_mc(&ctl->tfull[as], CTA_MASK);
      }
      if (*abort_flag && issued_any) {
        // make sure no MMA still reads shared memory or writes TMEM
        ptx::mma_commit_pair_mc(&ctl->drain, 1);
        int dummy = 0;
        ptx::mbar_wait(&ctl->drain, 0, tmo, &dummy);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;               // TMEM lane quadrant
    const int r = q * 32 + lane;          // tile row
    const int ep_tid = threadIdx.x - 64;  // 0..255
    const int ch = (warp - 2) >> 2;       // column half of this warp
    const uint32_t tempty_pair0 = ptx::mapa_shared(&ctl->tempty[0], 0);
    const uint32_t tempty_pair1 = ptx::mapa_shared(&ctl->tempty[1], 0);
    uint8_t* const stg = smem + L::STG_OFF;
    uint32_t sb = 0;                      // staging buffers used so far (all epilogue threads agree)
    int local = 0;
    const bool bilinear = (args.flags & MOE_FLAG_ACT_BILINEAR) != 0;
    // byte offset of 16-byte chunk cc of this thread's row inside a staged box (128-byte swizzle)
    auto chunk_off = [&](int cc) { return r * 128 + ((cc ^ (r & 7)) << 4); };
    // make the next staging buffer writable: its previous store has finished reading it
    auto acquire_stage = [&]() {
      if (ep_tid == 0) ptx::bulk_wait_read<NBUF - 1>();
      ptx::named_bar_sync(1, EPI_THREADS);
    };
    for (int i = t_begin + cluster; i < t_end; i += nclusters, ++local) {
      const int4 tl = args.tiles[i];
      const int ph = tl.x & 1, nb = (tl.x >> 1) & 0x7FFF, g = tl.w;
      const int as = local & 1;
      const uint32_t aphase = (local >> 1) & 1;
      // one thread waits, the named barrier broadcasts its decision to all epilogue threads
      unsigned long long* const ttr =
          tile_tracing ? args.tile_trace + ((size_t)i * PAIR + rank) * TILE_TRACE_SLOTS : nullptr;
      if (ep_tid == 0) {
        const bool okw = ptx::mbar_wait(&ctl->tfull[as], aphase, tmo, abort_flag, trp_a);
        if (!okw) set_abort(ctl, args.err, ERR_TIMEOUT);
        *(volatile int*)&ctl->ep_ok[local & 1] = okw ? 1 : 0;
        if (ttr && okw) {
          ttr[TT_SMID] = ptx::smid();
          ttr[TT_ACC] = ptx::globaltimer();
        }
      }
      ptx::named_bar_sync(1, EPI_THREADS);
      if (!*(volatile int*)&ctl->ep_ok[local & 1]) break;
      ptx::tc_fence_after();
      const int prow0 = g * UNIT_ROWS + rank * BM;   // the CTA's 128 padded rows
      const int rows_v = max(0, min(BM, (tl.x >> 16) - rank * BM));
      const int nfull = rows_v / ST_ROWS;             // quadrants whose rows are all valid
      const bool staged = q < nfull;                  // this warp pair's rows go through TMA stores
      const bool direct = !staged && r < rows_v;      // a valid row of the partial quadrant
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(as * MMA_N);
      const uint32_t tempty_addr = as ? tempty_pair1 : tempty_pair0;
      if (ph == 0) {
        // h = silu(gate) * up for columns [64 ch, 64 ch + 64) of the tile; the last tile of an
        // expert with I = 64 (mod 128) has no second half (its values are computed, not stored)
        const bool col_ok = nb * L1_COLS + ch * 64 < args.I;
        acquire_stage();
        uint8_t* box = stg + (sb % NBUF) * STG_BYTES + ch * STG_BOX_BYTES;
        uint16_t* hrow = args.h_pad + (size_t)(prow0 + r) * args.I + nb * L1_COLS + ch * 64;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld32(taddr + ch * 64 + c * 32, gv);
          ptx::tmem_ld32(taddr + L1_COLS + ch * 64 + c * 32, uv);
          ptx::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(gv[2 * j]), g1 = __uint_as_float(gv[2 * j + 1]);
            const float u0 = __uint_as_float(uv[2 * j]), u1 = __uint_as_float(uv[2 * j + 1]);
            const float v0 = bilinear ? g0 * u0 : silu_mul(g0, u0);
            const float v1 = bilinear ? g1 * u1 : silu_mul(g1, u1);
            pk[j] = pack_bf16x2(v0, v1);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 v4 = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            if (staged) *reinterpret_cast<uint4*>(box + chunk_off(4 * c + j)) = v4;
            else if (direct && col_ok) reinterpret_cast<uint4*>(hrow)[4 * c + j] = v4;
          }
        }
        ptx::tc_fence_before();
        ptx::fence_proxy_async_smem();
        if (direct) ptx::fence_proxy_async_global();   // h rows will be read by TMA (async proxy)
        ptx::named_bar_sync(1, EPI_THREADS);
        if (ep_tid == 0) {
          ptx::mbar_arrive_cluster(tempty_addr);     // accumulator free for the next tile
          uint8_t* buf = stg + (sb % NBUF) * STG_BYTES;
          const bool half2 = nb * L1_COLS + 64 < args.I;
          for (int gq = 0; gq < nfull; ++gq) {
            ptx::tma_store_2d(tmH, buf + gq * ST_BOX_BYTES, nb * L1_COLS, prow0 + gq * ST_ROWS);
            if (half2)
              ptx::tma_store_2d(tmH, buf + STG_BOX_BYTES + gq * ST_BOX_BYTES, nb * L1_COLS + 64,
                                prow0 + gq * ST_ROWS);
          }
          ptx::bulk_commit();
          ptx::bulk_wait<0>();                       // h rows written: publish them to Linear-2
          ptx::fence_proxy_async_global();
          if (ttr) ttr[TT_END] = ptx::globaltimer();
          __threadfence();
          ptx::red_release_add_gpu(args.ready + g, 1);
        }
        ++sb;
      } else {
        // P = w * acc; warp half ch owns columns [128 ch, 128 ch + 128) of the tile, one
        // scale block.  Sweep 1: the block's largest finite |acc| of this row sets its
        // scale 2^se; sweep 2: two passes of 64 columns, each value fp16(fl(w * acc) * 2^-se).
        const float wgt = (staged || direct) ? args.prow_w[prow0 + r] : 0.0f;
        float amax = 0.0f;
#pragma unroll 1
        for (int c4 = 0; c4 < P_SCALE_COLS / 32; ++c4) {
          uint32_t v[32];
          ptx::tmem_ld32(taddr + ch * P_SCALE_COLS + c4 * 32, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float a = fabsf(__uint_as_float(v[j]));
            amax = (a < INFINITY) ? fmaxf(amax, a) : amax;   // finite values only (NaN compares false)
          }
        }
        // M >= every finite |fl(w * acc)| of the block; se = ceil(log2 M) - 15
        const float M = amax * fabsf(wgt) * (1.0f + 0x1p-20f);
        int se = 0;
        if (M > 0.0f) {
          int cl2 = 128;                              // M rounded up past the largest float
          if (M < INFINITY) {
            const uint32_t mb = __float_as_uint(M);
            const int ex = (int)((mb >> 23) & 0xFFu);
            cl2 = (ex == 0) ? -126 : ex - 127 + ((mb & 0x7FFFFFu) ? 1 : 0);
          }
          se = max(-126, min(127, cl2 - 15));
        }
        const float inv = __uint_as_float((uint32_t)(127 - se) << 23);   // 2^-se, exact
        const int nS = p_scale_blocks(args.H);
        // columns of this warp's block that exist: 128, or 64 for the last block of an H that is
        // 64 (mod 128), or none past H (the tile's B columns there were read as zeros)
        const int col0 = nb * L2_COLS + ch * P_SCALE_COLS;
        const int ncols = max(0, min(P_SCALE_COLS, args.H - col0));
        if ((staged || direct) && ncols > 0)
          args.S_pad[(size_t)(prow0 + r) * nS + nb * (L2_COLS / P_SCALE_COLS) + ch] =
              __uint_as_float((uint32_t)(127 + se) << 23);
        uint16_t* prow = args.P_pad + (size_t)(prow0 + r) * args.H + nb * L2_COLS + ch * P_SCALE_COLS;
#pragma unroll 1
        for (int pass = 0; pass < MMA_N / 128; ++pass) {
          acquire_stage();
          uint8_t* box = stg + (sb % NBUF) * STG_BYTES + ch * STG_BOX_BYTES;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            ptx::tmem_ld32(taddr + ch * P_SCALE_COLS + pass * 64 + c * 32, v);
            ptx::tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float p0 = (wgt * __uint_as_float(v[2 * j])) * inv;
              const float p1 = (wgt * __uint_as_float(v[2 * j + 1])) * inv;
              __half2 hv = __floats2half2_rn(p0, p1);
              pk[j] = *reinterpret_cast<uint32_t*>(&hv);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 v4 = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              if (staged) *reinterpret_cast<uint4*>(box + chunk_off(4 * c + j)) = v4;
              else if (direct && pass * 64 < ncols) reinterpret_cast<uint4*>(prow + pass * 64)[4 * c + j] = v4;
            }
          }
          if (pass == MMA_N / 128 - 1) ptx::tc_fence_before();
          ptx::fence_proxy_async_smem();
          ptx::named_bar_sync(1, EPI_THREADS);
          if (ep_tid == 0) {
            if (pass == MMA_N / 128 - 1) ptx::mbar_arrive_cluster(tempty_addr);
            uint8_t* buf = stg + (sb % NBUF) * STG_BYTES;
            const bool box0 = nb * L2_COLS + pass * 64 < args.H;
            const bool box1 = nb * L2_COLS + P_SCALE_COLS + pass * 64 < args.H;
            for (int gq = 0; gq < nfull; ++gq) {
              if (box0)
                ptx::tma_store_2d(tmP, buf + gq * ST_BOX_BYTES, nb * L2_COLS + pass * 64, prow0 + gq * ST_ROWS);
              if (box1)
                ptx::tma_store_2d(tmP, buf + STG_BOX_BYTES + gq * ST_BOX_BYTES,
                                  nb * L2_COLS + P_SCALE_COLS + pass * 64, prow0 + gq * ST_ROWS);
            }
            ptx::bulk_commit();                      // one group per pass, possibly empty
            if (ttr && pass == MMA_N / 128 - 1) ttr[TT_END] = ptx::globaltimer();
          }
          ++sb;
        }
      }
    }
    if (ep_tid == 0) ptx::bulk_wait<0>();   // every store of this CTA performed before it exits
  }

  if (tracing) {
    unsigned long long* tr = args.trace + (size_t)blockIdx.x * TRACE_SLOTS;
    if (threadIdx.x == 0) {
      atomicAdd(tr + TR_PROD_WAIT_EMPTY, (unsigned long long)tr_a);
      atomicAdd(tr + TR_PROD_WAIT_READY, (unsigned long long)tr_b);
    } else if (threadIdx.x == 32) {
      atomicAdd(tr + TR_MMA_WAIT_TEMPTY, (unsigned long long)tr_a);
      atomicAdd(tr + TR_MMA_WAIT_FULL, (unsigned long long)tr_b);
    } else if (threadIdx.x == 64) {
      atomicAdd(tr + TR_EPI_WAIT_TFULL, (unsigned long long)tr_a);
      int n1 = 0, n2 = 0;
      for (int i = t_begin + cluster; i < t_end; i += nclusters) (args.tiles[i].x & 1) ? ++n2 : ++n1;
      atomicAdd(tr + TR_TILES_L1, (unsigned long long)n1);
      atomicAdd(tr + TR_TILES_L2, (unsigned long long)n2);
      atomicAdd(tr + TR_KERNEL_NS, (unsigned long long)(ptx::globaltimer() - t_start));
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();     // both CTAs finished every role: no arrival or load crosses any more
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair<TMEM_COLS>(tmem_base);
  }
}

}  // namespace gemm_detail
}  // namespace moe
