// The whole MoE layer in one launch (MOE_FLAG_SINGLE_LAUNCH).
//
// The X-Stage paper's MegaMoE paragraph (introduction) describes the expert layer as
// one persistent, warp-specialised kernel that covers Dispatch, Linear-1, the
// activation, Linear-2 and Combine.  This kernel is that single launch for one GPU:
// it runs on the grouped GEMM's grid (2-CTA clusters, 320 threads, every cluster
// resident at once) and goes through the layer's steps as phases separated by
// grid-wide barriers:
//
//   A  router logits in the canonical fp32 order on the CUDA cores (W_router given), x and
//      W_router staged in shared memory per task of 32, 16 or 8 tokens x 8 experts
//   B  top-k, softmax weights, expert counts (one warp per token)
//   C  Dispatch: counting sort, padded rows, tile list (dispatch_body, 320-thread blocks)
//   D  gather of the x rows into the padded row space
//   E  the grouped GEMM (grouped_gemm_body: Linear-1 + SwiGLU, Linear-2 + router weight)
//   F  Combine (combine_item)
//
// Each phase is the code of the multi-launch path (shared device functions), so the
// results are bitwise those of that path with MOE_FLAG_EXACT_LOGITS.  What the single
// launch removes is the launch and drain gap between the steps, which dominates when
// the layer holds few tokens.
//
// Grid barrier: one arrival counter in the plan's workspace, zeroed with the expert
// counts before the launch; barrier n waits until n * gridDim.x arrivals.  Every CTA is
// resident (the grid is the GEMM's co-resident cluster count), so the wait ends; it is
// still bounded by timeout_ns, after which the CTA records MOE_ERR_TIMEOUT and skips the
// work of the remaining phases - but keeps arriving at every barrier and runs the GEMM
// body with an empty tile range, so no CTA waits for it unboundedly and both CTAs of
// each cluster meet at the cluster barriers.
//
// Memory ordering across phases: before arriving, each CTA synchronises its threads and
// one thread issues a gpu-scope fence; the waiter reads the counter with an acquire load.
// Data read in a later phase through the TMA unit (the gathered rows) is preceded by a
// generic-to-async proxy fence on both sides, and data the GEMM's TMA stores wrote (P)
// by one before the next barrier.
#include "gemm_body.cuh"
#include "layer_parts.cuh"
#include "routing.cuh"

namespace moe {

namespace {

using namespace gemm_detail;

struct FusedArgs {
  const uint16_t* x;
  const uint16_t* Wr;   // null: the logits are the caller's input
  const float* bias;
  float* logits;
  uint16_t* y;
  Workspace ws;
  unsigned int* gbar;
  int T, H, E, k;
  int workers, mode, wave_experts, lead, dead_row, test_bad_id;
  int64_t timeout_ns;
  int trace_ctas;   // CTAs whose counters precede the phase stamps in the trace buffer
  int rtok;         // tokens per router task: 32, 16 or 8 (router_task_tokens)
  GemmArgs ga;
};

constexpr int FZ_WARPS = GEMM_THREADS / 32;
constexpr int FZ_BAR_OFF = 128 * 1024;  // shared word of the grid barrier (beyond the router ring and DispatchSmem)
static_assert(sizeof(DispatchSmem) + 1024 <= FZ_BAR_OFF, "Dispatch shared memory overlaps the barrier word");

// Arrive at grid barrier n (1-based) and, when `wait`, wait for all CTAs (bounded).  Returns
// whether this CTA may go on with the next phase's work.
__device__ bool grid_barrier(unsigned int* ctr, unsigned int n, bool wait, int64_t tmo, uint32_t* err,
                             volatile int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    bool ok = wait;
    if (wait) {
      const unsigned int target = n * gridDim.x;
      const uint64_t t0 = ptx::globaltimer();
      while ((unsigned int)ptx::ld_acquire_gpu(reinterpret_cast<const int*>(ctr)) < target) {
        if ((int64_t)(ptx::globaltimer() - t0) > tmo) {
          atomicOr(err, ERR_TIMEOUT);
          ok = false;
          break;
        }
        __nanosleep(32);
      }
    }
    *s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Top-k of token t by one warp from its logits row l (global memory, or the CTA's shared copy):
// the selection and weights of routing.cuh, counts by atomics.
__device__ __forceinline__ void topk_token(const FusedArgs& a, int t, const float* l, int lane) {
  const int nkey = (a.E + 31) >> 5;
  uint64_t key[MAX_E / 32];
#pragma unroll
  for (int i = 0; i < MAX_E / 32; ++i) {
    const int e = lane + 32 * i;
    key[i] = (i < nkey && e < a.E) ? select_key(l[e], e) : 0ull;
  }
  const int my_e = warp_select_topk(key, a.k, lane);
  const float my_l = (lane < a.k) ? l[my_e] : 0.0f;
  const float wt = warp_softmax_weight(my_l, a.k, lane);
  if (lane < a.k) {
    a.ws.ids[(size_t)t * a.k + lane] = my_e;
    a.ws.w[(size_t)t * a.k + lane] = wt;
    atomicAdd(&a.ws.counts[my_e], 1);
    atomicAdd(&a.ws.chist[(size_t)(t / DS_CHUNK_TOK) * a.E + my_e], 1);
  }
}

// Phase B, one warp per token.
__device__ void topk_phase(const FusedArgs& a, int gw, int nw, int lane) {
  for (int t = gw; t < a.T; t += nw) topk_token(a, t, a.logits + (size_t)t * a.E, lane);
}

// Phase A: a CTA task is FR_TOK tokens x FR_EXP experts.  x and W_router stream through a
// FR_NS-stage cp.async ring in shared memory in chunks of FR_HC h; compute warp w (of 8) owns
// tokens 4w .. 4w+3 of the task and all FR_EXP experts: lane j accumulates h = j, j+32, ... in
// ascending h with one fused multiply-add each, then the xor butterfly adds the 32 partials
// pairwise (j, j+16), (j, j+8), ..., (j, j+1) - the canonical order of the library's logits.
constexpr int FR_TOK = 32, FR_EXP = 8, FR_HC = 256, FR_NS = 4;
constexpr int FR_XROW = FR_HC + 8;                   // bf16 per staged x row (conflict-free, 16-B multiple)
constexpr int FR_STAGE_X = FR_TOK * FR_XROW;         // elements
constexpr int FR_STAGE_W = FR_HC * FR_EXP;           // elements: [h][8 experts]
constexpr int FR_STAGE = FR_STAGE_X + FR_STAGE_W;
constexpr int FR_CWARPS = FR_TOK / 4;                // compute warps
static_assert(FR_NS * FR_STAGE * 2 + FR_TOK * FR_EXP * 4 + 1024 <= FZ_BAR_OFF, "router ring overlaps the barrier word");
static_assert(FR_CWARPS <= FZ_WARPS, "router tile needs more warps than the CTA has");

__device__ __forceinline__ void fr_cp16(uint16_t* dst, const uint16_t* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

// with_topk (one expert group, E <= FR_EXP): the CTA that wrote a task's logits - every expert
// of its tokens - selects those tokens' experts right away (a CTA barrier orders the writes).
// A task holds a.rtok tokens (32, 16 or 8: fewer when the batch would leave SMs without a task),
// one compute warp per 4 of them; every logit's fused multiply-adds are the same either way.
__device__ void router_phase(const FusedArgs& a, uint16_t* rs, int lane, int warp, bool with_topk) {
  float* lg = reinterpret_cast<float*>(rs + FR_NS * FR_STAGE);   // [FR_TOK][FR_EXP] logits (with_topk)
  const int rtok = a.rtok;
  const int nT = (a.T + rtok - 1) / rtok, nE = (a.E + FR_EXP - 1) / FR_EXP;
  const bool wvec = (a.E % FR_EXP) == 0;     // 16-byte rows of W_router (else element copies)
  // the last chunk of an H that is not a multiple of FR_HC holds zeros past H (a fused
  // multiply-add of 0 * 0 leaves a partial sum unchanged: the canonical value is the same)
  const int nchunk = (a.H + FR_HC - 1) / FR_HC;
  for (int task = blockIdx.x; task < nT * nE; task += gridDim.x) {
    const int t0 = (task / nE) * rtok, e0 = (task % nE) * FR_EXP;
    auto issue = [&](int c) {
      uint16_t* xs = rs + (c % FR_NS) * FR_STAGE;
      uint16_t* ws = xs + FR_STAGE_X;
      const int h0 = c * FR_HC;
      for (int q = threadIdx.x; q < rtok * (FR_HC / 8); q += GEMM_THREADS) {     // x: 16-byte pieces
        const int tok = q / (FR_HC / 8), pc = q % (FR_HC / 8);
        const bool ok = t0 + tok < a.T && h0 + pc * 8 < a.H;
        fr_cp16(xs + tok * FR_XROW + pc * 8, ok ? a.x + (size_t)(t0 + tok) * a.H + h0 + pc * 8 : a.x, ok);
      }
      for (int r = threadIdx.x; r < FR_HC; r += GEMM_THREADS) {                   // W_router rows h0 + r
        const bool h_ok = h0 + r < a.H;
        const uint16_t* src = a.Wr + (size_t)(h_ok ? h0 + r : 0) * a.E + e0;
        if (wvec) {
          fr_cp16(ws + r * FR_EXP, src, h_ok);
        } else {
#pragma unroll
          for (int b = 0; b < FR_EXP; ++b) ws[r * FR_EXP + b] = (e0 + b < a.E && h_ok) ? src[b] : (uint16_t)0;
        }
      }
    };
    float acc[4][FR_EXP];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < FR_EXP; ++b) acc[i][b] = 0.0f;
#pragma unroll
    for (int c = 0; c < FR_NS - 1; ++c) {
      if (c < nchunk) issue(c);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int c = 0; c < nchunk; ++c) {
      if (c + FR_NS - 1 < nchunk) issue(c + FR_NS - 1);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group %0;" ::"n"(FR_NS - 1) : "memory");
      __syncthreads();
      if (warp < rtok / 4) {
        const uint16_t* xs = rs + (c % FR_NS) * FR_STAGE + (warp * 4) * FR_XROW;
        const uint16_t* ws = rs + (c % FR_NS) * FR_STAGE + FR_STAGE_X;
#pragma unroll
        for (int i = 0; i < FR_HC / 32; ++i) {
          const int hr = i * 32 + lane;        // global h = c * FR_HC + 32 i + lane == lane (mod 32)
          const uint4 wv4 = *reinterpret_cast<const uint4*>(ws + hr * FR_EXP);
          const uint32_t u[4] = {wv4.x, wv4.y, wv4.z, wv4.w};
          float wv[FR_EXP];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            wv[2 * q] = __uint_as_float(u[q] << 16);
            wv[2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
          }
#pragma unroll
          for (int ti = 0; ti < 4; ++ti) {
            const float xv = __uint_as_float((uint32_t)xs[ti * FR_XROW + hr] << 16);
#pragma unroll
            for (int b = 0; b < FR_EXP; ++b) acc[ti][b] = __fmaf_rn(xv, wv[b], acc[ti][b]);
          }
        }
      }
      __syncthreads();                         // the stage is refilled next round
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (warp < rtok / 4) {
      float mine = 0.0f;
#pragma unroll
      for (int ti = 0; ti < 4; ++ti)
#pragma unroll
        for (int b = 0; b < FR_EXP; ++b) {
          float v = acc[ti][b];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
          if (lane == ti * FR_EXP + b) mine = v;
        }
      const int t = t0 + warp * 4 + lane / FR_EXP, e = e0 + lane % FR_EXP;
      const float v = a.bias ? __fadd_rn(mine, a.bias[e < a.E ? e : 0]) : mine;
      if (t < a.T && e < a.E) {
        a.logits[(size_t)t * a.E + e] = v;
        if (with_topk) lg[(t - t0) * FR_EXP + e] = v;   // the CTA's copy for the top-k below
      }
    }
    __syncthreads();                           // the ring is reused by the next task
    if (with_topk) {
      for (int tt = warp; tt < rtok && t0 + tt < a.T; tt += FZ_WARPS) topk_token(a, t0 + tt, lg + tt * FR_EXP, lane);
      __syncthreads();                         // lg is rewritten by the next task
    }
  }
}

// Phase A as a kernel of its own: the multi-launch path's canonical router for small token
// counts, where its tasks (32, 16 or 8 tokens x 8 experts, one CTA each) spread over every SM while the
// tensor-core router's selection and the 32 x 32 canonical kernel leave most SMs idle.  With
// E <= FR_EXP the CTA that wrote a task's logits also selects its tokens' experts.
constexpr int FR_SMEM = FR_NS * FR_STAGE * 2 + FR_TOK * FR_EXP * 4;

__global__ void __launch_bounds__(GEMM_THREADS)
router_tasks_kernel(const FusedArgs a) {
  extern __shared__ __align__(16) uint8_t rsm_raw[];
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  router_phase(a, reinterpret_cast<uint16_t*>(rsm_raw), threadIdx.x & 31, threadIdx.x >> 5, a.E <= FR_EXP);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
fused_layer_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmP,
                   const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * FZ_WARPS + warp, nw = gridDim.x * FZ_WARPS;
  volatile int* s_ok = reinterpret_cast<volatile int*>(smem_raw + FZ_BAR_OFF);
  unsigned int nbar = 0;
  bool ok = true;
  // MOE_FLAG_TRACE: CTA 0 stamps the start and the end of every phase (%globaltimer) in the 8
  // slots after the per-CTA counters: start, after A, B, C, D, E, F (A's slot repeats the start
  // when there is no router phase)
  unsigned long long* stamp = (a.ga.trace && blockIdx.x == 0 && threadIdx.x == 0)
                                  ? a.ga.trace + (size_t)a.trace_ctas * TRACE_SLOTS : nullptr;
  if (stamp) stamp[0] = ptx::globaltimer();
  // barrier after phase p (1 = A .. 5 = E); nbar counts the barriers actually passed
  auto barrier = [&](int p) {
    ok = grid_barrier(a.gbar, ++nbar, ok, a.timeout_ns, a.ws.err, s_ok);
    if (stamp) stamp[p] = ptx::globaltimer();
  };

  const bool ab_local = a.Wr && a.E <= FR_EXP;   // A and B in one pass, no grid barrier between
  if (a.Wr) {                                                           // A
    if (ok) router_phase(a, reinterpret_cast<uint16_t*>(smem_raw), lane, warp, ab_local);
    if (!ab_local) barrier(1);
    else if (stamp) stamp[1] = ptx::globaltimer();
  } else if (stamp) {
    stamp[1] = stamp[0];
  }
  if (ok && !ab_local) topk_phase(a, gw, nw, lane);                     // B
  barrier(2);
  if (ok) {                                                             // C
    DispatchSmem* dsm = reinterpret_cast<DispatchSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~(uintptr_t)15);
    const int nvb = DS_SCHED_CTAS + (a.T + DS_CHUNK_TOK - 1) / DS_CHUNK_TOK;
    for (int vb = blockIdx.x; vb < nvb; vb += gridDim.x) {
      dispatch_body<GEMM_THREADS>(vb, *dsm, a.ws.ids, a.ws.w, a.ws.counts, a.ws.chist, a.T, a.E, a.k, a.ga.nL1,
                                  a.ga.nL2, a.workers, a.mode, a.wave_experts, a.lead, a.ws.offsets, a.ws.row_pair,
                                  a.ws.row_of, a.ws.prow_of, a.ws.prow_w, a.ws.tiles, a.ws.sched, a.ws.ready,
                                  a.ws.err, a.dead_row, a.test_bad_id);
      __syncthreads();
    }
  }
  barrier(3);
  if (ok) {                                                             // D
    const int ntask = a.T * gather_chunks(a.H);
    for (int task = gw; task < ntask; task += nw) gather_task(a.x, a.ws.prow_of, a.H, a.k, a.ws.x_pad, task, lane);
    ptx::fence_proxy_async_global();   // the rows are read by the GEMM's TMA loads
  }
  barrier(4);
  ptx::fence_proxy_async_global();
  {                                                                     // E
    GemmArgs ga = a.ga;
    ga.range_sel = ok ? 2 : 3;
    grouped_gemm_body<6, 1>(&tmA1, &tmB1, &tmA2, &tmB2, &tmH, &tmP, ga, smem_raw);
    ptx::fence_proxy_async_global();   // P and its scales are read by Combine's loads
  }
  barrier(5);
  if (ok) {                                                             // F
    const int64_t n8 = (int64_t)a.T * a.H / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x)
      combine_item<true>(a.ws.P_pad, a.ws.S_pad, a.ws.prow_of, a.H, a.k, a.y, i);   // small batches: latency-bound
  }
  if (a.ga.trace) {   // the end of Combine: the last CTA to finish writes the stamp
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned int done = atomicAdd(a.gbar + 1, 1u);
      if (done == gridDim.x - 1) a.ga.trace[(size_t)a.trace_ctas * TRACE_SLOTS + 6] = ptx::globaltimer();
    }
  }
}

}  // namespace

cudaError_t router_tasks_prepare() {
  return cudaFuncSetAttribute(router_tasks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FR_SMEM);
}

int router_tasks(int T, int E) { return ((T + FR_TOK - 1) / FR_TOK) * ((E + FR_EXP - 1) / FR_EXP); }

// Tokens per router task: the largest of 32, 16, 8 that still gives `ctas` tasks (so that a
// small batch spreads over the grid), else 8.
int router_task_tokens(int T, int E, int ctas) {
  const int nE = (E + FR_EXP - 1) / FR_EXP;
  for (int tpt = FR_TOK; tpt > 8; tpt /= 2)
    if ((int64_t)((T + tpt - 1) / tpt) * nE >= ctas) return tpt;
  return 8;
}

cudaError_t launch_router_tasks(const uint16_t* x, const uint16_t* Wr, const float* bias, float* logits,
                                const Workspace& ws, int T, int H, int E, int k, int num_sms, bool* topk_done,
                                cudaStream_t st) {
  FusedArgs a = {};
  a.x = x;
  a.Wr = Wr;
  a.bias = bias;
  a.logits = logits;
  a.ws = ws;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  *topk_done = E <= FR_EXP;
  a.rtok = router_task_tokens(T, E, num_sms);
  const int tasks = ((T + a.rtok - 1) / a.rtok) * ((E + FR_EXP - 1) / FR_EXP);
  const int cap = 2 * num_sms;   // two resident CTAs per SM
  return launch_pdl(router_tasks_kernel, dim3((unsigned)(tasks < cap ? tasks : cap)), dim3(GEMM_THREADS),
                    (size_t)FR_SMEM, st, a);
}

cudaError_t fused_prepare(int device, int* grid) {
  using L = Layout<6, 1>;
  cudaError_t e = cudaFuncSetAttribute(fused_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(sms / PAIR * PAIR, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, fused_layer_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters > sms / PAIR) clusters = sms / PAIR;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  *grid = clusters * PAIR;
  return cudaSuccess;
}

cudaError_t launch_fused_layer(const CUtensorMap& tA1, const CUtensorMap& tB1, const CUtensorMap& tA2,
                               const CUtensorMap& tB2, const CUtensorMap& tH, const CUtensorMap& tP, const Workspace& ws,
                               unsigned int* gbar, const uint16_t* x, const uint16_t* Wr, const float* bias,
                               float* logits, uint16_t* y, int T, int H, int I, int E, int k, int grid, int mode,
                               int wave_experts, int lead, int dead_row, bool test_bad_id, const GemmArgs& ga,
                               int trace_ctas, cudaStream_t st) {
  FusedArgs a;
  a.x = x;
  a.Wr = Wr;
  a.bias = bias;
  a.logits = logits;
  a.y = y;
  a.ws = ws;
  a.gbar = gbar;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.workers = grid / PAIR;
  a.mode = mode;
  a.wave_experts = wave_experts;
  a.lead = lead;
  a.dead_row = dead_row;
  a.test_bad_id = test_bad_id ? 1 : 0;
  a.timeout_ns = ga.timeout_ns;
  a.trace_ctas = trace_ctas;
  a.rtok = router_task_tokens(T, E, grid);
  a.ga = ga;
  (void)I;
  using L = Layout<6, 1>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fused_layer_kernel, tA1, tB1, tA2, tB2, tH, tP, a);
}

}  // namespace moe
