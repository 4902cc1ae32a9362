// C ABI of the MoE layer (include/moe_gb300.h): plan, forward, status, debug
// hooks.  Host code only; every step of the layer runs in this library's
// kernels (router_tc.cu, router.cu, dispatch.cu, gemm.cu, combine.cu, and fused.cu for
// the single-launch layer).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kernels.cuh"

using namespace moe;

struct moe_plan_s {
  moe_config_t cfg;
  int device;
  int num_sms;
  int gemm_grid;   // CTAs of the grouped GEMM (all 2-CTA clusters co-resident)
  int fused_grid;  // CTAs of the single-launch layer (all 2-CTA clusters co-resident)
  int64_t R_max, max_mt, max_tiles, R_pad_max;
  void* base;
  size_t bytes;
  void* x_stage;
  void* y_stage[2];   // [1]: MOE_FLAG_HOST_PIPELINE only
  float* bias;
  Workspace ws;
  RouterWs rw;
  cudaEvent_t ev[MOE_NUM_STAGES + 1];
  bool timing;
  // moe_forward_host: x streams in from page-locked host memory on st_aux in HOST_RANGES
  // token ranges, each routed as soon as it has landed
  cudaStream_t st_aux;
  cudaEvent_t ev_fork;    // recorded on st at the start of a host-buffer forward (strict stream order)
  cudaEvent_t ev_xfree;   // MOE_FLAG_HOST_PIPELINE: recorded on st after each forward's gather (or single
                          // launch): x_stage and the routing buffers (last read by Dispatch) are free
  cudaEvent_t ev_routed;  // recorded on st_aux after a pipelined host forward's routing
  cudaEvent_t ev_range[4];
  // MOE_FLAG_HOST_PIPELINE with page-locked y_host: Combine writes y_stage[y_slot] (alternating),
  // whose copy to y_host runs on st_out beside the next forward
  cudaStream_t st_out;
  cudaEvent_t ev_ydone;      // recorded on st after the forward's Combine
  cudaEvent_t ev_yfree[2];   // recorded on st_out after the copy out of y_stage[s]
  cudaEvent_t ev_ylast;      // moe_host_wait: every output copy enqueued so far
  int y_slot;
  int last_launches;
  unsigned long long* trace;   // [max(gemm_grid, fused_grid) + 1][TRACE_SLOTS] when MOE_FLAG_TRACE
  unsigned long long* tile_trace;   // [max_tiles][PAIR][TILE_TRACE_SLOTS] when MOE_FLAG_TRACE
};

namespace {

constexpr int HOST_RANGES = 4;   // token ranges of the pipelined host-to-device transfer
static_assert(HOST_RANGES <= (int)(sizeof(moe_plan_s::ev_range) / sizeof(cudaEvent_t)), "one event per range");

// Everything a plan holds (partially built plans included).
void release(moe_plan_s* p) {
  if (p->timing)
    for (int i = 0; i <= MOE_NUM_STAGES; ++i)
      if (p->ev[i]) cudaEventDestroy(p->ev[i]);
  for (int r = 0; r < HOST_RANGES; ++r)
    if (p->ev_range[r]) cudaEventDestroy(p->ev_range[r]);
  if (p->ev_xfree) cudaEventDestroy(p->ev_xfree);
  if (p->ev_routed) cudaEventDestroy(p->ev_routed);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->st_aux) cudaStreamDestroy(p->st_aux);
  for (int s = 0; s < 2; ++s)
    if (p->ev_yfree[s]) cudaEventDestroy(p->ev_yfree[s]);
  if (p->ev_ydone) cudaEventDestroy(p->ev_ydone);
  if (p->ev_ylast) cudaEventDestroy(p->ev_ylast);
  if (p->st_out) cudaStreamDestroy(p->st_out);
  if (p->base) cudaFree(p->base);
  if (p->bias) cudaFree(p->bias);
  if (p->trace) cudaFree(p->trace);
  if (p->tile_trace) cudaFree(p->tile_trace);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D tensor [outer, inner] (bf16, or fp32 when f32), row pitch = inner * element size; box of
// 128 bytes x box_outer rows, 128-byte swizzle, out-of-bounds elements read as zero.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer,
               bool f32 = false) {
  const uint32_t es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * es_bytes};
  cuuint32_t box[2] = {128 / es_bytes, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Address at which the current device reaches host pointer h, if h lies in page-locked
// memory mapped into its address space and that address is 16-byte aligned; else null.
const void* mapped_host(const void* h) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned16(a.devicePointer)) return nullptr;
  return a.devicePointer;
}
void* mapped_host(void* h) { return const_cast<void*>(mapped_host(static_cast<const void*>(h))); }

moe_status_t validate_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T_max < 1 || c->H < 1 || c->I < 1 || c->E < 1 || c->top_k < 1) return MOE_ERR_INVALID_ARG;
  if (c->schedule < 0 || c->schedule > MOE_SCHED_AUTO || c->wave_experts < 0 || c->lead_waves < 0 ||
      c->timeout_ns < 0)
    return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_GEMM_STREAMING) && (c->flags & MOE_FLAG_GEMM_COMPUTE)) return MOE_ERR_INVALID_ARG;
  if (c->H % SHAPE_ALIGN != 0 || c->I % SHAPE_ALIGN != 0) return MOE_ERR_UNSUPPORTED;
  if (l1_blocks(c->I) >= (1 << 15) || l2_blocks(c->H) >= (1 << 15)) return MOE_ERR_UNSUPPORTED;   // tile field
  if (c->E > MAX_E || c->top_k > MAX_K || c->top_k > c->E) return MOE_ERR_UNSUPPORTED;
  const int64_t R = (int64_t)c->T_max * c->top_k;
  if (R >= (1ll << 30) || (int64_t)c->E * c->H >= (1ll << 31) || (int64_t)c->E * c->I >= (1ll << 31) ||
      (int64_t)c->T_max * c->H >= (1ll << 32))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Sub-buffers of the plan workspace (one allocation), by name.
enum Buf {
  B_IDS, B_W, B_COUNTS, B_OFFSETS, B_ROW_PAIR, B_ROW_OF, B_PROW_OF, B_PROW_W, B_X_PAD, B_H_PAD, B_P_PAD, B_S_PAD,
  B_TILES, B_SCHED, B_READY, B_ERR, B_X_STAGE, B_Y_STAGE, B_WRT, B_NW, B_PART, N_BUFS
};

struct Layout {
  size_t off[N_BUFS];
  size_t total;
};

Layout layout_of(const moe_config_t& c, int64_t R, int64_t max_mt, int64_t max_tiles) {
  // padded rows, plus the dead row (index max_mt * UNIT_ROWS: no unit reaches it; P and its
  // scale are zero there) that Dispatch gives a pair it cannot place
  const int64_t Rp = max_mt * UNIT_ROWS + 1;
  size_t sizes[N_BUFS] = {};
  sizes[B_IDS] = (size_t)R * 4;
  sizes[B_W] = (size_t)R * 4;
  sizes[B_COUNTS] = 16 + (size_t)c.E * 4 * (1 + (c.T_max + DS_CHUNK_TOK - 1) / DS_CHUNK_TOK);   // gbar, counts, chist
  sizes[B_OFFSETS] = (size_t)(c.E + 1) * 4;
  sizes[B_ROW_PAIR] = (size_t)R * 4;
  sizes[B_ROW_OF] = (size_t)R * 4;
  sizes[B_PROW_OF] = (size_t)R * 4;
  sizes[B_PROW_W] = (size_t)Rp * 4;
  sizes[B_X_PAD] = (size_t)Rp * c.H * 2;
  sizes[B_H_PAD] = (size_t)Rp * c.I * 2;
  sizes[B_P_PAD] = (size_t)Rp * c.H * 2;                 // fp16
  sizes[B_S_PAD] = (size_t)Rp * p_scale_blocks(c.H) * 4;   // per-(row, 128 columns) scale of P_pad
  sizes[B_TILES] = (size_t)max_tiles * 16;
  sizes[B_SCHED] = 16;
  sizes[B_READY] = (size_t)max_mt * 4;
  sizes[B_ERR] = 16;
  sizes[B_X_STAGE] = (size_t)c.T_max * c.H * 2;          // moe_forward_host staging
  sizes[B_Y_STAGE] = (size_t)c.T_max * c.H * 2 * ((c.flags & MOE_FLAG_HOST_PIPELINE) ? 2 : 1);
  sizes[B_WRT] = (size_t)c.E * c.H * 2;                  // router: Wr transposed
  sizes[B_NW] = (size_t)c.E * 4;                         // router: column norm bounds
  sizes[B_PART] = (size_t)router_part_rows(c.T_max) * c.E * 4;   // router: split-K partial estimates
  Layout L;
  size_t o = 0;
  for (int i = 0; i < N_BUFS; ++i) {
    L.off[i] = o;
    o += (sizes[i] + 255) & ~(size_t)255;
  }
  L.total = o;
  return L;
}

}  // namespace

namespace {

// Argument checks of moe_forward (before anything is enqueued).
moe_status_t check_forward_args(moe_plan_t p, int32_t T, const void* x, const float* router_logits,
                                const void* W_router, const void* W1, const void* W2, const void* y) {
  if (!p) return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = p->cfg;
  if (T < 0 || T > c.T_max) return MOE_ERR_INVALID_ARG;
  if (!x || !router_logits || !W1 || !W2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_logits) || !aligned16(W1) || !aligned16(W2) || !aligned16(y) ||
      (W_router && !aligned16(W_router)))
    return MOE_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ERR_CUDA;
  if (cur != p->device) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Router of a forward with W_router given.  ROUTER_TC: tensor-core estimates + certified
// canonical selection; ROUTER_CANON_32: canonical logits, 32 tokens x 32 experts per CTA, then
// top-k; ROUTER_CANON_TASKS: canonical logits by tasks of 32, 16 or 8 tokens x 8 experts over
// every SM (top-k in the same kernel for E <= 8).  Routing is the same whichever runs; the
// canonical ones write every logit canonical (MOE_FLAG_EXACT_LOGITS asks for one of them).  The
// rule follows a same-box measurement of each router forced on every shape (router stage, us:
// tensor-core / 32 x 32 / tasks): T=256 H=512 E=8 16.0 / 14.0 / 11.7 (steps 40.2 / 37.9 / 34.2),
// T=1024 E=8 16.1 / 16.0 / 13.7 (steps 42.8 / 40.2 / 37.7), T=4096 H=1024 E=8 21.5 / 22.1 / 17.9;
// H=2048 E=128: T=64 24.2 / 29.5 / 19.9, T=256 26.2 / 29.5 / 22.4, T=512 26.6 / 29.3 / 28.0,
// T=1024 28.3 / 29.8 / 43.6; H=7168 E=256: T=32 48.8 / 71.3 / 32.4, T=128 53.0 / 72.7 / 44.4,
// T=256 47.6 / 73.0 / 61.5, T=512 46.8 / 73.4 / 109.1.  So: the tasks while 32-token tasks
// would fit one per SM, the tensor-core router above (or the 32 x 32 kernel when all logits
// must be canonical).
enum { ROUTER_TC = 0, ROUTER_CANON_32 = 1, ROUTER_CANON_TASKS = 2 };
int router_choice(uint32_t flags, int T, int E, int sms) {
  if (router_tasks(T, E) <= sms) return ROUTER_CANON_TASKS;
  return (flags & MOE_FLAG_EXACT_LOGITS) ? ROUTER_CANON_32 : ROUTER_TC;
}

// CTA rows of the trace buffer (the larger grid of the two launch paths); one more row of
// TRACE_SLOTS values follows them: the phase stamps of a single-launch forward.
int trace_ctas(const moe_plan_s* p) { return p->gemm_grid > p->fused_grid ? p->gemm_grid : p->fused_grid; }
size_t tile_trace_bytes(const moe_plan_s* p) {
  return sizeof(unsigned long long) * PAIR * TILE_TRACE_SLOTS * (size_t)p->max_tiles;
}
// zero both trace buffers before a forward's grouped GEMM (MOE_FLAG_TRACE)
cudaError_t clear_traces(const moe_plan_s* p, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(p->trace, 0, sizeof(unsigned long long) * TRACE_SLOTS * (trace_ctas(p) + 1), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->tile_trace, 0, tile_trace_bytes(p), st);
  return e;
}

// Arguments of the grouped GEMM (both launch paths) other than the tile range.
GemmArgs gemm_args(const moe_plan_s* p) {
  const moe_config_t& c = p->cfg;
  GemmArgs ga;
  ga.tiles = reinterpret_cast<const int4*>(p->ws.tiles);
  ga.sched = p->ws.sched;
  ga.counts = p->ws.counts;
  ga.prow_w = p->ws.prow_w;
  ga.h_pad = p->ws.h_pad;
  ga.P_pad = p->ws.P_pad;
  ga.S_pad = p->ws.S_pad;
  ga.ready = p->ws.ready;
  ga.err = p->ws.err;
  ga.trace = p->trace;
  ga.tile_trace = p->tile_trace;
  ga.range_sel = 2;
  ga.H = c.H;
  ga.I = c.I;
  ga.E = c.E;
  ga.R_pad = (int)p->R_pad_max;
  ga.nL1 = l1_blocks(c.I);
  ga.nL2 = l2_blocks(c.H);
  ga.flags = c.flags;
  ga.timeout_ns = c.timeout_ns;
  return ga;
}

// One forward, enqueued on st.  x_src, when not null, is page-locked host memory mapped into
// the device's address space: the layer's input is copied from it into x (the plan's staging
// buffer) inside this call by the copy engines, on st_aux - in HOST_RANGES token ranges when the
// tensor-core router runs, which starts on each range as soon as it has landed, else whole.  A
// copy into the staging buffer waits for all work enqueued on st before the call, or with
// MOE_FLAG_HOST_PIPELINE only for ev_xfree: the previous forward's gather (or single launch), the
// last kernel that reads x_stage, so it runs beside that forward's later kernels (the copy
// engines need no SM; an SM copy kernel measured slower there) - and the routing follows it
// there (see forward_impl).
cudaError_t wait_staging_free(moe_plan_t p, cudaStream_t st) {
  if (p->cfg.flags & MOE_FLAG_HOST_PIPELINE) return cudaStreamWaitEvent(p->st_aux, p->ev_xfree, 0);
  cudaError_t e = cudaEventRecord(p->ev_fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->st_aux, p->ev_fork, 0);
  return e;
}
cudaError_t stage_whole_input(moe_plan_t p, const void* x_src, size_t bytes, cudaStream_t st) {
  cudaError_t e = wait_staging_free(p, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->x_stage, x_src, bytes, cudaMemcpyDefault, p->st_aux);
  if (e == cudaSuccess) e = cudaEventRecord(p->ev_range[0], p->st_aux);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, p->ev_range[0], 0);
  return e;
}

moe_status_t forward_impl(moe_plan_t p, int32_t T, const void* x, const void* x_src, float* router_logits,
                          const void* W_router, const void* W1, const void* W2, void* y, cudaStream_t st) {
  const moe_config_t& c = p->cfg;
  p->last_launches = 0;
  if (T == 0) return MOE_OK;
  const int k = c.top_k, E = c.E, H = c.H, I = c.I;
  int nl = 0;
  auto rec = [&](int i) {
    if (p->timing) cudaEventRecord(p->ev[i], st);
  };
#define MOE_CK(x)                                   \
  do {                                              \
    if ((x) != cudaSuccess) {                       \
      p->last_launches = nl;                        \
      return MOE_ERR_CUDA;                          \
    }                                               \
  } while (0)
  rec(0);
  const int chunks = (T + DS_CHUNK_TOK - 1) / DS_CHUNK_TOK;
  // grid-barrier word, counts and chist (one contiguous range), zeroed before each forward's routing
  const size_t zero_bytes = 16 + sizeof(int32_t) * E * (1 + chunks);
  if (c.flags & MOE_FLAG_SINGLE_LAUNCH) {
    MOE_CK(cudaMemsetAsync(p->ws.gbar, 0, zero_bytes, st));
    if (x_src) MOE_CK(stage_whole_input(p, x_src, (size_t)T * H * 2, st));   // the input lands whole first
    rec(1);
    rec(2);
    rec(3);
    CUtensorMap tA1, tB1, tA2, tB2, tH, tP;
    const uint64_t Rp = (uint64_t)p->R_pad_max;
    if (!make_tmap(&tA1, p->ws.x_pad, H, Rp, BM) || !make_tmap(&tB1, W1, 2 * I, (uint64_t)E * H, BK) ||
        !make_tmap(&tA2, p->ws.h_pad, I, Rp, BM) || !make_tmap(&tB2, W2, H, (uint64_t)E * I, BK) ||
        !make_tmap(&tH, p->ws.h_pad, I, Rp, 32) || !make_tmap(&tP, p->ws.P_pad, H, Rp, 32)) {
      p->last_launches = nl;
      return MOE_ERR_CUDA;
    }
    GemmArgs ga = gemm_args(p);
    if (p->trace)
      MOE_CK(clear_traces(p, st));
    const int sched_mode = (c.schedule == MOE_SCHED_AUTO) ? MOE_SCHED_WAVE_SERIAL : c.schedule;
    const int sched_we = (c.schedule == MOE_SCHED_AUTO) ? E : c.wave_experts;
    MOE_CK(launch_fused_layer(tA1, tB1, tA2, tB2, tH, tP, p->ws, p->ws.gbar, static_cast<const uint16_t*>(x),
                              static_cast<const uint16_t*>(W_router), p->bias, router_logits,
                              static_cast<uint16_t*>(y), T, H, I, E, k, p->fused_grid, sched_mode, sched_we,
                              c.lead_waves, (int)p->R_pad_max, (c.flags & MOE_FLAG_TEST_BAD_ID) != 0, ga,
                              trace_ctas(p), st));
    ++nl;
    if (c.flags & MOE_FLAG_HOST_PIPELINE)   // x_stage and the routing buffers free for the next forward
      MOE_CK(cudaEventRecord(p->ev_xfree, st));
    rec(4);
    rec(5);
    p->last_launches = nl;
    return MOE_OK;
  }
  const int rchoice = W_router ? router_choice(c.flags, T, E, p->num_sms) : ROUTER_CANON_32;
  const bool tc_router = rchoice == ROUTER_TC;
  // Stream of the routing: with MOE_FLAG_HOST_PIPELINE and a page-locked host input (stage timing
  // off), the plan's copy stream, right behind the input's upload there - both wait only until the
  // previous forward's gather is done (so its Dispatch, the last reader of the routing buffers),
  // and the routing then runs beside that forward's GEMM tail and Combine; st joins it before
  // Dispatch.  Otherwise st, the input copied in ranges (tensor-core router) or whole.
  const bool aside = x_src && (c.flags & MOE_FLAG_HOST_PIPELINE) && !p->timing;
  cudaStream_t sr = aside ? p->st_aux : st;
  if (aside) {
    MOE_CK(wait_staging_free(p, st));
    MOE_CK(cudaMemcpyAsync(p->x_stage, x_src, (size_t)T * H * 2, cudaMemcpyDefault, sr));
  } else if (x_src && !tc_router) {
    MOE_CK(stage_whole_input(p, x_src, (size_t)T * H * 2, st));   // whole copy first
  }
  MOE_CK(cudaMemsetAsync(p->ws.gbar, 0, zero_bytes, sr));
  if (tc_router) {
    // split plan of the whole forward, whatever the ranges: the same logits either way
    const RouterSplit sp = router_split(T, H, E, p->num_sms);
    CUtensorMap tW;
    const int n_pad = ((E + 15) / 16) * 16;
    if (!make_tmap(&tW, p->rw.WrT, H, (uint64_t)E, n_pad)) {
      p->last_launches = nl;
      return MOE_ERR_CUDA;
    }
    // token ranges of whole 128-token chunks: up to HOST_RANGES while x streams in, else one
    // (with MOE_FLAG_HOST_PIPELINE the upload ran beside the previous forward: no range waits)
    const int nr = (x_src && !(c.flags & MOE_FLAG_HOST_PIPELINE)) ? std::min(HOST_RANGES, chunks) : 1;
    const int per = ((chunks + nr - 1) / nr) * DS_CHUNK_TOK;
    if (x_src && !aside) {
      MOE_CK(wait_staging_free(p, st));
      for (int r = 0; r * per < T; ++r) {
        const size_t off = (size_t)r * per * H * 2, n = (size_t)std::min(per, T - r * per) * H * 2;
        MOE_CK(cudaMemcpyAsync(static_cast<char*>(p->x_stage) + off, static_cast<const char*>(x_src) + off, n,
                               cudaMemcpyDefault, p->st_aux));
        MOE_CK(cudaEventRecord(p->ev_range[r], p->st_aux));
      }
    }
    MOE_CK(launch_router_prep(static_cast<const uint16_t*>(W_router), H, E, p->rw, sr));
    ++nl;
    for (int r = 0; r * per < T; ++r) {
      const int t0 = r * per, tn = std::min(per, T - t0);
      if (x_src && !aside) MOE_CK(cudaStreamWaitEvent(st, p->ev_range[r], 0));
      const uint16_t* xr = static_cast<const uint16_t*>(x) + (size_t)t0 * H;
      CUtensorMap tX;
      if (!make_tmap(&tX, xr, H, (uint64_t)tn, 128)) {
        p->last_launches = nl;
        return MOE_ERR_CUDA;
      }
      MOE_CK(launch_router_tc(tX, tW, xr, p->bias, p->rw, sp, tn, H, E, k, p->num_sms,
                              router_logits + (size_t)t0 * E, p->ws.ids + (size_t)t0 * k, p->ws.w + (size_t)t0 * k,
                              p->ws.counts, p->ws.chist + (size_t)(t0 / DS_CHUNK_TOK) * E, p->ws.err, c.timeout_ns,
                              sr));
      nl += 2;
    }
  } else {
    bool topk_done = false;
    if (W_router && rchoice == ROUTER_CANON_TASKS) {
      MOE_CK(launch_router_tasks(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(W_router), p->bias,
                                 router_logits, p->ws, T, H, E, k, p->num_sms, &topk_done, sr));
      ++nl;
    } else if (W_router) {
      MOE_CK(launch_router_logits(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(W_router),
                                  p->bias, router_logits, T, H, E, sr));
      ++nl;
    }
    if (!topk_done) {
      MOE_CK(launch_topk(router_logits, T, E, k, p->ws.ids, p->ws.w, p->ws.counts, p->ws.chist, p->num_sms, sr));
      ++nl;
    }
  }
  if (aside) {
    MOE_CK(cudaEventRecord(p->ev_routed, sr));
    MOE_CK(cudaStreamWaitEvent(st, p->ev_routed, 0));
  }
  rec(1);
  // schedule actually run: MOE_SCHED_AUTO resolves to wave-serial with one wave of all experts
  const int sched_mode = (c.schedule == MOE_SCHED_AUTO) ? MOE_SCHED_WAVE_SERIAL : c.schedule;
  const int sched_we = (c.schedule == MOE_SCHED_AUTO) ? E : c.wave_experts;
  MOE_CK(launch_dispatch(p->ws, T, E, k, H, I, p->gemm_grid / PAIR, sched_mode, sched_we, c.lead_waves,
                         (int)p->R_pad_max, (c.flags & MOE_FLAG_TEST_BAD_ID) != 0, st));
  ++nl;
  rec(2);
  MOE_CK(launch_gather(static_cast<const uint16_t*>(x), p->ws.prow_of, T, H, k, p->ws.x_pad, st));
  if (c.flags & MOE_FLAG_HOST_PIPELINE)   // x_stage and the routing buffers free for the next forward
    MOE_CK(cudaEventRecord(p->ev_xfree, st));
  ++nl;
  rec(3);
  CUtensorMap tA1, tB1, tA2, tB2, tH, tP;
  const uint64_t Rp = (uint64_t)p->R_pad_max;
  if (!make_tmap(&tA1, p->ws.x_pad, H, Rp, BM) || !make_tmap(&tB1, W1, 2 * I, (uint64_t)E * H, BK) ||
      !make_tmap(&tA2, p->ws.h_pad, I, Rp, BM) || !make_tmap(&tB2, W2, H, (uint64_t)E * I, BK) ||
      !make_tmap(&tH, p->ws.h_pad, I, Rp, 32) || !make_tmap(&tP, p->ws.P_pad, H, Rp, 32)) {
    p->last_launches = nl;
    return MOE_ERR_CUDA;
  }
  GemmArgs ga = gemm_args(p);
  if (p->trace)
    MOE_CK(clear_traces(p, st));
  const bool streaming = !(c.flags & MOE_FLAG_GEMM_COMPUTE);   // the deeper operand ring by default
  if (c.schedule == MOE_SCHED_PHASED) {
    ga.range_sel = 0;
    MOE_CK(launch_grouped_gemm(tA1, tB1, tA2, tB2, tH, tP, ga, p->gemm_grid, streaming, st));
    ga.range_sel = 1;
    MOE_CK(launch_grouped_gemm(tA1, tB1, tA2, tB2, tH, tP, ga, p->gemm_grid, streaming, st));
    nl += 2;
  } else {
    ga.range_sel = 2;
    MOE_CK(launch_grouped_gemm(tA1, tB1, tA2, tB2, tH, tP, ga, p->gemm_grid, streaming, st));
    ++nl;
  }
  rec(4);
  MOE_CK(launch_combine(p->ws.P_pad, p->ws.S_pad, p->ws.prow_of, T, H, k, static_cast<uint16_t*>(y), p->num_sms,
                        st));
  ++nl;
  rec(5);
#undef MOE_CK
  p->last_launches = nl;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

moe_status_t moe_workspace_bytes(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const int64_t R = (int64_t)cfg->T_max * cfg->top_k;
  const int64_t max_mt = max_mtiles(R, cfg->E);
  const int64_t max_tiles = max_mt * (l1_blocks(cfg->I) + l2_blocks(cfg->H));
  *bytes = layout_of(*cfg, R, max_mt, max_tiles).total;
  return MOE_OK;
}

moe_status_t moe_plan(const moe_config_t* cfg, int device, moe_plan_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status_t st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!get_encode()) return MOE_ERR_CUDA;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_INVALID_ARG;
  moe_plan_s* p = new (std::nothrow) moe_plan_s();
  if (!p) return MOE_ERR_OOM;
  p->cfg = *cfg;
  p->cfg.router_bias = nullptr;
  if (p->cfg.timeout_ns == 0) p->cfg.timeout_ns = 1000000000ll;
  if (p->cfg.lead_waves == 0) p->cfg.lead_waves = 1;
  p->device = device;
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, device);
  p->R_max = (int64_t)cfg->T_max * cfg->top_k;
  p->max_mt = max_mtiles(p->R_max, cfg->E);
  p->max_tiles = p->max_mt * (l1_blocks(cfg->I) + l2_blocks(cfg->H));
  p->R_pad_max = p->max_mt * UNIT_ROWS;
  Layout L = layout_of(*cfg, p->R_max, p->max_mt, p->max_tiles);
  p->bytes = L.total;
  auto fail = [&](moe_status_t s) {
    release(p);
    delete p;
    cudaSetDevice(cur);
    return s;
  };
  if (cudaMalloc(&p->base, L.total) != cudaSuccess) {
    cudaGetLastError();
    p->base = nullptr;
    return fail(MOE_ERR_OOM);
  }
  char* b = static_cast<char*>(p->base);
  auto at = [&](Buf i) { return b + L.off[i]; };
  p->ws.ids = reinterpret_cast<int32_t*>(at(B_IDS));
  p->ws.w = reinterpret_cast<float*>(at(B_W));
  p->ws.gbar = reinterpret_cast<unsigned int*>(at(B_COUNTS));
  p->ws.counts = reinterpret_cast<int32_t*>(at(B_COUNTS) + 16);
  p->ws.chist = p->ws.counts + cfg->E;
  p->ws.offsets = reinterpret_cast<int32_t*>(at(B_OFFSETS));
  p->ws.row_pair = reinterpret_cast<int32_t*>(at(B_ROW_PAIR));
  p->ws.row_of = reinterpret_cast<int32_t*>(at(B_ROW_OF));
  p->ws.prow_of = reinterpret_cast<int32_t*>(at(B_PROW_OF));
  p->ws.prow_w = reinterpret_cast<float*>(at(B_PROW_W));
  p->ws.x_pad = reinterpret_cast<uint16_t*>(at(B_X_PAD));
  p->ws.h_pad = reinterpret_cast<uint16_t*>(at(B_H_PAD));
  p->ws.P_pad = reinterpret_cast<uint16_t*>(at(B_P_PAD));
  p->ws.S_pad = reinterpret_cast<float*>(at(B_S_PAD));
  p->ws.tiles = reinterpret_cast<int32_t*>(at(B_TILES));
  p->ws.sched = reinterpret_cast<int32_t*>(at(B_SCHED));
  p->ws.ready = reinterpret_cast<int32_t*>(at(B_READY));
  p->ws.err = reinterpret_cast<uint32_t*>(at(B_ERR));
  p->x_stage = at(B_X_STAGE);
  p->y_stage[0] = at(B_Y_STAGE);
  p->y_stage[1] = (cfg->flags & MOE_FLAG_HOST_PIPELINE) ? at(B_Y_STAGE) + (size_t)cfg->T_max * cfg->H * 2 : nullptr;
  p->rw.WrT = reinterpret_cast<uint16_t*>(at(B_WRT));
  p->rw.nw = reinterpret_cast<float*>(at(B_NW));
  p->rw.part = reinterpret_cast<float*>(at(B_PART));
  if (cudaMemset(p->ws.err, 0, 16) != cudaSuccess) return fail(MOE_ERR_CUDA);
  {   // the dead row: P and its scales zero, so a pair sent there adds nothing in Combine
    const size_t dead = (size_t)p->R_pad_max, nS = (size_t)p_scale_blocks(cfg->H);
    if (cudaMemset(p->ws.P_pad + dead * cfg->H, 0, (size_t)cfg->H * 2) != cudaSuccess ||
        cudaMemset(p->ws.S_pad + dead * nS, 0, nS * 4) != cudaSuccess)
      return fail(MOE_ERR_CUDA);
  }
  if (cfg->router_bias) {
    if (cudaMalloc(&p->bias, sizeof(float) * cfg->E) != cudaSuccess) {
      cudaGetLastError();
      p->bias = nullptr;
      return fail(MOE_ERR_OOM);
    }
    if (cudaMemcpy(p->bias, cfg->router_bias, sizeof(float) * cfg->E, cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(MOE_ERR_CUDA);
  }
  if (gemm_prepare(device, &p->gemm_grid) != cudaSuccess || router_prepare() != cudaSuccess ||
      router_tc_prepare() != cudaSuccess || router_tasks_prepare() != cudaSuccess ||
      fused_prepare(device, &p->fused_grid) != cudaSuccess)
    return fail(MOE_ERR_CUDA);
  if (cfg->flags & MOE_FLAG_TRACE) {
    if (cudaMalloc(&p->trace, sizeof(unsigned long long) * TRACE_SLOTS * (trace_ctas(p) + 1)) != cudaSuccess) {
      cudaGetLastError();
      p->trace = nullptr;
      return fail(MOE_ERR_OOM);
    }
    if (cudaMalloc(&p->tile_trace, tile_trace_bytes(p)) != cudaSuccess) {
      cudaGetLastError();
      p->tile_trace = nullptr;
      return fail(MOE_ERR_OOM);
    }
  }
  p->timing = (cfg->flags & MOE_FLAG_STAGE_TIMING) != 0;
  if (p->timing)
    for (int i = 0; i <= MOE_NUM_STAGES; ++i)
      if (cudaEventCreate(&p->ev[i]) != cudaSuccess) return fail(MOE_ERR_CUDA);
  if (cudaStreamCreateWithFlags(&p->st_aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_xfree, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_routed, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p->st_out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_ydone, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_ylast, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_yfree[0], cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_yfree[1], cudaEventDisableTiming) != cudaSuccess)
    return fail(MOE_ERR_CUDA);
  for (int r = 0; r < HOST_RANGES; ++r)
    if (cudaEventCreateWithFlags(&p->ev_range[r], cudaEventDisableTiming) != cudaSuccess) return fail(MOE_ERR_CUDA);
  cudaSetDevice(cur);
  *out = p;
  return MOE_OK;
}

moe_status_t moe_forward(moe_plan_t p, int32_t T, const void* x, float* router_logits, const void* W_router,
                         const void* W1, const void* W2, void* y, void* stream) {
  const moe_status_t v = check_forward_args(p, T, x, router_logits, W_router, W1, W2, y);
  if (v != MOE_OK) return v;
  return forward_impl(p, T, x, nullptr, router_logits, W_router, W1, W2, y, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_host(moe_plan_t p, int32_t T, const void* x_host, float* router_logits,
                              const void* W_router, const void* W1, const void* W2, void* y_host, void* stream) {
  if (!p || !x_host || !y_host) return MOE_ERR_INVALID_ARG;
  // Page-locked buffers: x streams in by the copy engines in token ranges (overlapping the
  // router, and the previous forward's later kernels), Combine writes y in place - or, with
  // MOE_FLAG_HOST_PIPELINE, into the alternating staging buffers that the copy engines drain
  // on st_out beside the next forward.  Pageable ones go through the copy engines and the
  // staging buffers whole.
  const bool pipe = (p->cfg.flags & MOE_FLAG_HOST_PIPELINE) != 0;
  const void* x_dev = mapped_host(x_host);
  void* y_dev = mapped_host(y_host);
  const bool y_out = pipe && y_dev;   // y leaves on st_out
  const int slot = y_out ? p->y_slot : 0;
  void* y = (y_dev && !y_out) ? y_dev : p->y_stage[slot];
  const moe_status_t v = check_forward_args(p, T, p->x_stage, router_logits, W_router, W1, W2, y);
  if (v != MOE_OK) return v;
  if (T == 0) {
    p->last_launches = 0;
    return MOE_OK;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * p->cfg.H * 2;
  // the staging buffer Combine writes has been copied out (a no-op until a first copy)
  if (pipe && cudaStreamWaitEvent(st, p->ev_yfree[slot], 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (!x_dev) {   // pageable: the copy engines, on st_aux once x_stage is free (as stage_whole_input)
    if (wait_staging_free(p, st) != cudaSuccess ||
        cudaMemcpyAsync(p->x_stage, x_host, bytes, cudaMemcpyHostToDevice, p->st_aux) != cudaSuccess ||
        cudaEventRecord(p->ev_range[0], p->st_aux) != cudaSuccess || cudaStreamWaitEvent(st, p->ev_range[0], 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  const moe_status_t s = forward_impl(p, T, p->x_stage, x_dev, router_logits, W_router, W1, W2, y, st);
  if (s != MOE_OK) return s;
  if (y_out) {
    if (cudaEventRecord(p->ev_ydone, st) != cudaSuccess || cudaStreamWaitEvent(p->st_out, p->ev_ydone, 0) != cudaSuccess ||
        cudaMemcpyAsync(y_host, y, bytes, cudaMemcpyDeviceToHost, p->st_out) != cudaSuccess ||
        cudaEventRecord(p->ev_yfree[slot], p->st_out) != cudaSuccess)
      return MOE_ERR_CUDA;
    p->y_slot ^= 1;
    return MOE_OK;
  }
  if (!y_dev && cudaMemcpyAsync(y_host, p->y_stage[0], bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (pipe && cudaEventRecord(p->ev_yfree[0], st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_host_wait(moe_plan_t p, void* stream) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (cudaEventRecord(p->ev_ylast, p->st_out) != cudaSuccess ||
      cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), p->ev_ylast, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_get_status(moe_plan_t p, void* stream) {
  if (!p) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess || cudaStreamSynchronize(p->st_aux) != cudaSuccess ||
      cudaStreamSynchronize(p->st_out) != cudaSuccess)
    return MOE_ERR_CUDA;
  uint32_t e = 0;
  if (cudaMemcpy(&e, p->ws.err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (e != 0 && cudaMemset(p->ws.err, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  if (e & ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (e & ERR_CHECK) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

moe_status_t moe_debug_routing(moe_plan_t p, int32_t T, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                               int32_t* row_pair, int32_t* row_of, void* stream) {
  if (!p || T < 0 || T > p->cfg.T_max) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t R = (size_t)T * p->cfg.top_k;
  const size_t E = p->cfg.E;
  auto cp = [&](void* dst, const void* src, size_t n) {
    return (dst && n) ? cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, st) : cudaSuccess;
  };
  if (cp(ids, p->ws.ids, R * 4) || cp(w, p->ws.w, R * 4) || cp(counts, p->ws.counts, E * 4) ||
      cp(offsets, p->ws.offsets, (E + 1) * 4) || cp(row_pair, p->ws.row_pair, R * 4) ||
      cp(row_of, p->ws.row_of, R * 4))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_debug_intermediates(moe_plan_t p, int32_t T, void* h, float* P, void* stream) {
  if (!p || T < 0 || T > p->cfg.T_max) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t R = (size_t)T * p->cfg.top_k;
  if (R && (h || P) &&
      launch_compact_intermediates(p->ws.row_pair, p->ws.prow_of, (int)R, (int)p->R_pad_max + 1, p->cfg.H, p->cfg.I,
                                   p->ws.h_pad,
                                   p->ws.P_pad, p->ws.S_pad, static_cast<uint16_t*>(h), P, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_stage_times(moe_plan_t p, float* ms) {
  if (!p || !ms || !p->timing) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_NUM_STAGES; ++i) {
    if (cudaEventSynchronize(p->ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventElapsedTime(&ms[i], p->ev[i], p->ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t moe_trace_read(moe_plan_t p, uint64_t* host_buf, size_t cap, size_t* n) {
  if (!p || !n || !p->trace) return MOE_ERR_INVALID_ARG;
  const size_t cnt = (size_t)TRACE_SLOTS * (trace_ctas(p) + 1);
  *n = cnt;
  if (!host_buf) return MOE_OK;
  if (cap < cnt) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(host_buf, p->trace, cnt * sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_trace_tiles(moe_plan_t p, uint64_t* host_buf, size_t cap, size_t* n) {
  if (!p || !n || !p->tile_trace) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t sc[4] = {0, 0, 0, 0};
  if (p->last_launches > 0 && cudaMemcpy(sc, p->ws.sched, sizeof(sc), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  const size_t tiles = (sc[1] > 0 && sc[1] <= p->max_tiles) ? (size_t)sc[1] : 0;
  const size_t cnt = tiles * PAIR * TILE_TRACE_SLOTS;
  *n = cnt;
  if (!host_buf || cnt == 0) return MOE_OK;
  if (cap < cnt) return MOE_ERR_INVALID_ARG;
  if (cudaMemcpy(host_buf, p->tile_trace, cnt * sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_router_bound(moe_plan_t p, int32_t T, float* cH) {
  if (!p || !cH || T < 1 || T > p->cfg.T_max) return MOE_ERR_INVALID_ARG;
  *cH = router_bound_coef(p->cfg.H, router_split(T, p->cfg.H, p->cfg.E, p->num_sms));
  return MOE_OK;
}

moe_status_t moe_last_launch_count(moe_plan_t p, int32_t* n) {
  if (!p || !n) return MOE_ERR_INVALID_ARG;
  *n = p->last_launches;
  return MOE_OK;
}

moe_status_t moe_plan_destroy(moe_plan_t p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  int cur = 0;
  cudaGetDevice(&cur);
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  release(p);
  cudaSetDevice(cur);
  delete p;
  return MOE_OK;
}

moe_status_t moe_debug_schedule(moe_plan_t p, int32_t* tiles_out, int64_t cap, int64_t* n_out, void* stream) {
  if (!p || !n_out) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t sc[4] = {0, 0, 0, 0};
  if (p->last_launches > 0 && cudaMemcpy(sc, p->ws.sched, sizeof(sc), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  n_out[0] = sc[0];
  n_out[1] = sc[1];
  n_out[2] = ((p->cfg.flags & MOE_FLAG_SINGLE_LAUNCH) ? p->fused_grid : p->gemm_grid) / PAIR;
  if (tiles_out && sc[1] > 0) {
    if (cap < sc[1]) return MOE_ERR_INVALID_ARG;
    if (cudaMemcpy(tiles_out, p->ws.tiles, sizeof(int32_t) * 4 * (size_t)sc[1], cudaMemcpyDeviceToHost) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t moe_schedule_host(const int32_t* counts, int32_t E, int32_t H, int32_t I, int32_t num_sms,
                               int32_t schedule, int32_t wave_experts, int32_t lead_waves, int32_t* tiles_out,
                               int64_t cap, int64_t* n_out) {
  if (!counts || !n_out || E < 1 || E > MAX_E || H < 1 || I < 1 || H % SHAPE_ALIGN || I % SHAPE_ALIGN || num_sms < 1 || schedule < 0 ||
      schedule > 2)
    return MOE_ERR_INVALID_ARG;
  SchedTables* s = new (std::nothrow) SchedTables();
  if (!s) return MOE_ERR_OOM;
  sched_build(*s, counts, E, l1_blocks(I), l2_blocks(H), num_sms, schedule, wave_experts,
              lead_waves == 0 ? 1 : lead_waves);
  n_out[0] = s->n1_total;
  n_out[1] = s->total;
  if (tiles_out) {
    if (cap < s->total) {
      delete s;
      return MOE_ERR_INVALID_ARG;
    }
    for (int g = 0; g < s->total_mt; ++g) sched_emit_mtile(*s, g, tiles_out);
  }
  delete s;
  return MOE_OK;
}

}  // extern "C"
