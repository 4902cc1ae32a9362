// Host-side launchers of the MoE layer kernels (internal to libmoe_gb300.so).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace moe {

// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel of the stream drains; every kernel launched this way calls
// ptx::grid_dep_wait() before its first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Row spaces: "compact" rows 0..R-1 group the (token, slot) pairs by expert
// (row_pair / row_of, as returned by moe_debug_routing); "padded" rows give every
// 256-row unit of an expert its own block (unit g owns rows 256 g .. 256 g + 255),
// so the grouped GEMM loads and stores whole 128-row boxes without touching another
// expert's rows.  x_pad, h_pad and P_pad are indexed by padded row.
// Tokens per chunk of Dispatch's counting sort; the router counts each chunk's pairs
// per expert.
constexpr int DS_CHUNK_TOK = 128;

struct Workspace {
  int32_t* ids;       // [T_max*k]
  float* w;           // [T_max*k]
  int32_t* counts;    // [E]
  int32_t* chist;     // [ceil(T_max / DS_CHUNK_TOK) * E] expert counts per chunk of tokens (follows counts)
  int32_t* offsets;   // [E+1] compact
  int32_t* row_pair;  // [R_max] compact row -> t*k+j
  int32_t* row_of;    // [R_max] t*k+j -> compact row
  int32_t* prow_of;   // [R_max] t*k+j -> padded row
  float* prow_w;      // [R_pad_max] router weight of each padded row (valid rows only)
  uint16_t* x_pad;    // [R_pad_max, H] bf16
  uint16_t* h_pad;    // [R_pad_max, I] bf16
  uint16_t* P_pad;    // [R_pad_max, H] fp16: w[t,j] * expert output / S_pad
  float* S_pad;       // [R_pad_max, H/128] fp32 powers of two: scale of each 128-column block of P_pad
  int32_t* tiles;     // [max_tiles*4]
  int32_t* sched;     // [4]: linear-1 tiles, total tiles, units
  int32_t* ready;     // [max_units]
  uint32_t* err;      // [1]
  unsigned long long* trace;   // [gemm grid][TRACE_SLOTS] wait-time counters (MOE_FLAG_TRACE)
  unsigned int* gbar; // [4] grid-barrier arrivals of the single-launch layer (just before counts; zeroed with them)
};

// Per-CTA counters of the grouped GEMM under MOE_FLAG_TRACE (nanoseconds unless noted).
enum TraceSlot {
  TR_PROD_WAIT_EMPTY = 0,  // producer blocked on a free stage
  TR_PROD_WAIT_READY = 1,  // producer blocked on Linear-1 readiness of a Linear-2 tile
  TR_MMA_WAIT_TEMPTY = 2,  // MMA issuer blocked on a free TMEM accumulator (epilogue behind)
  TR_MMA_WAIT_FULL = 3,    // MMA issuer blocked on operands (loads behind)
  TR_EPI_WAIT_TFULL = 4,   // epilogue blocked on an accumulator (MMA behind)
  TR_KERNEL_NS = 5,        // CTA lifetime
  TR_TILES_L1 = 6,         // Linear-1 tiles (count)
  TR_TILES_L2 = 7,         // Linear-2 tiles (count)
  TRACE_SLOTS = 8
};
// Per-tile records of the grouped GEMM under MOE_FLAG_TRACE: for tile i of the tile list
// and CTA rank r of its cluster, 4 values at tile_trace[(2 i + r) * 4]: the SM id, then the
// %globaltimer (ns) when the CTA's producer started the tile, when its accumulator was ready
// for the epilogue, and when the epilogue finished it (Linear-1: its h rows written, just
// before the unit's readiness count is raised; Linear-2: the last P stores issued).
enum TileTraceSlot { TT_SMID = 0, TT_START = 1, TT_ACC = 2, TT_END = 3, TILE_TRACE_SLOTS = 4 };

struct GemmArgs {
  const int4* tiles;
  const int32_t* sched;
  const int32_t* counts;
  const float* prow_w;
  uint16_t* h_pad;     // direct stores of partial quadrants
  uint16_t* P_pad;    // fp16
  float* S_pad;
  int32_t* ready;
  uint32_t* err;
  unsigned long long* trace;
  unsigned long long* tile_trace;   // [tiles][PAIR][TILE_TRACE_SLOTS] (MOE_FLAG_TRACE) or null
  int range_sel;  // 0: linear-1 tiles, 1: linear-2 tiles, 2: all, 3: none
  int H, I, E, R_pad, nL1, nL2;
  uint32_t flags;
  int64_t timeout_ns;
};

cudaError_t router_prepare();

// Tensor-core router with certified exact selection (router_tc.cu).
constexpr int ROUTER_MAX_SPLITS = 16;   // K splits of the logit estimate
struct RouterSplit {
  int m_tiles, splits, kb_total, kb_per;
  int n_chain;       // TMEM accumulators per CTA, K blocks dealt round-robin
  int chain_steps;   // 16-deep MMA steps of the longest chain
};
struct RouterWs {
  uint16_t* WrT;    // [E][H] bf16: Wr transposed
  float* nw;        // [E] upper bounds of the column norms
  float* part;      // [splits][T][E] fp32 partial estimates
};
// Rows of `part` needed for any T <= T_max (splits * T is at most this).
inline int64_t router_part_rows(int64_t T_max) {
  const int64_t tp = (T_max + 127) / 128 * 128;
  const int64_t split_rows = 32768 < ROUTER_MAX_SPLITS * tp ? 32768 : ROUTER_MAX_SPLITS * tp;
  return tp > split_rows ? tp : split_rows;
}
cudaError_t router_tc_prepare();
RouterSplit router_split(int T, int H, int E, int num_sms);
float router_bound_coef(int H, const RouterSplit& r);
// WrT = Wr^T (once per forward, before any launch_router_tc).
cudaError_t launch_router_prep(const uint16_t* Wr, int H, int E, const RouterWs& rw, cudaStream_t st);
// Tensor-core estimates + certified selection for T tokens starting at x (tmX covers those T
// rows; logits, ids, w and chist point at the range's first token, which starts a 128-token
// chunk), with the split plan sp - planned for the whole forward, so that a forward routed in
// several ranges writes the same logits as one routed in a single call.
cudaError_t launch_router_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, const uint16_t* x, const float* bias,
                             const RouterWs& rw, const RouterSplit& sp, int T, int H, int E, int k, int num_sms,
                             float* logits, int32_t* ids, float* w, int32_t* counts, int32_t* chist,
                             uint32_t* err, int64_t timeout_ns, cudaStream_t st);
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* Wr, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t st);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                        int32_t* chist, int num_sms, cudaStream_t st);
// A pair that inconsistent routing leaves without a row (reported as ERR_CHECK) gets dead_row:
// a padded row past every unit whose P and scale are zero.  test_bad_id (test only): Dispatch
// sees pair 0's expert id out of range.
cudaError_t launch_dispatch(const Workspace& ws, int T, int E, int k, int H, int I, int num_sms, int mode,
                            int wave_experts, int lead, int dead_row, bool test_bad_id, cudaStream_t st);
cudaError_t launch_gather(const uint16_t* x, const int32_t* prow_of, int T, int H, int k, uint16_t* x_pad,
                          cudaStream_t st);
cudaError_t launch_compact_intermediates(const int32_t* row_pair, const int32_t* prow_of, int R, int R_pad, int H,
                                         int I,
                                         const uint16_t* h_pad, const uint16_t* P_pad, const float* S_pad,
                                         uint16_t* h, float* P,
                                         cudaStream_t st);
cudaError_t gemm_prepare(int device, int* grid);   // grid: CTAs of the co-resident 2-CTA clusters
cudaError_t launch_grouped_gemm(const CUtensorMap& tA1, const CUtensorMap& tB1, const CUtensorMap& tA2,
                                const CUtensorMap& tB2, const CUtensorMap& tH, const CUtensorMap& tP,
                                const GemmArgs& a, int grid, bool streaming, cudaStream_t st);
// Canonical router logits by tasks of 32, 16 or 8 tokens x 8 experts, one CTA each (fused.cu,
// the single launch's router phase as a kernel of its own); with E <= 8 the same CTAs also select
// the top-k (*topk_done = true), else the caller runs launch_topk.  router_tasks: the number of
// 32-token tasks (the router rule's measure of batch size).
cudaError_t router_tasks_prepare();
int router_tasks(int T, int E);
cudaError_t launch_router_tasks(const uint16_t* x, const uint16_t* Wr, const float* bias, float* logits,
                                const Workspace& ws, int T, int H, int E, int k, int num_sms, bool* topk_done,
                                cudaStream_t st);
// The whole layer as one launch (fused.cu): grid = the co-resident 2-CTA clusters of that kernel.
cudaError_t fused_prepare(int device, int* grid);
cudaError_t launch_fused_layer(const CUtensorMap& tA1, const CUtensorMap& tB1, const CUtensorMap& tA2,
                               const CUtensorMap& tB2, const CUtensorMap& tH, const CUtensorMap& tP, const Workspace& ws,
                               unsigned int* gbar, const uint16_t* x, const uint16_t* Wr, const float* bias,
                               float* logits, uint16_t* y, int T, int H, int I, int E, int k, int grid, int mode,
                               int wave_experts, int lead, int dead_row, bool test_bad_id, const GemmArgs& ga,
                               int trace_ctas, cudaStream_t st);
cudaError_t launch_combine(const uint16_t* P_pad, const float* S_pad, const int32_t* prow_of, int T, int H, int k,
                           uint16_t* y, int num_sms,
                           cudaStream_t st);

}  // namespace moe
