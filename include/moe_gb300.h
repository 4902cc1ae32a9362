/* moe_gb300.h - C ABI of the single-GPU mixture-of-experts layer (GB300, sm_103a).
 *
 * The operation is the expert layer described in "X-Stage: An Overlooked
 * Pipeline Stage for Communication-Computation Overlap in DiT Inference",
 * MegaMoE background paragraph: a router selects the top-k experts of every
 * token; Dispatch moves each token to its experts; each expert applies
 * Linear-1 (hidden H -> intermediate I), the SwiGLU activation (Shazeer 2020,
 * cited there) and Linear-2 (I -> H); Combine brings the k expert outputs
 * back to the token and sums them weighted by the router weights.  On one
 * GPU, Dispatch and Combine are permutations inside device memory.
 *
 * Numerics (fixed by this library; the page leaves them open):
 *   - logits[t,e] = sum_h x[t,h]*Wr[h,e] (+bias[e]) in fp32 in one canonical
 *     order: 32 partial sums, partial j over h = j, j+32, ... with fused
 *     multiply-adds, then pairwise (j, j+16), (j, j+8), (j, j+4), (j, j+2),
 *     (j, j+1) additions;
 *   - top-k by descending logit, ties to the lower expert id, NaN below -inf;
 *     weights = softmax over the k selected logits;
 *   - Linear-1 / Linear-2: bf16 inputs, fp32 accumulation on the tensor cores;
 *     the SwiGLU intermediate silu(g)*u is rounded to bf16; Linear-2's output
 *     is scaled by the router weight in fp32;
 *   - Combine: fp32 sum over the k slots in slot order j = 0..k-1, rounded to
 *     bf16.  Results are bitwise reproducible run to run and across schedules.
 *
 * Memory: every tensor argument is a DEVICE pointer owned by the caller,
 * 16-byte aligned, row-major and densely packed.  The plan owns only its
 * workspace (sized for T_max at plan time) and never frees caller memory.
 *
 * Errors: arguments are validated on the host before anything is launched
 * (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED, nothing enqueued).  Launch
 * failures return MOE_ERR_CUDA.  Problems detected on the device (a wait that
 * ran past timeout_ns, an index out of range) set a sticky error word in the
 * plan that moe_get_status() reports (MOE_ERR_TIMEOUT / MOE_ERR_DEVICE_CHECK);
 * no kernel of this library traps or spins without a time limit.
 *
 * Threading: a plan may be used by one stream at a time.
 *
 * Concurrency between plans: the grouped GEMM is one persistent launch sized to the SMs,
 * and with MOE_SCHED_WAVE_SERIAL, MOE_SCHED_INTERLEAVED and MOE_SCHED_AUTO its Linear-2 tiles
 * wait for Linear-1 tiles that other CTAs of the same launch compute, so all its CTAs must
 * be resident together.  Forwards of different plans on one device may overlap (different
 * streams, no ordering) only if every overlapping plan uses MOE_SCHED_PHASED, whose two
 * launches never wait on other CTAs; otherwise order them (one stream, or events): two such
 * GEMMs that each got part of the SMs can wait on each other until timeout_ns expires and
 * the forward reports MOE_ERR_TIMEOUT.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, T out of range, bad config value   */
  MOE_ERR_UNSUPPORTED = 2,  /* shape outside the supported set (see moe_config_t)          */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                           */
  MOE_ERR_OOM = 4,          /* workspace allocation failed                                 */
  MOE_ERR_TIMEOUT = 5,      /* a device-side wait ran past timeout_ns (reported by status) */
  MOE_ERR_DEVICE_CHECK = 6  /* a device-side consistency check failed (reported by status) */
} moe_status_t;

/* Tile schedules of the grouped GEMMs.  An expert wave is a run of
 * consecutive experts (the X-Stage paper's MegaMoE discussion: waves group
 * local experts; the original schedule runs a wave's Linear-1 and then its
 * Linear-2 before the next wave; the cross-wave interleave places later
 * waves' Linear-1 tiles between the current wave's Linear-2 tiles). */
#define MOE_SCHED_WAVE_SERIAL 0 /* L1(w0) L2(w0) L1(w1) L2(w1) ... in one persistent launch      */
#define MOE_SCHED_INTERLEAVED 1 /* L1(w0..wD-1), then L2(w) merged with L1(w+D), D = lead_waves  */
#define MOE_SCHED_PHASED 2      /* all Linear-1 tiles in one launch, then all Linear-2 tiles     */
#define MOE_SCHED_AUTO 3        /* chosen per forward; currently always wave-serial with one wave
                                   of all experts (every Linear-1 tile, then every Linear-2 tile,
                                   one launch): measured fastest or tied on every workload tried,
                                   since one GPU has no Combine-store backpressure to shape       */

/* flags */
#define MOE_FLAG_ACT_BILINEAR (1u << 0) /* activation g*u instead of silu(g)*u (GLU "bilinear"
                                           variant, same paper as SwiGLU); used by exactness tests */
#define MOE_FLAG_STAGE_TIMING (1u << 1) /* record CUDA events between stages (moe_stage_times)    */
#define MOE_FLAG_TRACE (1u << 2)        /* grouped GEMM records per-CTA wait times (moe_trace_read)
                                           and per-tile SM ids and timestamps (moe_trace_tiles)    */
/* Shared-memory split of the grouped GEMM (results are bit-identical).  Default: a 6-stage
 * operand ring with one output staging buffer (measured faster on every workload tried, from
 * weight streaming to 1k rows per expert).  MOE_FLAG_GEMM_COMPUTE selects a 5-stage ring with
 * two output staging buffers; MOE_FLAG_GEMM_STREAMING names the default explicitly; setting
 * both is an invalid argument. */
#define MOE_FLAG_GEMM_STREAMING (1u << 3) /* 6-stage operand ring, one output staging buffer   */
#define MOE_FLAG_GEMM_COMPUTE (1u << 4)   /* 5-stage operand ring, two output staging buffers  */
/* Router (W_router != NULL).  Routing is always the top-k of the canonical fp32 logits (per
 * logit: 32 partial sums, partial j accumulating h = j (mod 32) in ascending h with fused
 * multiply-adds, then the pairwise tree (j, j+16), (j, j+8), ..., (j, j+1), then + bias).
 * Default: tensor-core estimates of all logits plus an a-priori error bound; only experts the
 * bound cannot exclude from the top-k get their canonical logit evaluated.  The logits row
 * written out then holds canonical values for those experts (always including the k selected)
 * and the tensor-core estimate (+ bias) elsewhere, within
 *   d = cH * ||x_t||_2 * ||Wr[:,e]||_2 + 2^-20 (|estimate - bias| + |bias|) of the canonical value,
 *   cH from moe_router_bound (at most (H/16 + 1) 2^-17 + (H/32 + 8 + 64) 2^-22).
 * MOE_FLAG_EXACT_LOGITS evaluates every logit in the canonical order on the CUDA cores; so does
 * the default where that measured faster (every logit then canonical): batches of at most
 * (number of SMs) tasks of 32 tokens x 8 experts, i.e. ceil(T/32) * ceil(E/8) <= SMs. */
#define MOE_FLAG_EXACT_LOGITS (1u << 5)
/* The whole layer as ONE kernel launch (after the per-forward memset of the expert counts):
 * the MegaMoE design of the X-Stage paper's introduction - one persistent kernel for routing,
 * Dispatch, Linear-1, the activation, Linear-2 and Combine.  The kernel runs on the grouped
 * GEMM's grid and goes through the steps as phases separated by grid-wide barriers (each
 * bounded by timeout_ns; on expiry MOE_ERR_TIMEOUT as for any device wait).  The router is
 * the all-canonical one (as MOE_FLAG_EXACT_LOGITS: every logit written is canonical), and y,
 * the logits and the routing are bitwise those of the multi-launch path with
 * MOE_FLAG_EXACT_LOGITS.  It removes the launch gaps between the steps, which dominate when a
 * forward holds few tokens; with many tokens the multi-launch path (tensor-core router)
 * is faster.  MOE_SCHED_PHASED runs its tile list in the one launch; MOE_FLAG_GEMM_COMPUTE is
 * ignored (the default ring split); with MOE_FLAG_STAGE_TIMING the whole launch is reported
 * as stage 3 (the grouped GEMM) and the other stages as 0. */
#define MOE_FLAG_SINGLE_LAUNCH (1u << 6)
/* moe_forward_host only (library plumbing: no counterpart in the paper): pipelined host
 * forwards, whose copies and routing run beside the neighbouring forwards' kernels.  Default:
 * the input upload waits for all work enqueued on the stream before the call, and y is in
 * y_host when the stream reaches the end of the forward, like any stream-ordered operation.
 * With this flag
 *  - the upload waits only until the previous forward of this plan no longer reads the plan's
 *    input buffer or its routing (its gather), so back-to-back host forwards upload the next
 *    input while the previous one is still computing; with a page-locked x_host the routing
 *    (router and top-k) follows the upload on a stream of the plan's own, beside the previous
 *    forward's last kernels, and the stream joins it before Dispatch.  The caller must have
 *    written x_host on the host, and W_router (router_logits when it is the input) on the
 *    device, before the call: a write by work enqueued on the stream between two such calls
 *    (a copy, a kernel, a host callback) is not waited for.  A forward's routing outputs
 *    (router_logits, and what moe_debug_routing reads) may be overwritten as soon as the next
 *    pipelined host forward of the plan has been called;
 *  - a page-locked y_host is filled by the copy engines on a stream of the plan's own, from one
 *    of two plan-owned staging buffers that Combine writes in turn, and `stream` does not wait
 *    for that copy: y_host is complete once moe_host_wait has made a stream wait for it (or
 *    moe_get_status has returned).  Each staging buffer is reused by the forward after next,
 *    whose kernels start once that copy is done; the plan's workspace holds the second buffer. */
#define MOE_FLAG_HOST_PIPELINE (1u << 7)
#define MOE_FLAG_TEST_BAD_ID (1u << 9)  /* test only: Dispatch sees the first (token, slot) pair's expert
                                          id out of range; the pair is dropped, no access leaves the
                                          workspace, and moe_get_status reports MOE_ERR_DEVICE_CHECK */
#define MOE_FLAG_TEST_STALL (1u << 8)   /* test only: Linear-2 tiles wait for a readiness count that
                                           is never reached, so the bounded wait expires and
                                           moe_get_status reports MOE_ERR_TIMEOUT (no GPU fault)   */

#define MOE_NUM_STAGES 5 /* router+top-k, dispatch sort+schedule, gather, grouped GEMMs, combine */

typedef struct {
  int32_t T_max;        /* largest token count a forward may use (>= 1)                         */
  int32_t H;            /* hidden size: multiple of 64 (else MOE_ERR_UNSUPPORTED)               */
  int32_t I;            /* intermediate size per expert: multiple of 64 (else UNSUPPORTED)      */
  int32_t E;            /* experts: 1 <= E <= 256                                               */
  int32_t top_k;        /* 1 <= top_k <= min(E, 8)                                              */
  int32_t schedule;     /* MOE_SCHED_*                                                          */
  int32_t wave_experts; /* experts per wave; 0 = smallest run whose Linear-1 tiles fill the SMs */
  int32_t lead_waves;   /* interleave lead D >= 1 (0 = default 1)                               */
  uint32_t flags;       /* MOE_FLAG_*                                                           */
  int64_t timeout_ns;   /* limit of any device-side wait; 0 = 1 s                               */
  const float* router_bias; /* optional HOST pointer to E fp32 values added to every logit,
                               copied at plan time; NULL = no bias                               */
} moe_config_t;

typedef struct moe_plan_s* moe_plan_t;

/* Validate cfg, allocate the workspace for T_max on `device`, copy the bias.
 * On success *out receives a plan to pass to the calls below.  Passage: the layer's shape
 * (hidden, intermediate, experts, top-k) is the expert layer of the X-Stage paper's
 * introduction, MegaMoE paragraph; the plan and its workspace have no counterpart there. */
MOE_API moe_status_t moe_plan(const moe_config_t* cfg, int device, moe_plan_t* out);

/* Bytes of device workspace moe_plan allocates for cfg (no allocation).  Library plumbing:
 * no counterpart in the paper. */
MOE_API moe_status_t moe_workspace_bytes(const moe_config_t* cfg, size_t* bytes);

/* One forward of the layer for T tokens (0 <= T <= T_max; T = 0 enqueues nothing), enqueued
 * [the operation: X-Stage paper, introduction, MegaMoE paragraph - router top-k, Dispatch,
 * Linear-1, SwiGLU, Linear-2, Combine weighted by the router weights]
 * on `stream` (a cudaStream_t; NULL = the legacy default stream).  Never synchronises.
 *   x             bf16 [T, H]            input tokens
 *   router_logits fp32 [T, E]            OUTPUT when W_router != NULL (see MOE_FLAG_EXACT_LOGITS
 *                                        for which entries are canonical), else INPUT
 *   W_router      bf16 [H, E] or NULL    router weight
 *   W1_gate_up    bf16 [E, H, 2I]        Linear-1; columns [0,I) gate, [I,2I) up
 *   W2            bf16 [E, I, H]         Linear-2
 *   y             bf16 [T, H]            output
 * Device pointers, 16-byte aligned. */
MOE_API moe_status_t moe_forward(moe_plan_t plan, int32_t T, const void* x, float* router_logits,
                         const void* W_router, const void* W1_gate_up, const void* W2, void* y,
                         void* stream);

/* moe_forward with the token tensors in HOST memory (the same operation as moe_forward; the
 * host transfer has no counterpart in the paper): x_host (bf16 [T, H]) is brought into a
 * plan-owned device buffer, the layer runs, and y (bf16 [T, H]) lands in y_host, all enqueued
 * on `stream`.  A page-locked buffer that is mapped into the device's address space (any
 * cudaHostAlloc / cudaMallocHost buffer under unified addressing) at a 16-byte-aligned address
 * is copied into the plan's buffer by the copy engines in token ranges, each routed as it
 * lands, and Combine stores y into y_host in place (with MOE_FLAG_HOST_PIPELINE the copies
 * run beside the neighbouring forwards instead: see there).
 * Any other buffer goes through cudaMemcpyAsync and plan-owned staging buffers (synchronous for
 * pageable memory).  router_logits, W_router, W1_gate_up and W2 are
 * DEVICE pointers exactly as in moe_forward.  The caller must not touch y_host before the
 * stream reaches this point (e.g. cudaStreamSynchronize), and must not write x_host before then. */
MOE_API moe_status_t moe_forward_host(moe_plan_t plan, int32_t T, const void* x_host, float* router_logits,
                              const void* W_router, const void* W1_gate_up, const void* W2, void* y_host,
                              void* stream);

/* Make `stream` wait (without blocking the host) until every output copy of the plan's pipelined
 * host forwards (MOE_FLAG_HOST_PIPELINE) enqueued so far has landed in its y_host; a no-op
 * wait when there is none (library plumbing: no counterpart in the paper).
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (null plan) or MOE_ERR_CUDA. */
MOE_API moe_status_t moe_host_wait(moe_plan_t plan, void* stream);

/* Synchronise `stream` and the plan's pending output copies (MOE_FLAG_HOST_PIPELINE), then read
 * and clear the plan's device error word (library plumbing: no counterpart in the paper).
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK or MOE_ERR_CUDA. */
MOE_API moe_status_t moe_get_status(moe_plan_t plan, void* stream);

/* Copy the routing of the last forward (T tokens) into caller DEVICE buffers, stream-ordered
 * [the router's top-k and Dispatch's expert-contiguous row order: X-Stage paper, introduction,
 * MegaMoE paragraph]
 * (any pointer may be NULL to skip it):
 *   ids int32 [T,k], w fp32 [T,k], counts int32 [E], offsets int32 [E+1],
 *   row_pair int32 [T*k] (row -> t*k+j, rows grouped by expert, ascending t within an expert),
 *   row_of int32 [T*k] ((t,j) -> row). */
MOE_API moe_status_t moe_debug_routing(moe_plan_t plan, int32_t T, int32_t* ids, float* w, int32_t* counts,
                               int32_t* offsets, int32_t* row_pair, int32_t* row_of, void* stream);

/* Copy the intermediates of the last forward into caller DEVICE buffers (NULL skips)
 * [Linear-1 + SwiGLU output and the router-weighted Linear-2 output: X-Stage paper,
 * introduction, MegaMoE paragraph]:
 *   h   bf16 [T*k, I]   activation rows in dispatch (row) order
 *   P   fp32 [T*k, H]   router-weighted expert outputs, indexed by t*k+j */
MOE_API moe_status_t moe_debug_intermediates(moe_plan_t plan, int32_t T, void* h, float* P, void* stream);

/* Durations (ms) of the MOE_NUM_STAGES stages of the last forward (the steps of the X-Stage
 * paper's MegaMoE paragraph, timed); needs MOE_FLAG_STAGE_TIMING.
 * Synchronises on the recorded events.  ms[3] is the grouped-GEMM launch(es). */
MOE_API moe_status_t moe_stage_times(moe_plan_t plan, float* ms);

/* Wait-time trace of the last forward's grouped GEMM (the producer / tensor-core / epilogue
 * roles coupled through finite staging that the X-Stage paper's MegaMoE discussion describes;
 * needs MOE_FLAG_TRACE; synchronises the
 * device).  Writes n = (CTAs + 1) x 8 uint64 values to host_buf (CTAs: the larger of the two
 * launch paths' grids; a CTA the last launch did not have reads zero; the last row holds the
 * %globaltimer stamps of a MOE_FLAG_SINGLE_LAUNCH forward - start, end of router logits, top-k,
 * Dispatch, gather, grouped GEMM, Combine - and zeros otherwise) (cap = capacity in values); per CTA:
 * {producer waiting for a free stage, producer waiting for Linear-1 readiness, MMA issuer waiting
 * for a free accumulator, MMA issuer waiting for operands, epilogue waiting for an accumulator,
 * CTA lifetime} in nanoseconds, then {Linear-1 tiles, Linear-2 tiles}. */
MOE_API moe_status_t moe_trace_read(moe_plan_t plan, uint64_t* host_buf, size_t cap, size_t* n);

/* Per-tile trace of the last forward's grouped GEMM (the per-tile timing that the X-Stage
 * paper's experimental setup takes with in-kernel timer instrumentation, and the SM-id probe of
 * the TIDE paper's section 2.2, SM wave quantization: CTAs recording their SM id with entry and
 * exit timestamps); needs MOE_FLAG_TRACE; synchronises the device.  Writes n = tiles x 2 x 4
 * uint64 values to host_buf (cap = capacity in values; host_buf NULL: n only), tiles = the
 * length of the tile list moe_debug_schedule returns, in that order; for tile i and CTA rank r
 * of the 2-CTA cluster that ran it, values (2 i + r) * 4 .. + 3: {SM id, %globaltimer (ns)
 * when the CTA's TMA producer started the tile, when its accumulator was complete in TMEM,
 * when its epilogue finished (Linear-1: h rows written, before the unit's readiness count is
 * raised; Linear-2: the last P stores issued)}.  A tile a timed-out forward never reached reads
 * zeros.  MOE_ERR_INVALID_ARG without MOE_FLAG_TRACE or if cap < n. */
MOE_API moe_status_t moe_trace_tiles(moe_plan_t plan, uint64_t* host_buf, size_t cap, size_t* n);

/* The coefficient cH of the default router's error bound (the router used without
 * MOE_FLAG_EXACT_LOGITS; library numerics, no counterpart in the paper) for a forward
 * of T tokens (1 <= T <= T_max): n = the MMA steps of the longest accumulation chain, A the
 * chains per CTA, S the K splits; cH = (n + 1) 2^-17 + (A S + H/32 + 8) 2^-22.  Host only. */
MOE_API moe_status_t moe_router_bound(moe_plan_t plan, int32_t T, float* cH);

/* Number of kernels the last moe_forward launched (library plumbing). */
MOE_API moe_status_t moe_last_launch_count(moe_plan_t plan, int32_t* n);

/* Free the plan and its workspace (synchronises the device first; library plumbing). */
MOE_API moe_status_t moe_plan_destroy(moe_plan_t plan);

/* Static description of a status code (library plumbing). */
MOE_API const char* moe_status_string(moe_status_t s);

/* Dispatch (the stable counting sort of moe_forward's Dispatch step) for callers that cannot
 * allocate device memory.  The paper has no counterpart: it exists for code that may not call
 * cudaMalloc, e.g. under an allocator that owns all device memory or a fixed memory budget (a
 * cudaMalloc behind its back fails or breaks its accounting), or on paths that must not risk
 * the implicit synchronisation of cudaMalloc/cudaFree.  It allocates nothing: its scratch (one
 * row counter per expert) is a fixed array of 256 counters inside the library, present on every
 * device that loads it until the process exits.
 *   ids      int32 [T,k]  expert of each (token, slot)
 *   w        fp32  [T,k]  router weights, or NULL (then row_w must be NULL)
 *   offsets  int32 [E+1]  OUTPUT: rows of expert e are offsets[e] .. offsets[e+1]-1
 *   row_pair int32 [T*k]  OUTPUT: row -> t*k+j, ascending t within an expert
 *   row_of   int32 [T*k]  OUTPUT: t*k+j -> row
 *   row_w    fp32  [T*k]  OUTPUT: w of each row, or NULL
 * Device pointers (ids needs only 4-byte alignment), enqueued on `stream` (a cudaStream_t;
 * NULL = legacy default stream).  T = 0 writes offsets = 0 and nothing else.
 * A pair whose id lies outside [0, E) gets no row: row_of[t*k+j] = -1, and offsets[E] counts
 * only the placed pairs, so offsets[E] < T*k tells the caller that some id was out of range
 * (rows offsets[E] .. T*k-1 of row_pair and row_w are then not written).
 * Limits: E <= 256 and T*k < 2^30, else MOE_ERR_UNSUPPORTED.  The first call on a device (and
 * the first after its context was replaced, e.g. by cudaDeviceReset) looks up the array's
 * device address (cudaGetSymbolAddress) and should happen before any stream capture; later
 * calls only enqueue a memset of the counters and two kernels.  All calls share the one
 * array: calls whose work overlaps on the GPU (different streams without ordering) race and
 * give wrong rows; calls ordered on one stream are safe, each clears the counters first. */
MOE_API moe_status_t moe_dispatch_static(int32_t T, int32_t E, int32_t k, const int32_t* ids, const float* w,
                                 int32_t* offsets, int32_t* row_pair, int32_t* row_of, float* row_w,
                                 void* stream);

/* The tile list the last forward's Dispatch built on the device [the expert-wave schedule and
 * the cross-wave interleave: X-Stage paper, introduction (expert waves) and its X-Stage-aware
 * design section] (synchronises `stream`):
 * n_out[3] = {linear-1 tiles, total tiles, tile workers (2-CTA clusters) it was built for};
 * up to cap tiles are copied to HOST memory tiles_out (4 ints each, as moe_schedule_host), which
 * may be NULL to query the counts.  MOE_ERR_INVALID_ARG if cap is smaller than the total. */
MOE_API moe_status_t moe_debug_schedule(moe_plan_t plan, int32_t* tiles_out, int64_t cap, int64_t* n_out,
                                void* stream);

/* Host-side evaluation of the tile schedule the device builds (the same passages as
 * moe_debug_schedule; for tests; no GPU needed).
 * counts[E] rows per expert; num_sms = number of tile workers (2-CTA clusters on the GPU);
 * a unit is a pair of 128-row m-tiles of one expert.  Writes up to cap tiles as 4 ints each
 * {phase | n_block << 1, expert, unit within the expert, global unit index} into tiles_out and
 * the tile counts {linear-1 tiles, total tiles} into n_out[2].  A unit has ceil(I / 128)
 * Linear-1 tiles and ceil(H / 256) Linear-2 tiles (the last of each may be partial); H and I
 * must be positive multiples of 64, else MOE_ERR_INVALID_ARG. */
MOE_API moe_status_t moe_schedule_host(const int32_t* counts, int32_t E, int32_t H, int32_t I,
                               int32_t num_sms, int32_t schedule, int32_t wave_experts,
                               int32_t lead_waves, int32_t* tiles_out, int64_t cap, int64_t* n_out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
