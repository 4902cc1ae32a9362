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
#include "layer_parts.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int DS_THREADS = 512;

// Dispatch as its own launch: grid DS_SCHED_CTAS + ceil(T / DS_CHUNK_TOK), one virtual block per CTA.
__global__ void __launch_bounds__(DS_THREADS)
dispatch_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, const int32_t* __restrict__ counts,
                const int32_t* __restrict__ chist, int T, int E, int k, int nL1, int nL2, int workers, int mode,
                int wave_experts, int lead, int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair,
                int32_t* __restrict__ row_of, int32_t* __restrict__ prow_of, float* __restrict__ prow_w,
                int32_t* __restrict__ tiles, int32_t* __restrict__ sched, int32_t* __restrict__ ready,
                uint32_t* __restrict__ err, int dead_row, int test_bad_id) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  __shared__ DispatchSmem sm;
  dispatch_body<DS_THREADS>(blockIdx.x, sm, ids, w, counts, chist, T, E, k, nL1, nL2, workers, mode, wave_experts,
                            lead, offsets, row_pair, row_of, prow_of, prow_w, tiles, sched, ready, err, dead_row,
                            test_bad_id);
}

__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ prow_of, int T, int H, int k,
                   uint16_t* __restrict__ x_pad) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int task = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (task >= T * gather_chunks(H)) return;
  gather_task(x, prow_of, H, k, x_pad, task, threadIdx.x & 31);
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
      P[(size_t)f * H + c] = __half2float(__ushort_as_half(P_pad[pr * H + c])) * S_pad[pr * p_scale_blocks(H) + c / P_SCALE_COLS];
}

}  // namespace

cudaError_t launch_dispatch(const Workspace& ws, int T, int E, int k, int H, int I, int num_sms, int mode,
                            int wave_experts, int lead, int dead_row, bool test_bad_id, cudaStream_t st) {
  const int chunks = (T + DS_CHUNK_TOK - 1) / DS_CHUNK_TOK;
  return launch_pdl(dispatch_kernel, dim3(DS_SCHED_CTAS + chunks), dim3(DS_THREADS), 0, st, ws.ids, ws.w, ws.counts,
                    ws.chist, T, E, k, l1_blocks(I), l2_blocks(H), num_sms, mode, wave_experts, lead, ws.offsets,
                    ws.row_pair, ws.row_of, ws.prow_of, ws.prow_w, ws.tiles, ws.sched, ws.ready, ws.err, dead_row,
                    test_bad_id ? 1 : 0);
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* prow_of, int T, int H, int k, uint16_t* x_pad,
                          cudaStream_t st) {
  const int nch = gather_chunks(H);
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
