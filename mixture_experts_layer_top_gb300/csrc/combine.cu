// Combine on one GPU: y[t,:] = bf16( sum_{j=0..k-1} P[row(t,j), :] ), the fp32
// sum taken in slot order j = 0, 1, ..., k-1 so the result does not depend on
// which expert finished first.  P is stored as fp16 with a power-of-two scale per
// (row, 128 columns); each term is widened and rescaled exactly before the sum.
// P already holds w[t,j] * (expert output): this is the Combine of the X-Stage
// paper's MegaMoE paragraph (introduction) - the router-weighted sum of a
// token's top-k expert outputs - with the weights applied upstream.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "layer_parts.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// One thread per 8 consecutive outputs (combine_item), grid-stride.
template <bool ALL_IN_FLIGHT>
__global__ void __launch_bounds__(256)
combine_kernel(const uint16_t* __restrict__ P_pad, const float* __restrict__ S_pad, const int32_t* __restrict__ prow_of,
               int T, int H, int k, uint16_t* __restrict__ y) {
  ptx::grid_dep_wait();   // the previous kernel's results are visible from here on
  const int64_t n8 = (int64_t)T * H / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x)
    combine_item<ALL_IN_FLIGHT>(P_pad, S_pad, prow_of, H, k, y, i);
}

}  // namespace

cudaError_t launch_combine(const uint16_t* P_pad, const float* S_pad, const int32_t* prow_of, int T, int H, int k,
                           uint16_t* y, int sms, cudaStream_t st) {
  const int64_t n8 = (int64_t)T * H / 8;
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // a batch that one resident wave of threads covers (4 blocks of 256 per SM) is latency-bound:
  // all slots in flight; larger batches are bandwidth-bound: one slot at a time
  if (n8 <= (int64_t)sms * 4 * 256)
    return launch_pdl(combine_kernel<true>, dim3((unsigned)blocks), dim3(256), 0, st, P_pad, S_pad, prow_of, T, H, k, y);
  return launch_pdl(combine_kernel<false>, dim3((unsigned)blocks), dim3(256), 0, st, P_pad, S_pad, prow_of, T, H, k, y);
}

}  // namespace moe
