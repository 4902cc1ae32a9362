// Combine on one GPU: y[t,:] = bf16( sum_{j=0..k-1} P[row(t,j), :] ), the fp32
// sum taken in slot order j = 0, 1, ..., k-1 so the result does not depend on
// which expert finished first.  P already holds w[t,j] * (expert output), so
// this is the X-Stage paper's MegaMoE-background Combine ("aggregates the
// top-k results using the router weights") with the weights applied upstream.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace moe {

namespace {

// One thread per 4 consecutive outputs: k float4 loads from the slots' rows of P
// (padded row space, found through prow_of), fixed-order fp32 sum, 8-byte store.
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ P_pad, const int32_t* __restrict__ prow_of, int T, int H, int k,
               uint16_t* __restrict__ y) {
  const int64_t n4 = (int64_t)T * H / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = (i * 4) / H;
    const int64_t c = (i * 4) % H;
    const int32_t* pr = prow_of + t * k;
    float4 s = __ldcs(reinterpret_cast<const float4*>(P_pad + (int64_t)pr[0] * H + c));
    for (int j = 1; j < k; ++j) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(P_pad + (int64_t)pr[j] * H + c));
      s.x = s.x + v.x;
      s.y = s.y + v.y;
      s.z = s.z + v.z;
      s.w = s.w + v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(s.z, s.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + t * H + c) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const float* P_pad, const int32_t* prow_of, int T, int H, int k, uint16_t* y, int sms,
                           cudaStream_t st) {
  const int64_t n4 = (int64_t)T * H / 4;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  combine_kernel<<<(int)blocks, 256, 0, st>>>(P_pad, prow_of, T, H, k, y);
  return cudaGetLastError();
}

}  // namespace moe
