// Dispatch without any device allocation: moe_dispatch_static().
//
// The same stable counting sort as the Dispatch step of moe_forward (rows of
// expert e in ascending token order), but its scratch - one row counter per
// expert - lives in a fixed array in this file instead of a plan's workspace,
// so callers that may not call cudaMalloc can still use it.  Those are, for
// example, runtimes whose device memory is entirely owned by another allocator
// or capped at a fixed budget (a cudaMalloc behind its back would fail or break
// its accounting), and code paths that must not risk the implicit device
// synchronisation cudaMalloc and cudaFree can cause.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.cuh"

namespace moe {
namespace {

// Largest expert count the fixed scratch serves; larger E is rejected.
constexpr int STATIC_MAX_EXPERTS = 256;
// Per-expert row counters of the most recent call on this device.  Every GPU
// that loads the library holds this array until the process exits.
static __device__ __align__(256) int32_t g_static_counts[STATIC_MAX_EXPERTS];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mu;
// Per device: the array's address and the id of the context it was looked up in.  A context
// id is unique for the life of the process, so after cudaDeviceReset (a new primary context,
// the module loaded again, possibly elsewhere) the address is looked up anew.
int32_t* g_counts_ptr[MAX_DEVICES] = {};
unsigned long long g_counts_ctx[MAX_DEVICES] = {};

typedef CUresult (*PFN_ctx_get_current)(CUcontext*);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long*);
PFN_ctx_get_current g_ctx_get_current = nullptr;
PFN_ctx_get_id g_ctx_get_id = nullptr;

// Id of the context current on this thread (0 if there is none yet or the lookup fails).
unsigned long long current_context_id() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_ctx_get_current>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PFN_ctx_get_id>(f);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_get_current || !g_ctx_get_id || g_ctx_get_current(&c) != CUDA_SUCCESS || !c ||
      g_ctx_get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_static_counts on the current device: looked up once per device and
// context (host code must not pass the symbol itself to a kernel: that is a host-side
// stand-in, not a device address).
cudaError_t static_counts_address(int dev, int32_t** out) {
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_counts_ptr[dev] || ctx == 0 || ctx != g_counts_ctx[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_counts);   // binds the primary context if needed
    if (e != cudaSuccess) return e;
    g_counts_ptr[dev] = static_cast<int32_t*>(p);
    g_counts_ctx[dev] = current_context_id();
  }
  *out = g_counts_ptr[dev];
  return cudaSuccess;
}

constexpr int SS_THREADS = 1024;
constexpr int SS_PER_THREAD = 16;

// counts[e] += #{f : ids[f] == e}; a block histogram in shared memory, then one
// global atomic per non-empty bin.  Entries outside [0, E) are not counted; their
// row_of is set to -1 here (no row holds them).
__global__ void __launch_bounds__(256)
static_histogram_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
                        int32_t* __restrict__ row_of) {
  __shared__ int32_t bins[STATIC_MAX_EXPERTS];
  for (int i = threadIdx.x; i < E; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < R; f += gridDim.x * blockDim.x) {
    const int e = ids[f];
    if (e >= 0 && e < E) atomicAdd(&bins[e], 1);
    else row_of[f] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (bins[i]) atomicAdd(&counts[i], bins[i]);
}

__device__ __forceinline__ int static_block_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int s = sh[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, si, off);
      if (lane >= off) si += o;
    }
    sh[lane] = si - s;
    if (lane == 31) sh[32] = si;
  }
  __syncthreads();
  const int res = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return res;
}

// CTA e places expert e's pairs f = t*k + j in ascending f at rows
// offsets[e] .. offsets[e] + counts[e] - 1 and writes offsets[e] (the last CTA
// also offsets[E]).
__global__ void __launch_bounds__(SS_THREADS)
static_sort_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, const int32_t* __restrict__ counts,
                   int R, int E, int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair,
                   int32_t* __restrict__ row_of, float* __restrict__ row_w) {
  __shared__ int sh[33];
  __shared__ int s_base;
  const int e = blockIdx.x;
  if (threadIdx.x < 32) {
    int s = 0;
    for (int i = threadIdx.x; i < e; i += 32) s += counts[i];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    if (threadIdx.x == 0) {
      s_base = s;
      offsets[e] = s;
      if (e == E - 1) offsets[E] = s + counts[e];
    }
  }
  __syncthreads();
  if (counts[e] == 0) return;
  int running = s_base;
  const bool vec_ok = (R % 4) == 0 && (reinterpret_cast<uintptr_t>(ids) & 15u) == 0;
  for (int base = 0; base < R; base += SS_THREADS * SS_PER_THREAD) {
    const int f0 = base + threadIdx.x * SS_PER_THREAD;
    int v[SS_PER_THREAD];
    if (vec_ok && f0 + SS_PER_THREAD <= R) {
#pragma unroll
      for (int q = 0; q < SS_PER_THREAD / 4; ++q) {
        const int4 p = *reinterpret_cast<const int4*>(ids + f0 + 4 * q);
        v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < SS_PER_THREAD; ++q) v[q] = (f0 + q < R) ? ids[f0 + q] : -1;
    }
    int c = 0;
#pragma unroll
    for (int q = 0; q < SS_PER_THREAD; ++q) c += (v[q] == e);
    int total;
    int pos = running + static_block_scan(c, sh, &total);
#pragma unroll
    for (int q = 0; q < SS_PER_THREAD; ++q) {
      if (v[q] == e) {
        const int f = f0 + q;
        row_pair[pos] = f;
        row_of[f] = pos;
        if (row_w) row_w[pos] = w[f];
        ++pos;
      }
    }
    running += total;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_static(int32_t T, int32_t E, int32_t k, const int32_t* ids, const float* w,
                                            int32_t* offsets, int32_t* row_pair, int32_t* row_of, float* row_w,
                                            void* stream) {
  if (T < 0 || E < 1 || k < 1 || k > MAX_K || k > E || !offsets) return MOE_ERR_INVALID_ARG;
  if ((w == nullptr) != (row_w == nullptr)) return MOE_ERR_INVALID_ARG;
  if (E > STATIC_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
  const int64_t R64 = (int64_t)T * k;
  if (R64 >= (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!ids || !row_pair || !row_of)) return MOE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* counts = nullptr;
  if (static_counts_address(dev, &counts) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int R = (int)R64;
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (R == 0) {
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  int blocks = (R + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  static_histogram_kernel<<<blocks, 256, 0, st>>>(ids, R, E, counts, row_of);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  static_sort_kernel<<<E, SS_THREADS, 0, st>>>(ids, w, counts, R, E, offsets, row_pair, row_of, row_w);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
