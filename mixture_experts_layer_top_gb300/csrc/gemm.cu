// Persistent grouped GEMM for both expert projections of the MoE layer.
//
// Linear-1 tile (phase 0): 256 dispatch rows of one expert (two 128-row m-tiles)
//   of x_perm times W1[e][:, 128 n .. +128] (gate) and W1[e][:, I + 128 n .. +128]
//   (up): one M=256 x N=256 tcgen05 accumulator; epilogue h = bf16(silu(g) * u).
// Linear-2 tile (phase 1): the same rows of h times W2[e][:, 256 n .. +256];
//   epilogue P = w[t,j] * acc, the router-weight scale, stored as fp16 times an
//   exact power-of-two scale per (row, 128-column block): the scale puts the
//   block's largest finite |P| in [2^14, 2^15], so nothing overflows and every
//   value keeps fp16's 11 significant bits.
// (X-Stage paper, MegaMoE background: Linear-1 projects hidden to
// intermediate, SwiGLU is applied, Linear-2 projects back; the kernel design -
// persistent, warp-specialised, TMA producer, tensor-core issuer, epilogue
// roles coupled through finite accumulator staging - follows the fused-kernel
// description there, rebuilt here for tcgen05/TMEM on sm_103a.)
//
// Pairs of SMs: each tile runs on a 2-CTA cluster with the pair form of the MMA
// (cta_group::2, M = 256).  CTA rank r owns m-tile 2*unit + r: it loads those
// 128 rows of A and one half of B (Linear-1: r = 0 the gate columns, r = 1 the up
// columns; Linear-2: columns [128 r, 128 r + 128)) into its own shared memory,
// and its TMEM receives its 128 rows x 256 columns of the accumulator.  Per CTA a
// pipeline stage is 32 KB (16 KB A + 16 KB half of B), NST stages; both
// CTAs' loads complete on the even CTA's "stage full" barrier, whose single
// thread issues the MMAs for the pair and multicasts completion to both CTAs'
// "stage empty" and "accumulator full" barriers.  Each CTA's epilogue signals
// the even CTA's "accumulator empty" barrier.
//
// Roles (320 threads):  warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer
// (one thread, even CTA only), warps 2..9 = epilogue: warp w reads TMEM lanes
// 32*(w%4) .. +31 (tile rows) and one half of the tile's columns.  Tiles come
// from a ticket list built by the dispatch kernel; cluster c takes tickets c,
// c+clusters, ... in order.  A Linear-2 tile first waits until the ready counter
// of its unit shows all Linear-1 tiles of those rows stored by both CTAs;
// tickets are in a topological order and every cluster is resident (the grid is
// at most the number of co-resident clusters, 1 CTA/SM), so the waits finish.
// Every wait is bounded by timeout_ns; on expiry the CTA records ERR_TIMEOUT,
// waits (bounded) for its in-flight copies and MMAs, frees TMEM and exits.
//
// Rows live in a padded row space (unit g owns rows 256 g .. 256 g + 255), so a
// CTA's 128 rows are contiguous: A tiles are tiled TMA loads, and outputs go out
// per 32-row quadrant (one epilogue warp pair): a quadrant whose rows are all
// valid is staged in shared memory in the 128-byte swizzled layout
// (conflict-free row writes) and written by a bulk tensor store (h: bf16 32 x 64
// boxes for Linear-1; P: fp16 32 x 64 boxes in two passes for Linear-2); the valid rows of a partial quadrant are stored directly; empty
// quadrants write nothing.  NBUF 32 KB staging buffers rotate, each reused
// only after its previous store group has read it.  Linear-1 readiness is
// published after its h rows are written.
//
// Two shared-memory splits are compiled: <6 stages, 1 staging buffer> (the
// default: the deeper ring keeps more operand bytes in flight, which measured
// faster both when the GEMMs stream weights and when they are tensor-bound) and
// <5 stages, 2 staging buffers> (a store drains while the next chunk is
// written).  Both compute bit-identical results.
//
// Shared-memory operand layouts (128-byte swizzle, as written by TMA):
//   A (K-major): 128 rows x 128 B per stage; descriptor SBO = 1024 B (8-row
//     group), K step of 16 elements = +32 B on the start address.
//   B half (N-major): two 64-column boxes of 64 K-rows x 128 B (8 KB each);
//     descriptor LBO = 8 KB (next 64 columns), SBO = 1024 B (next 8 K-rows),
//     K step of 16 rows = +2048 B.
#include "gemm_body.cuh"

namespace moe {

namespace {

using namespace gemm_detail;

template <int NST, int NBUF>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmP,
                    const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  grouped_gemm_body<NST, NBUF>(&tmA1, &tmB1, &tmA2, &tmB2, &tmH, &tmP, args, smem_raw);
}

}  // namespace

using GemmStreaming = Layout<6, 1>;
using GemmCompute = Layout<5, 2>;
static_assert(GemmStreaming::SMEM == GemmCompute::SMEM, "both splits share one occupancy computation");

static cudaLaunchConfig_t gemm_config(int grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GemmCompute::SMEM;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t gemm_prepare(int device, int* grid) {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<6, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GemmStreaming::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<5, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemmCompute::SMEM);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return e;
  // every cluster of the grid must be resident at once (Linear-2 tiles wait for earlier tickets)
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = gemm_config(sms / PAIR * PAIR, nullptr, attr);
  int clusters = 0, clusters_s = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<5, 2>, &cfg);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveClusters(&clusters_s, grouped_gemm_kernel<6, 1>, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters_s < clusters) clusters = clusters_s;
  if (clusters > sms / PAIR) clusters = sms / PAIR;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  *grid = clusters * PAIR;
  return cudaSuccess;
}

cudaError_t launch_grouped_gemm(const CUtensorMap& tA1, const CUtensorMap& tB1, const CUtensorMap& tA2,
                                const CUtensorMap& tB2, const CUtensorMap& tH, const CUtensorMap& tP,
                                const GemmArgs& a, int grid, bool streaming, cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = gemm_config(grid, st, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap launch and setup with the previous kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  if (streaming) return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<6, 1>, tA1, tB1, tA2, tB2, tH, tP, a);
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<5, 2>, tA1, tB1, tA2, tB2, tH, tP, a);
}

}  // namespace moe
