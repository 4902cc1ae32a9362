/* A plain C99 caller of the library on the GPU, compiled and run by tests/test_c_abi.py: it
 * reads the tiny workload and the oracle's expectations from DIR (written by
 * tests/golden/make_c_abi_case.py), allocates every buffer with cudaMalloc, and calls
 * moe_plan, moe_forward, moe_get_status, moe_debug_routing and moe_plan_destroy as a C user
 * would.  Checks: the routing ids bit for bit, y within the stated bounds of the oracle's
 * result (absolute 2e-2 RMS everywhere, relative 3e-2 where |y_ref| > 0.1 RMS, measured from
 * the oracle's interval of y before rounding, the GPU's value standing for anything within
 * half a bf16 spacing of it), then a second forward on the same plan bitwise equal to the
 * first, then two back-to-back pipelined host forwards (MOE_FLAG_HOST_PIPELINE,
 * cudaMallocHost buffers, moe_forward_host + moe_host_wait) bitwise equal to it too.
 * Prints "ok ..." and exits 0 on success; prints the failed check otherwise. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_gb300.h"

#define CHECK(cond)                                        \
  do {                                                     \
    if (!(cond)) {                                         \
      printf("failed: %s (line %d)\n", #cond, __LINE__);   \
      return 1;                                            \
    }                                                      \
  } while (0)

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* p = malloc(bytes);
  size_t got = p ? fread(p, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* distance from a bf16 value to the spacing of bf16 numbers at it, halved */
static double half_spacing(double v) {
  if (v == 0.0) return ldexp(1.0, -134);
  int e;
  frexp(fabs(v), &e);
  return ldexp(0.5, e - 8 < -133 ? -133 : e - 8);
}

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  CHECK(argc == 2);
  const char* dir = argv[1];
  int T, H, I, E, k;
  {
    char path[4096];
    snprintf(path, sizeof(path), "%s/shape.txt", dir);
    FILE* f = fopen(path, "r");
    CHECK(f != NULL);
    CHECK(fscanf(f, "%d %d %d %d %d", &T, &H, &I, &E, &k) == 5);
    fclose(f);
  }
  const size_t nx = (size_t)T * H, nwr = (size_t)H * E, nw1 = (size_t)E * H * 2 * I, nw2 = (size_t)E * I * H;
  uint16_t* x = read_file(dir, "x.bin", nx * 2);
  uint16_t* Wr = read_file(dir, "Wr.bin", nwr * 2);
  uint16_t* W1 = read_file(dir, "W1.bin", nw1 * 2);
  uint16_t* W2 = read_file(dir, "W2.bin", nw2 * 2);
  int32_t* ids_ref = read_file(dir, "ids.bin", (size_t)T * k * 4);
  uint16_t* y_ref = read_file(dir, "y.bin", nx * 2);
  double* ylo = read_file(dir, "ylo.bin", nx * 8);
  double* yhi = read_file(dir, "yhi.bin", nx * 8);
  CHECK(x && Wr && W1 && W2 && ids_ref && y_ref && ylo && yhi);

  CHECK(cudaSetDevice(0) == cudaSuccess);
  cudaStream_t st;
  CHECK(cudaStreamCreate(&st) == cudaSuccess);
  void* dx = dev_copy(x, nx * 2);
  void* dWr = dev_copy(Wr, nwr * 2);
  void* dW1 = dev_copy(W1, nw1 * 2);
  void* dW2 = dev_copy(W2, nw2 * 2);
  void* dlogits = dev_copy(NULL, (size_t)T * E * 4);
  void* dy = dev_copy(NULL, nx * 2);
  void* dids = dev_copy(NULL, (size_t)T * k * 4);
  CHECK(dx && dWr && dW1 && dW2 && dlogits && dy && dids);

  moe_config_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.T_max = T;
  cfg.H = H;
  cfg.I = I;
  cfg.E = E;
  cfg.top_k = k;
  cfg.schedule = MOE_SCHED_AUTO;
  moe_plan_t plan = NULL;
  CHECK(moe_plan(&cfg, 0, &plan) == MOE_OK && plan != NULL);
  CHECK(moe_forward(plan, T, dx, (float*)dlogits, dWr, dW1, dW2, dy, (void*)st) == MOE_OK);
  CHECK(moe_get_status(plan, (void*)st) == MOE_OK);
  CHECK(moe_debug_routing(plan, T, (int32_t*)dids, NULL, NULL, NULL, NULL, NULL, (void*)st) == MOE_OK);
  uint16_t* y = malloc(nx * 2);
  uint16_t* y2 = malloc(nx * 2);
  int32_t* ids = malloc((size_t)T * k * 4);
  CHECK(y && y2 && ids);
  CHECK(cudaMemcpyAsync(y, dy, nx * 2, cudaMemcpyDeviceToHost, st) == cudaSuccess);
  CHECK(cudaMemcpyAsync(ids, dids, (size_t)T * k * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess);
  CHECK(cudaStreamSynchronize(st) == cudaSuccess);

  CHECK(memcmp(ids, ids_ref, (size_t)T * k * 4) == 0);
  double ss = 0.0;
  for (size_t i = 0; i < nx; ++i) ss += bf16_value(y_ref[i]) * bf16_value(y_ref[i]);
  const double rms = sqrt(ss / (double)nx);
  double worst_abs = 0.0, worst_rel = 0.0;
  for (size_t i = 0; i < nx; ++i) {
    const double g = bf16_value(y[i]), r = bf16_value(y_ref[i]);
    CHECK(isfinite(g));
    const double dist = (ylo[i] > g ? ylo[i] - g : 0.0) + (g > yhi[i] ? g - yhi[i] : 0.0);
    const double d = dist > half_spacing(g) ? dist - half_spacing(g) : 0.0;
    if (d > worst_abs) worst_abs = d;
    if (fabs(r) > 0.1 * rms && d / fabs(r) > worst_rel) worst_rel = d / fabs(r);
  }
  CHECK(worst_abs <= 2e-2 * rms);
  CHECK(worst_rel <= 3e-2);

  CHECK(moe_forward(plan, T, dx, (float*)dlogits, dWr, dW1, dW2, dy, (void*)st) == MOE_OK);
  CHECK(cudaMemcpyAsync(y2, dy, nx * 2, cudaMemcpyDeviceToHost, st) == cudaSuccess);
  CHECK(moe_get_status(plan, (void*)st) == MOE_OK);
  CHECK(memcmp(y, y2, nx * 2) == 0);
  CHECK(moe_plan_destroy(plan) == MOE_OK);

  /* pipelined host forwards: page-locked x in, two outputs, the copies waited for by moe_host_wait */
  cfg.flags = MOE_FLAG_HOST_PIPELINE;
  moe_plan_t hplan = NULL;
  CHECK(moe_plan(&cfg, 0, &hplan) == MOE_OK && hplan != NULL);
  void *hx = NULL, *hy0 = NULL, *hy1 = NULL;
  CHECK(cudaMallocHost(&hx, nx * 2) == cudaSuccess && cudaMallocHost(&hy0, nx * 2) == cudaSuccess &&
        cudaMallocHost(&hy1, nx * 2) == cudaSuccess);
  memcpy(hx, x, nx * 2);
  memset(hy0, 0xFF, nx * 2);
  memset(hy1, 0xFF, nx * 2);
  CHECK(moe_forward_host(hplan, T, hx, (float*)dlogits, dWr, dW1, dW2, hy0, (void*)st) == MOE_OK);
  CHECK(moe_forward_host(hplan, T, hx, (float*)dlogits, dWr, dW1, dW2, hy1, (void*)st) == MOE_OK);
  CHECK(moe_host_wait(hplan, (void*)st) == MOE_OK);
  CHECK(cudaStreamSynchronize(st) == cudaSuccess);
  CHECK(memcmp(y, hy0, nx * 2) == 0);
  CHECK(memcmp(y, hy1, nx * 2) == 0);
  CHECK(moe_get_status(hplan, (void*)st) == MOE_OK);
  CHECK(moe_plan_destroy(hplan) == MOE_OK);
  cudaFreeHost(hx);
  cudaFreeHost(hy0);
  cudaFreeHost(hy1);
  cudaFree(dx);
  cudaFree(dWr);
  cudaFree(dW1);
  cudaFree(dW2);
  cudaFree(dlogits);
  cudaFree(dy);
  cudaFree(dids);
  cudaStreamDestroy(st);
  printf("ok max_abs/rms %.3e max_rel %.3e\n", worst_abs / rms, worst_rel);
  return 0;
}
