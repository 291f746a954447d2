// Integer-pipe throughput microbenchmark (sm_103a): whole-GPU op/s of the
// instructions a Gotoh cell is built from.  Each thread runs CH independent
// dependency chains so that issue, not latency, limits the rate.  Chains mix
// in the loop counter so the compiler cannot fold them.
#include <cuda_runtime.h>

#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int CH = 8;
constexpr int ITERS = 4096;

__global__ void k_viaddmax(int* out, int b) {
  int a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x + k;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) a[k] = __viaddmax_s32(a[k], b, i);
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_vimax3(int* out, int b) {
  int a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x + k;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) a[k] = __vimax3_s32(a[k], i + k, b);
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_iadd(int* out, int b) {
  int a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x + k + b;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) asm volatile("add.s32 %0, %0, %1;" : "+r"(a[k]) : "r"(i));
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_imax(int* out, int b) {
  int a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x + k + b;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) asm volatile("max.s32 %0, %0, %1;" : "+r"(a[k]) : "r"(i + k));
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

cudaError_t bench_int_rates(double rates[4]) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256, blocks = sms * 8;
  int* out = nullptr;
  e = cudaMalloc(&out, (size_t)threads * blocks * sizeof(int));
  if (e != cudaSuccess) return e;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  typedef void (*kfn)(int*, int);
  kfn ks[4] = {k_viaddmax, k_vimax3, k_iadd, k_imax};
  for (int k = 0; k < 4; ++k) {
    ks[k]<<<blocks, threads>>>(out, 3);
    float best = 1e30f;
    for (int rep = 0; rep < 5; ++rep) {
      cudaEventRecord(e0);
      ks[k]<<<blocks, threads>>>(out, 3);
      cudaEventRecord(e1);
      cudaEventSynchronize(e1);
      float ms = 0.f;
      cudaEventElapsedTime(&ms, e0, e1);
      if (ms < best) best = ms;
    }
    rates[k] = (double)blocks * threads * ITERS * CH / (best * 1e-3);
  }
  e = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  return e;
}

}  // namespace fz
