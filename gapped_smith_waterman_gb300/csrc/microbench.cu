// Integer-pipe throughput microbenchmark (sm_103a): whole-GPU op/s of the
// instructions a Gotoh cell is built from, in 32-bit and 16-bit pair forms,
// and cells/s of the costed cell itself in both forms.  Each thread runs CH independent
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

// The 16-bit pair forms the first inspector tier issues: each instruction
// advances two cells (two 16-bit halves).
__global__ void k_viaddmax16(int* out, int b) {
  unsigned a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x * 0x10001u + k;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) a[k] = __viaddmax_s16x2_relu(a[k], (unsigned)b, (unsigned)i);
  }
  unsigned s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

__global__ void k_vimax3_16(int* out, int b) {
  unsigned a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x * 0x10001u + k;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) a[k] = __vimax3_s16x2_relu(a[k], (unsigned)(i + k), (unsigned)b);
  }
  unsigned s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

__global__ void k_vadd2(int* out, int b) {
  unsigned a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x * 0x10001u + k + (unsigned)b;
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) a[k] = __vadd2(a[k], (unsigned)i);
  }
  unsigned s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

// A 32-bit add written as a multiply-add by a runtime 1 (the form the kernels
// use to put adds on the FMA pipe).
__global__ void k_imad(int* out, int b) {
  int a[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) a[k] = threadIdx.x + k + b;
  const int one = b - 2;   // 1 at run time (b = 3)
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CH; ++k) asm volatile("mad.lo.s32 %0, %0, %1, %2;" : "+r"(a[k]) : "r"(one), "r"(i));
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CH; ++k) s ^= a[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// The costed operations of one Gotoh cell pair in the 16-bit pair form, with
// independent cells per thread: two add-max (I, D), the diagonal add, the
// 3-way max and the add for h = S - (o + e).  Cells per second of this loop
// is the integer-pipe roofline of the pair sweep measured directly (the DPX
// forms and the packed adds issue on different pipes, so this is not the
// harmonic mean of the single-operation rates).
constexpr int CC = 4;   // independent cell chains per thread
__global__ void k_cellmix16(int* out, int b) {
  unsigned h[CC], hp[CC], I[CC], D[CC];
#pragma unroll
  for (int k = 0; k < CC; ++k) {
    h[k] = threadIdx.x * 0x10001u + k;
    hp[k] = h[k] ^ 0x00070007u;
    I[k] = h[k] + 0x00030003u;
    D[k] = h[k] + 0x00050005u;
  }
  const unsigned ne2 = (unsigned)b * 0x10001u, noe2 = (unsigned)(b + 1) * 0x10001u;
  for (int i = 0; i < ITERS; ++i) {
    const unsigned s = (unsigned)i * 0x10001u;
#pragma unroll
    for (int k = 0; k < CC; ++k) {
      I[k] = __viaddmax_s16x2_relu(I[k], ne2, h[k]);
      D[k] = __viaddmax_s16x2_relu(D[k], ne2, hp[k]);
      const unsigned g = __vadd2(hp[k], s);
      const unsigned sv = __vimax3_s16x2_relu(g, I[k], D[k]);
      hp[k] = h[k];
      h[k] = __vadd2(sv, noe2);
    }
  }
  unsigned s = 0;
#pragma unroll
  for (int k = 0; k < CC; ++k) s ^= h[k] ^ I[k] ^ D[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

// The cell pair of k_cellmix16 plus the four direction tests of the traced
// sweep (g - S, I - S, h_left - I, h_up - D as packed subtractions).
__global__ void k_cellmix16t(int* out, int b) {
  unsigned h[CC], hp[CC], I[CC], D[CC], f[CC];
#pragma unroll
  for (int k = 0; k < CC; ++k) {
    h[k] = threadIdx.x * 0x10001u + k;
    hp[k] = h[k] ^ 0x00070007u;
    I[k] = h[k] + 0x00030003u;
    D[k] = h[k] + 0x00050005u;
    f[k] = 0u;
  }
  const unsigned ne2 = (unsigned)b * 0x10001u, noe2 = (unsigned)(b + 1) * 0x10001u;
  for (int i = 0; i < ITERS; ++i) {
    const unsigned s = (unsigned)i * 0x10001u;
#pragma unroll
    for (int k = 0; k < CC; ++k) {
      const unsigned ic = __viaddmax_s16x2_relu(I[k], ne2, h[k]);
      const unsigned dc = __viaddmax_s16x2_relu(D[k], ne2, hp[k]);
      const unsigned g = __vadd2(hp[k], s);
      const unsigned sv = __vimax3_s16x2_relu(g, ic, dc);
      f[k] ^= __vsub2(g, sv) ^ __vsub2(ic, sv) ^ __vsub2(h[k], ic) ^ __vsub2(hp[k], dc);
      I[k] = ic;
      D[k] = dc;
      hp[k] = h[k];
      h[k] = __vadd2(sv, noe2);
    }
  }
  unsigned s = 0;
#pragma unroll
  for (int k = 0; k < CC; ++k) s ^= h[k] ^ I[k] ^ D[k] ^ f[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

// The same cell in 32-bit form (one cell per lane and instruction), adds as
// multiply-adds by a runtime 1 as the 32-bit sweeps and the local fill write them.
__global__ void k_cellmix32(int* out, int b) {
  int h[CC], hp[CC], I[CC], D[CC];
#pragma unroll
  for (int k = 0; k < CC; ++k) {
    h[k] = threadIdx.x + k;
    hp[k] = h[k] ^ 7;
    I[k] = h[k] + 3;
    D[k] = h[k] + 5;
  }
  const int one = b - 2, ne = -b, noe = -(b + 1);
  for (int i = 0; i < ITERS; ++i) {
#pragma unroll
    for (int k = 0; k < CC; ++k) {
      I[k] = __viaddmax_s32(I[k], ne, h[k]);
      D[k] = __viaddmax_s32(D[k], ne, hp[k]);
      int g, hn;
      asm volatile("mad.lo.s32 %0, %1, %2, %3;" : "=r"(g) : "r"(hp[k]), "r"(one), "r"(i));
      const int sv = __vimax3_s32(g, I[k], D[k]);
      asm volatile("mad.lo.s32 %0, %1, %2, %3;" : "=r"(hn) : "r"(sv), "r"(one), "r"(noe));
      hp[k] = h[k];
      h[k] = hn;
    }
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CC; ++k) s ^= h[k] ^ I[k] ^ D[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

cudaError_t bench_int_rates(double rates[FZ_INT_RATES]) {
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
  // operations per thread and loop iteration (cells for the two cell mixes)
  const double per[FZ_INT_RATES] = {CH, CH, CH, CH, CH, CH, CH, CH, 2.0 * CC, CC, 2.0 * CC};
  kfn ks[FZ_INT_RATES] = {k_viaddmax, k_vimax3, k_iadd, k_imax, k_viaddmax16, k_vimax3_16, k_vadd2, k_imad,
                          k_cellmix16, k_cellmix32, k_cellmix16t};
  for (int k = 0; k < FZ_INT_RATES; ++k) {
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
    rates[k] = (double)blocks * threads * ITERS * per[k] / (best * 1e-3);
  }
  e = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  return e;
}

}  // namespace fz
