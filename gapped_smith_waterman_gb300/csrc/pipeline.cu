// Device-side length binning, scans and CIGAR emission (sm_103a).
//
// Binning follows FastZ section 3.3: an extension whose best cell (i*, j*) lies
// outside the 16x16 eager corner goes to the smallest bin whose box contains it,
// boxes 512, 2048, 8192, 32768 (the paper's four) and 131072 (one more 4x step,
// as the paper allows).  The paper sorts on the host; here a block-local
// histogram and scatter build the executor's work list on the device, largest
// bin first so that the longest extensions start first.
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int TB = 256;

__device__ __forceinline__ uint32_t bin_of(int32_t i, int32_t j) {
  const int32_t mx = imax(i, j);
  return mx <= 512 ? 1u : mx <= 2048 ? 2u : mx <= 8192 ? 3u : mx <= 32768 ? 4u : 5u;
}

// Upper bound on the CIGAR runs of an alignment ending at (i, j).  The traced
// alignment scores S* >= 0, so its g gap runs (each costing at least o + e)
// are paid for by at most min(i, j) diagonal scores of at most max_sub each:
// g <= max_sub * min(i, j) / (o + e); match runs number at most g + 1; and no
// alignment has more runs than ops (i + j).
__device__ __forceinline__ uint64_t cigar_cap(int32_t i, int32_t j, int32_t oe, int32_t max_sub) {
  const uint64_t ops = (uint64_t)i + (uint64_t)j;
  const uint64_t g = (uint64_t)max_sub * (uint64_t)imin(i, j) / (uint64_t)(oe > 0 ? oe : 1);
  const uint64_t runs = 2 * g + 1;
  return runs < ops ? runs : ops;
}

__global__ void k_classify(PipeArgs a) {
  __shared__ uint32_t h[8];
  if (threadIdx.x < 8) h[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x < a.n_ext) {
    const ExtRec r = a.rec[x];
    uint32_t bin = 0;
    uint64_t cap = 0;
    if (r.flags & FZ_FLAG_DONE) {
      atomicAdd(&h[7], 1u);
      if (!a.local) {
        cap = cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub);
        if (r.flags & FZ_FLAG_EAGER) {
          atomicAdd(&h[0], 1u);
        } else {
          bin = bin_of(r.i_end, r.j_end);
          atomicAdd(&h[bin], 1u);
        }
      }
    }
    a.ext_bin[x] = bin;
    a.cig_cap[x] = cap;
  }
  __syncthreads();
  if (threadIdx.x < 8 && h[threadIdx.x]) atomicAdd(&a.bin_count[threadIdx.x], h[threadIdx.x]);
}

// cursor[k] = first executor slot of bin k; bins are laid out 5, 4, 3, 2, 1
__global__ void k_bin_starts(PipeArgs a) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    uint32_t c = 0;
    for (int k = 5; k >= 1; --k) {
      a.bin_cursor[k] = c;
      c += a.bin_count[k];
    }
    a.bin_cursor[0] = c;   // executor items
  }
}

__global__ void k_scatter(PipeArgs a) {
  __shared__ uint32_t cnt[8], base[8];
  if (threadIdx.x < 8) cnt[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t bin = 0, local_pos = 0;
  if (x < a.n_ext) {
    bin = a.ext_bin[x];
    if (bin) local_pos = atomicAdd(&cnt[bin], 1u);
  }
  __syncthreads();
  if (threadIdx.x >= 1 && threadIdx.x <= 5 && cnt[threadIdx.x])
    base[threadIdx.x] = atomicAdd(&a.bin_cursor[threadIdx.x], cnt[threadIdx.x]);
  __syncthreads();
  if (x < a.n_ext && bin) {
    const uint32_t pos = base[bin] + local_pos;
    const ExtRec r = a.rec[x];
    a.exec_list[pos] = x;
    a.exec_pos[x] = pos;
    a.trace_sz[pos] = trace_bytes(r.width, r.i_end + r.j_end);
  }
}

// ---- exclusive scan of uint64 (3 passes, 2048 elements per block) ----
constexpr int SCAN_T = 1024;
constexpr int SCAN_E = 2 * SCAN_T;

__device__ __forceinline__ uint64_t block_excl_scan(uint64_t v, uint64_t* warp_tot, uint64_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint64_t t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(FULL, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  total = warp_tot[31];
  const uint64_t before = wid ? warp_tot[wid - 1] : 0;
  return before + x - v;
}

__global__ void __launch_bounds__(SCAN_T) k_scan1(uint64_t* d, uint32_t n, uint64_t* bsum) {
  __shared__ uint64_t wt[32];
  const uint64_t i0 = (uint64_t)blockIdx.x * SCAN_E + 2 * threadIdx.x;
  const uint64_t a = i0 < n ? d[i0] : 0, b = i0 + 1 < n ? d[i0 + 1] : 0;
  uint64_t total;
  const uint64_t ex = block_excl_scan(a + b, wt, total);
  if (i0 < n) d[i0] = ex;
  if (i0 + 1 < n) d[i0 + 1] = ex + a;
  if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

__global__ void __launch_bounds__(SCAN_T) k_scan2(uint64_t* bsum, uint32_t nb, uint64_t* total_out) {
  __shared__ uint64_t wt[32];
  uint64_t carry = 0;
  for (uint32_t c = 0; c < nb; c += SCAN_T) {
    const uint32_t k = c + threadIdx.x;
    const uint64_t v = k < nb ? bsum[k] : 0;
    uint64_t total;
    const uint64_t ex = block_excl_scan(v, wt, total);
    if (k < nb) bsum[k] = carry + ex;
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) *total_out = carry;
}

__global__ void k_scan3(uint64_t* d, uint32_t n, const uint64_t* bsum) {
  const uint64_t i = (uint64_t)blockIdx.x * SCAN_E + threadIdx.x;
  const uint64_t add = bsum[blockIdx.x];
  if (i < n) d[i] += add;
  if (i + SCAN_T < n) d[i + SCAN_T] += add;
}

// ---- CIGAR emission ----
// Ops arrive in walk order (from the best cell back to the anchor) and are
// merged into runs.  Right side: the genomic order is the reverse of the walk,
// so runs are written backwards from the end of the extension's slot; left
// side: the walk order is already genomic.
struct RunWriter {
  uint32_t* dst;
  uint64_t off, cap;
  bool backwards;
  uint32_t op, len, nruns;
  bool overflow;
  __device__ void init(uint32_t* c, uint64_t o, uint64_t k, bool bw) {
    dst = c; off = o; cap = k; backwards = bw; op = 0xffu; len = 0; nruns = 0; overflow = false;
  }
  __device__ void flush() {
    if (!len) return;
    if (nruns >= cap) { overflow = true; return; }   // never write outside the slot
    const uint64_t at = backwards ? off + cap - 1 - nruns : off + nruns;
    dst[at] = (len << 4) | op;
    ++nruns;
  }
  __device__ void push(uint32_t o) {
    if (o == op) { ++len; return; }
    flush();
    op = o;
    len = 1;
  }
  __device__ uint32_t first() const { return (uint32_t)(backwards ? off + cap - nruns : off); }
};

__device__ __forceinline__ void write_out(fz_result* out, const ExtRec& r, uint32_t coff, uint32_t clen, uint32_t bin) {
  fz_result o;
  o.score = r.score;
  o.t_end = r.i_end;
  o.q_end = r.j_end;
  o.cigar_off = coff;
  o.cigar_len = clen;
  o.flags = (r.flags & (FZ_FLAG_DONE | FZ_FLAG_EAGER | FZ_FLAG_WIDE)) | (bin << FZ_FLAG_BIN_SHIFT);
  *out = o;
}

__global__ void k_emit_direct(EmitArgs a) {
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= a.n_ext) return;
  const ExtRec r = a.rec[x];
  if (!(r.flags & FZ_FLAG_DONE)) {
    fz_result z = {0, 0, 0, 0, 0, 0};
    a.out[x] = z;
    return;
  }
  if (a.local) { write_out(a.out + x, r, 0, 0, 0); return; }
  if (!(r.flags & FZ_FLAG_EAGER)) return;       // executor extension: k_emit_exec
  const uint64_t off = a.cig_off[x];
  const uint64_t cap = cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub);
  RunWriter wr;
  wr.init(a.cigar, off, cap, (x & 1u) == 0u);
  for (uint32_t k = 0; k < r.npath; ++k) wr.push((uint32_t)(r.path >> (2 * k)) & 3u);
  wr.flush();
  if (wr.overflow) atomicOr(a.err, 16u);
  write_out(a.out + x, r, wr.nruns ? wr.first() : (uint32_t)off, wr.nruns, 0);
}

__global__ void k_emit_exec(EmitArgs a) {
  const uint32_t pos = a.exec_begin + blockIdx.x * blockDim.x + threadIdx.x;
  if (pos >= a.exec_end) return;
  const uint32_t x = a.exec_list[pos];
  const ExtRec r = a.rec[x];
  const int32_t dend = r.i_end + r.j_end;
  const uint32_t W = r.width;
  const uint8_t* base = a.trace + (a.trace_off[pos] - a.trace_sub);
  const int32_t* lo = reinterpret_cast<const int32_t*>(base + trace_lo_offset(W, dend));
  const uint64_t off = a.cig_off[x];
  RunWriter wr;
  wr.init(a.cigar, off, cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub), (x & 1u) == 0u);
  int32_t i = r.i_end, j = r.j_end, st = 0;
  int64_t guard = 2 * (int64_t)dend + 4;
  while ((i > 0 || j > 0) && --guard > 0) {
    if (i < 0 || j < 0) { atomicOr(a.err, 1u); break; }
    const int32_t d = i + j;
    const int32_t u = i - lo[d];
    if (u < 0 || (uint32_t)u >= W) { atomicOr(a.err, 1u); break; }
    const uint32_t c = (base[(uint64_t)d * (W / 2) + (uint32_t)(u >> 1)] >> (4 * (u & 1))) & 15u;
    // The walk visits one row per step, going down in d: pull the row it will
    // reach PF anti-diagonals later (around where the path should be) and the
    // row origins further ahead into L2.  Addresses stay inside this
    // extension's rows.
    constexpr int32_t PF = 12;
    if (d >= PF) {
      const int32_t dp = d - PF;
      int32_t up = i - PF / 2 - lo[dp];
      up = up < 0 ? 0 : ((uint32_t)up >= W ? (int32_t)W - 1 : up);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (uint64_t)dp * (W / 2) + (uint32_t)(up >> 1)));
      if (d >= 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(lo + (d - 64)));
    }
    if (st == 0) {
      const uint32_t sc = c & 3u;
      if (sc == 0) { wr.push(0); --i; --j; }
      else if (sc == 3) { atomicOr(a.err, 2u); break; }
      else st = (int)sc;
    } else if (st == 1) {
      wr.push(1);
      st = (c & 4u) ? 0 : 1;
      --j;
    } else {
      wr.push(2);
      st = (c & 8u) ? 0 : 2;
      --i;
    }
  }
  if (guard <= 0) atomicOr(a.err, 4u);
  wr.flush();
  if (wr.overflow) atomicOr(a.err, 16u);
  write_out(a.out + x, r, wr.nruns ? wr.first() : (uint32_t)off, wr.nruns, a.local ? 0u : bin_of(r.i_end, r.j_end));
}

}  // namespace

cudaError_t launch_classify(const PipeArgs& a, cudaStream_t st) {
  const uint32_t g = (a.n_ext + TB - 1) / TB;
  if (g) k_classify<<<g, TB, 0, st>>>(a);
  k_bin_starts<<<1, 32, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const PipeArgs& a, cudaStream_t st) {
  const uint32_t g = (a.n_ext + TB - 1) / TB;
  if (g) k_scatter<<<g, TB, 0, st>>>(a);
  return cudaGetLastError();
}

uint32_t scan_tmp_elems(uint32_t n) { return (n + SCAN_E - 1) / SCAN_E + 1; }

cudaError_t launch_scan_u64(uint64_t* data, uint32_t n, uint64_t* block_tmp, uint64_t* total, cudaStream_t st) {
  const uint32_t nb = (n + SCAN_E - 1) / SCAN_E;
  if (nb == 0) {
    cudaMemsetAsync(total, 0, sizeof(uint64_t), st);
    return cudaGetLastError();
  }
  k_scan1<<<nb, SCAN_T, 0, st>>>(data, n, block_tmp);
  k_scan2<<<1, SCAN_T, 0, st>>>(block_tmp, nb, total);
  k_scan3<<<nb, SCAN_T, 0, st>>>(data, n, block_tmp);
  return cudaGetLastError();
}

cudaError_t launch_emit_direct(const EmitArgs& a, cudaStream_t st) {
  const uint32_t g = (a.n_ext + TB - 1) / TB;
  if (g) k_emit_direct<<<g, TB, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_emit_exec(const EmitArgs& a, cudaStream_t st) {
  const uint32_t n = a.exec_end - a.exec_begin;
  const uint32_t g = (n + 127) / 128;
  if (g) k_emit_exec<<<g, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fz
