// Unpruned local fill, score and end cell only (sm_103a).
//
// Recurrence with a zero floor (the local cell of the DPX intrinsics article,
// section 1.1, with affine gaps):
//   E(i,j) = max(E(i,j-1) - e, H(i,j-1) - o - e)
//   F(i,j) = max(F(i-1,j) - e, H(i-1,j) - o - e)
//   H(i,j) = max(0, H(i-1,j-1) + M[t_i][q_j], E(i,j), F(i,j))
// H = 0 and E = F = NEG on row and column 0.  Result: max H, earliest cell by
// (i + j, then i).
//
// One warp per pair.  The query is cut into strips of 32 * KC columns; in a
// strip lane l owns KC consecutive columns and works on row i = tau - l + 1 at
// step tau (a wavefront across lanes), so each step needs only H and E of the
// column left of its block, from lane l-1 by shuffle.  The column between two
// strips is kept per row in a spill buffer (shared memory when it fits).  H
// and F of a lane's columns stay in registers; the substitution score is one
// byte permute of the column's 4-byte score profile by the row's target base.
// The DPX 3-way max with ReLU does the zero floor for free.
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int WL = 4;          // warps per block
constexpr int KC = 32;         // columns per lane
constexpr int SW = 32 * KC;    // strip width

struct Res {
  uint64_t res;
  uint32_t pend;
  int32_t cnt;
  int64_t next;
};

__device__ __forceinline__ void rinit(Res& r, const uint8_t* s, uint64_t len, int64_t g0, int dir, int64_t first) {
  r.res = fetch16(s, len, g0, dir, first);
  r.pend = fetch16(s, len, g0, dir, first + 16);
  r.cnt = 16;
  r.next = first + 32;
}

__device__ __forceinline__ uint32_t rtake(Res& r, const uint8_t* s, uint64_t len, int64_t g0, int dir) {
  const uint32_t b = (uint32_t)r.res & 3u;
  r.res >>= 2;
  if (--r.cnt < 16) {
    r.res |= (uint64_t)r.pend << (2 * r.cnt);
    r.cnt += 16;
    r.pend = fetch16(s, len, g0, dir, r.next);
    r.next += 16;
  }
  return b;
}

template <bool PARTIAL>
__device__ __forceinline__ void strip(const Params& p, const Window& w, int lane, int32_t s, int32_t nstrips,
                                      const uint32_t* s_mcol, int32_t* spH, int32_t* spE, int32_t& bv,
                                      int32_t& bd, int32_t& bi) {
  // Scores are kept as h = H - o - e (the gap-open source of both neighbours),
  // so each cell subtracts o + e once.
  const int32_t m = w.m, n = w.n, oe = p.oe, ne = -p.e, c1 = oe - 128;
  const int32_t c0 = s * SW + lane * KC + 1;
  const int32_t kv = imax(0, imin(KC, n - c0 + 1));
  uint32_t QPF[KC];
  int32_t hc[KC], F[KC];
  {
    const uint32_t q0 = fetch16(p.q2, p.q_len, w.qg0, w.dir, c0);
    const uint32_t q1 = fetch16(p.q2, p.q_len, w.qg0, w.dir, c0 + 16);
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const uint32_t qb = ((k < 16 ? q0 : q1) >> (2 * (k & 15))) & 3u;
      QPF[k] = s_mcol[qb];
      hc[k] = -oe;                                       // row 0: H = 0
      F[k] = NEG;
    }
  }
  Res tr;
  rinit(tr, p.t2, p.t_len, w.tg0, w.dir, 1);
  int32_t h_out = -oe, e_out = NEG, hh_prev = -oe;
  uint32_t t_cur = 0;
  const bool first = s == 0, last = s == nstrips - 1;
  for (int32_t tau = 0; tau < m + 31; ++tau) {
    const int32_t i = tau - lane + 1;
    int32_t hh = __shfl_up_sync(FULL, h_out, 1);
    int32_t eh = __shfl_up_sync(FULL, e_out, 1);
    uint32_t tb = __shfl_up_sync(FULL, t_cur, 1);
    const uint32_t t0 = rtake(tr, p.t2, p.t_len, w.tg0, w.dir);
    if (lane == 0) {
      tb = t0;
      if (first) { hh = -oe; eh = NEG; }                 // column 0: H = 0
      else if (i <= m) { hh = spH[i]; eh = spE[i]; }
    }
    if (i >= 1 && i <= m) {
      const uint32_t tsel = 0x4440u | tb;
      int32_t E = eh, hl = hh, hd = hh_prev, rmax = 0;
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        E = __viaddmax_s32(E, ne, hl);
        F[k] = __viaddmax_s32(F[k], ne, hc[k]);
        const int32_t G = hd + (int32_t)prmt(QPF[k], 0u, tsel) + c1;
        int32_t H = __vimax3_s32_relu(G, E, F[k]);
        if (PARTIAL) H = k < kv ? H : 0;
        const int32_t h = H - oe;
        hd = hc[k];
        hc[k] = h;
        hl = h;
        rmax = imax(rmax, H);   // row max in score space
      }
      h_out = hl;
      e_out = E;
      if (rmax >= bv && rmax > 0) {
        const int32_t rh = rmax - oe;
        int kf = KC;
#pragma unroll
        for (int k = KC - 1; k >= 0; --k) kf = hc[k] == rh ? k : kf;
        const int32_t c = c0 + kf, d = i + c;
        if (rmax > bv || d < bd || (d == bd && i < bi)) { bv = rmax; bd = d; bi = i; }
      }
      if (lane == 31 && !last) { spH[i] = hl; spE[i] = E; }
    }
    hh_prev = hh;
    t_cur = tb;
  }
  __syncwarp();
}

__global__ void __launch_bounds__(WL * 32, 3) k_local(Params p, LocalArgs la) {
  extern __shared__ int32_t smem[];
  __shared__ uint32_t s_mcol[4];
  if (threadIdx.x < 4) s_mcol[threadIdx.x] = la.mcol[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t cap = p.max_len + 1;
  int32_t* sp = la.use_smem ? smem + (size_t)warp * 2 * cap
                            : la.spill + ((uint64_t)blockIdx.x * WL + warp) * la.spill_stride;
  int32_t* spH = sp;
  int32_t* spE = sp + cap;
  for (;;) {
    uint32_t ext = 0;
    if (lane == 0) ext = atomicAdd(la.counter, 1u);
    ext = __shfl_sync(FULL, ext, 0);
    if (ext >= la.n_work) break;
    const Window w = make_window(p, ext);
    ExtRec* R = la.rec + ext;
    if (!w.requested) {
      if (lane == 0) { ExtRec z = {}; *R = z; }
      continue;
    }
    int32_t bv = 0, bd = 0, bi = 0;
    const int32_t nstrips = (w.n + SW - 1) / SW;
    if (w.m > 0) {
      for (int32_t s = 0; s < nstrips; ++s) {
        const bool partial = (s + 1) * SW > w.n;
        if (partial) strip<true>(p, w, lane, s, nstrips, s_mcol, spH, spE, bv, bd, bi);
        else strip<false>(p, w, lane, s, nstrips, s_mcol, spH, spE, bv, bd, bi);
      }
    }
    const int32_t wm = __reduce_max_sync(FULL, bv);
    const uint32_t dmin = __reduce_min_sync(FULL, bv == wm ? (uint32_t)bd : 0xffffffffu);
    const uint32_t imn = __reduce_min_sync(FULL, (bv == wm && (uint32_t)bd == dmin) ? (uint32_t)bi : 0xffffffffu);
    if (lane == 0) {
      ExtRec o;
      o.score = wm;
      o.i_end = wm > 0 ? (int32_t)imn : 0;
      o.j_end = wm > 0 ? (int32_t)dmin - (int32_t)imn : 0;
      o.d_last = w.m + w.n;
      o.live = (uint64_t)w.m * (uint64_t)w.n;
      o.path = 0; o.flags = FZ_FLAG_DONE; o.npath = 0;
      o.m = w.m; o.n = w.n; o.width = 0; o.ckpt = 0;
      *R = o;
      atomicAdd(la.live_total, (unsigned long long)o.live);
    }
  }
}

}  // namespace

int local_warps_per_block() { return WL; }
size_t local_smem_bytes(int32_t max_len) { return (size_t)WL * 2 * (size_t)(max_len + 1) * sizeof(int32_t); }

int local_blocks_per_sm(size_t smem) {
  int nb = 0;
  if (smem > 48 * 1024) cudaFuncSetAttribute(k_local, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_local, WL * 32, smem);
  return nb > 0 ? nb : 1;
}

cudaError_t launch_local(const Params& p, const LocalArgs& la, int grid, cudaStream_t st) {
  const size_t smem = la.use_smem ? local_smem_bytes(p.max_len) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_local, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_local<<<grid, WL * 32, smem, st>>>(p, la);
  return cudaGetLastError();
}

}  // namespace fz

// ---------------------------------------------------------------------------
// Allocation-free local fill (fz_local_fill_noalloc in fz.h).
//
// For callers that cannot allocate device memory at run time (an allocator
// that is already locked, an embedding runtime that forbids cudaMalloc on its
// hot path).  Its scratch -- the work counter and the per-warp strip spill
// rows -- lives in one file-scope device array instead of context memory; the
// kernel always uses these global spill rows, never dynamic shared memory.
// ---------------------------------------------------------------------------
#include <mutex>

namespace fz {

namespace {

constexpr int32_t NA_MAX_LEN = 2048;                        // longest window per side
constexpr int NA_MAX_BLOCKS = 152;                          // one block of WL warps per SM
constexpr uint64_t NA_SPILL = 2ull * (NA_MAX_LEN + 1);      // int32 per warp
constexpr uint64_t NA_HEAD = 64;                            // word 0: work counter
constexpr uint64_t NA_WORDS = NA_HEAD + (uint64_t)NA_MAX_BLOCKS * WL * NA_SPILL;   // ~10 MB

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) int32_t g_noalloc_scratch[NA_WORDS];

__global__ void __launch_bounds__(WL * 32) k_local_noalloc(Params p, uint32_t n_work, int32_t* scratch,
                                                           fz_result* out, uint4 mcol) {
  __shared__ uint32_t s_mcol[4];
  if (threadIdx.x == 0) {
    s_mcol[0] = mcol.x; s_mcol[1] = mcol.y; s_mcol[2] = mcol.z; s_mcol[3] = mcol.w;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* counter = reinterpret_cast<uint32_t*>(scratch);
  int32_t* sp = scratch + NA_HEAD + ((uint64_t)blockIdx.x * WL + warp) * NA_SPILL;
  int32_t* spH = sp;
  int32_t* spE = sp + (p.max_len + 1);
  for (;;) {
    uint32_t ext = 0;
    if (lane == 0) ext = atomicAdd(counter, 1u);
    ext = __shfl_sync(FULL, ext, 0);
    if (ext >= n_work) break;
    const Window w = make_window(p, ext);
    if (!w.requested) {
      if (lane == 0) { fz_result z = {0, 0, 0, 0, 0, 0}; out[ext] = z; }
      continue;
    }
    int32_t bv = 0, bd = 0, bi = 0;
    const int32_t nstrips = (w.n + SW - 1) / SW;
    if (w.m > 0) {
      for (int32_t s = 0; s < nstrips; ++s) {
        if ((s + 1) * SW > w.n) strip<true>(p, w, lane, s, nstrips, s_mcol, spH, spE, bv, bd, bi);
        else strip<false>(p, w, lane, s, nstrips, s_mcol, spH, spE, bv, bd, bi);
      }
    }
    const int32_t wm = __reduce_max_sync(FULL, bv);
    const uint32_t dmin = __reduce_min_sync(FULL, bv == wm ? (uint32_t)bd : 0xffffffffu);
    const uint32_t imn = __reduce_min_sync(FULL, (bv == wm && (uint32_t)bd == dmin) ? (uint32_t)bi : 0xffffffffu);
    if (lane == 0) {
      fz_result o;
      o.score = wm;
      o.t_end = wm > 0 ? (int32_t)imn : 0;
      o.q_end = wm > 0 ? (int32_t)dmin - (int32_t)imn : 0;
      o.cigar_off = 0;
      o.cigar_len = 0;
      o.flags = FZ_FLAG_DONE;
      out[ext] = o;
    }
  }
}

}  // namespace

}  // namespace fz

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[256] = {};   // device address of g_noalloc_scratch, per device ordinal

// Resolves the scratch array's device address for the current device.  The
// name g_noalloc_scratch in host code is only a host-side stand-in; kernels
// must be given this address instead.  Outside stream capture the address is
// looked up again on every call (a context made after cudaDeviceReset gets a
// new one); while the stream is capturing, the address cached by the last
// call outside capture is used, and without one the call fails.
cudaError_t noalloc_scratch(int dev, cudaStream_t st, int32_t** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t ce = cudaStreamIsCapturing(st, &cs);
  if (ce != cudaSuccess) return ce;
  if (cs == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, fz::g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  } else if (!g_noalloc_ptr[dev]) {
    return cudaErrorStreamCaptureUnsupported;
  }
  *out = static_cast<int32_t*>(g_noalloc_ptr[dev]);
  return cudaSuccess;
}

}  // namespace

extern "C" fz_status fz_local_fill_noalloc(const int32_t sub[16], int32_t gap_open, int32_t gap_extend,
                                           int32_t max_len, const uint8_t* d_target2, uint64_t t_len,
                                           const uint8_t* d_query2, uint64_t q_len, const fz_seed* d_seeds,
                                           uint32_t n_seeds, fz_result* d_out, void* cuda_stream) {
  using namespace fz;
  if (!sub || gap_open < 0 || gap_extend < 1 || max_len < 1 || max_len > NA_MAX_LEN) return FZ_ERR_ARG;
  if (n_seeds > 0x7fffffffu) return FZ_ERR_ARG;
  if (n_seeds && (!d_seeds || !d_out)) return FZ_ERR_ARG;
  if ((t_len && !d_target2) || (q_len && !d_query2)) return FZ_ERR_ARG;
  int64_t amax = (int64_t)gap_open + gap_extend;
  for (int k = 0; k < 16; ++k) {
    if (sub[k] < -128 || sub[k] > 127) return FZ_ERR_ARG;
    amax = amax > (sub[k] < 0 ? -(int64_t)sub[k] : sub[k]) ? amax : (sub[k] < 0 ? -(int64_t)sub[k] : sub[k]);
  }
  if (amax * (2 * (int64_t)max_len + 1) >= (1ll << 28)) return FZ_ERR_ARG;
  if (n_seeds == 0) return FZ_OK;
  // an error left pending by earlier, unrelated work is the caller's: report
  // it without clearing it and before touching the stream
  if (cudaPeekAtLastError() != cudaSuccess) return FZ_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) { (void)cudaGetLastError(); return FZ_ERR_CUDA; }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return FZ_ERR_CUDA;
  }
  int32_t* scratch = nullptr;
  if (noalloc_scratch(dev, st, &scratch) != cudaSuccess) { (void)cudaGetLastError(); return FZ_ERR_CUDA; }
  Params p{};
  p.t2 = d_target2; p.q2 = d_query2; p.t_len = t_len; p.q_len = q_len;
  p.seeds = d_seeds; p.n_seeds = n_seeds;
  p.o = gap_open; p.e = gap_extend; p.oe = gap_open + gap_extend;
  p.ydrop = FZ_YDROP_INF; p.max_len = max_len; p.one = 1;
  for (int k = 0; k < 16; ++k) p.sub[k] = sub[k];
  uint32_t mc[4];
  for (int t = 0; t < 4; ++t) {
    uint32_t col = 0;
    for (int q = 0; q < 4; ++q) col |= (uint32_t)(sub[q * 4 + t] + 128) << (8 * q);
    mc[t] = col;
  }
  // the work counter must start at zero; the spill rows need no clearing
  if (cudaMemsetAsync(scratch, 0, NA_HEAD * sizeof(int32_t), st) != cudaSuccess) {
    (void)cudaGetLastError();
    return FZ_ERR_CUDA;
  }
  const int grid = sms < NA_MAX_BLOCKS ? sms : NA_MAX_BLOCKS;
  k_local_noalloc<<<grid, WL * 32, 0, st>>>(p, 2 * n_seeds, scratch, d_out, make_uint4(mc[0], mc[1], mc[2], mc[3]));
  if (cudaGetLastError() != cudaSuccess) return FZ_ERR_CUDA;   // this launch's error (none was pending)
  return FZ_OK;
}
