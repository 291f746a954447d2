// General-band anti-diagonal sweep (sm_103a): the path for extensions whose
// live band outgrows the register window (very large ydrop, long gapped
// regions).  One warp per extension; the last three anti-diagonals live in a
// per-warp global scratch indexed by target row (L1/L2 resident), each lane
// computes one cell of a 32-cell chunk, chunks cover the candidate band
// [lo, hi] of the anti-diagonal: rows that have a live predecessor on one of
// the two previous anti-diagonals (FastZ section 3.2 strips, spilled to memory
// instead of kept in registers).  Liveness is tracked exactly as written in
// the y-drop rule: dead cells hold NEG in S, I and D.
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int WW = 4;   // warps per block

__device__ __forceinline__ uint32_t base_at(const uint8_t* __restrict__ s, uint64_t len, int64_t g0, int dir,
                                            int64_t w) {
  const int64_t g = g0 + dir * w;
  if (g < 0 || (uint64_t)g >= len) return 0u;
  return ((uint32_t)__ldg(s + (g >> 2)) >> ((g & 3) * 2)) & 3u;
}

__device__ __forceinline__ int mod3(int32_t d) { return ((d % 3) + 3) % 3; }

template <bool TRACE>
__device__ void wide_ext(const Params& p, const WorkArgs& wa, uint32_t ext, uint32_t idx, int lane,
                         int32_t* buf, int32_t cap, const int32_t* s_sub) {
  const Window w = make_window(p, ext);
  ExtRec* R = wa.rec + ext;
  if (!w.requested) {
    if (!TRACE && lane == 0) {
      ExtRec z = {};
      *R = z;
    }
    return;
  }
  const int32_t m = w.m, n = w.n, oe = p.oe, e = p.e;
  int32_t* Sb[3];
  int32_t* Ib[3];
  int32_t* Db[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    Sb[k] = buf + (3 * k + 0) * (int64_t)cap;
    Ib[k] = buf + (3 * k + 1) * (int64_t)cap;
    Db[k] = buf + (3 * k + 2) * (int64_t)cap;
  }
  int32_t blo[3], bhi[3], llo[3], lhi[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) { blo[k] = 1; bhi[k] = 0; llo[k] = 1; lhi[k] = 0; }
  if (lane == 0) { Sb[0][0] = 0; Ib[0][0] = NEG; Db[0][0] = NEG; }
  blo[0] = 0; bhi[0] = 0; llo[0] = 0; lhi[0] = 0;

  int32_t d_stop = 0x7fffffff;
  uint32_t W = 0;
  uint8_t* tbase = nullptr;
  int32_t* lo_arr = nullptr;
  if (TRACE) {
    d_stop = R->i_end + R->j_end;
    W = R->width;
    tbase = wa.trace + (wa.trace_off[idx] - wa.trace_sub);
    lo_arr = reinterpret_cast<int32_t*>(tbase + trace_lo_offset(W, d_stop));
    if (lane == 0) lo_arr[0] = 0;
  }
  int32_t best = 0, bi = 0, bj = 0, d_last = 0, wrun = 1, wbest = 1;
  uint32_t cnt = lane == 0 ? 1u : 0u;
  __syncwarp();

  for (int32_t dn = 1; dn <= m + n; ++dn) {
    if (dn > d_stop) break;
    const int k1 = mod3(dn - 1), k2 = mod3(dn - 2), kc = mod3(dn);
    int32_t lo = 0x7fffffff, hi = -0x7fffffff;
    if (lhi[k1] >= llo[k1]) { lo = llo[k1]; hi = lhi[k1] + 1; }
    if (lhi[k2] >= llo[k2]) { lo = imin(lo, llo[k2] + 1); hi = imax(hi, lhi[k2] + 1); }
    lo = imax(lo, imax(0, dn - n));
    hi = imin(hi, imin(m, dn));
    if (lo > hi) break;
    const int32_t T = threshold(best, p.ydrop);
    int32_t mx = NEG, mi = 0x7fffffff, a_lo = 0x7fffffff, a_hi = -1;
    for (int32_t c = lo; c <= hi; c += 32) {
      const int32_t i = c + lane;
      const bool act = i <= hi;
      const int32_t j = dn - i;
      int32_t sl = NEG, il = NEG, su = NEG, du = NEG, sd = NEG;
      if (act) {
        if (j >= 1 && i >= blo[k1] && i <= bhi[k1]) { sl = Sb[k1][i]; il = Ib[k1][i]; }
        if (i >= 1 && i - 1 >= blo[k1] && i - 1 <= bhi[k1]) { su = Sb[k1][i - 1]; du = Db[k1][i - 1]; }
        if (i >= 1 && j >= 1 && i - 1 >= blo[k2] && i - 1 <= bhi[k2]) sd = Sb[k2][i - 1];
      }
      const int32_t Iv = j >= 1 ? imax(il - e, sl - oe) : NEG;
      const int32_t Dv = i >= 1 ? imax(du - e, su - oe) : NEG;
      int32_t G = NEG;
      if (act && i >= 1 && j >= 1) {
        const uint32_t tb = base_at(p.t2, p.t_len, w.tg0, w.dir, i);
        const uint32_t qb = base_at(p.q2, p.q_len, w.qg0, w.dir, j);
        G = sd + s_sub[tb * 4 + qb];
      }
      const int32_t S = imax(G, imax(Iv, Dv));
      const bool alive = act && S >= T;
      if (act) {
        Sb[kc][i] = alive ? S : NEG;
        Ib[kc][i] = alive ? Iv : NEG;
        Db[kc][i] = alive ? Dv : NEG;
      }
      if (alive) {
        ++cnt;
        if (S > mx) { mx = S; mi = i; }
        a_lo = imin(a_lo, i);
        a_hi = imax(a_hi, i);
      }
      if (TRACE) {
        const uint32_t code = (G == S ? 0u : (Iv == S ? 1u : 2u)) | (j >= 1 && Iv == sl - oe ? 4u : 0u) |
                              (i >= 1 && Dv == su - oe ? 8u : 0u);
        const uint32_t hi4 = __shfl_down_sync(FULL, code, 1);
        const uint32_t u = (uint32_t)(i - lo);
        if (act && !(lane & 1) && u < W) tbase[(uint64_t)dn * (W / 2) + (u >> 1)] = (uint8_t)(code | (hi4 << 4));
      }
    }
    const int32_t wm = __reduce_max_sync(FULL, mx);
    const uint32_t wi = __reduce_min_sync(FULL, (mx == wm && mx != NEG) ? (uint32_t)mi : 0xffffffffu);
    const int32_t nlo = (int32_t)__reduce_min_sync(FULL, (uint32_t)a_lo);
    const int32_t nhi = (int32_t)__reduce_max_sync(FULL, (uint32_t)(a_hi + 1)) - 1;
    blo[kc] = lo; bhi[kc] = hi;
    llo[kc] = nlo; lhi[kc] = nhi;
    wrun = imax(wrun, hi - lo + 1);
    if (wm != NEG) {
      d_last = dn;
      if (wm > best) { best = wm; bi = (int32_t)wi; bj = dn - bi; wbest = wrun; }
    }
    if (TRACE && lane == 0) lo_arr[dn] = lo;
    __syncwarp();
  }
  uint64_t tot = cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  if (TRACE) {
    if (lane == 0) {
      atomicAdd(wa.exec_total, (unsigned long long)tot);
      atomicAdd(wa.exec_live, (unsigned long long)tot);
    }
    return;
  }
  if (lane == 0) {
    ExtRec o;
    o.score = best; o.i_end = bi; o.j_end = bj; o.d_last = d_last;
    o.live = tot; o.path = 0; o.flags = FZ_FLAG_DONE | FZ_FLAG_WIDE; o.npath = 0;
    o.m = m; o.n = n; o.width = (uint32_t)((wbest + 31) & ~31); o.ckpt = 0;
    *R = o;
    atomicAdd(wa.live_total, (unsigned long long)tot);
  }
}

template <bool TRACE>
__global__ void __launch_bounds__(WW * 32) k_wide(Params p, WorkArgs wa) {
  __shared__ int32_t s_sub[16];
  if (threadIdx.x < 16) s_sub[threadIdx.x] = p.sub[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t gw = (uint64_t)blockIdx.x * WW + warp;
  int32_t* buf = wa.scratch + gw * wa.scratch_stride;
  const int32_t cap = (int32_t)(wa.scratch_stride / 9);
  for (;;) {
    uint32_t idx = 0;
    if (lane == 0) idx = atomicAdd(wa.counter, 1u);
    idx = __shfl_sync(FULL, idx, 0);
    const uint32_t nw = TRACE ? wa.n_work : *wa.wide_count;
    if (idx >= nw) break;
    if (TRACE) {
      // executor segment (wide-band extensions have only the origin segment)
      const uint4 sg = wa.seg[idx];
      const uint32_t ext = wa.list[sg.x];
      if (!(wa.rec[ext].flags & FZ_FLAG_WIDE)) continue;
      wide_ext<TRACE>(p, wa, ext, sg.x, lane, buf, cap, s_sub);
    } else {
      wide_ext<TRACE>(p, wa, wa.list[idx], idx, lane, buf, cap, s_sub);
    }
  }
}

}  // namespace

uint64_t wide_scratch_elems(int32_t max_len) { return 9ull * (uint64_t)(max_len + 1); }
int wide_warps_per_block() { return WW; }

cudaError_t launch_inspect_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  k_wide<false><<<grid, WW * 32, 0, st>>>(p, wa);
  return cudaGetLastError();
}

cudaError_t launch_execute_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  k_wide<true><<<grid, WW * 32, 0, st>>>(p, wa);
  return cudaGetLastError();
}

}  // namespace fz
