// General-band anti-diagonal sweep (sm_103a): the path for extensions whose
// live band outgrows the register windows (very large ydrop, long gapped
// regions), and for every extension when the scores do not fit the byte forms.
//
// One block (CTA) per extension.  Each anti-diagonal's candidate band [lo, hi]
// (rows with a live predecessor on one of the two previous anti-diagonals) is
// cut into 32-row strips, dealt round-robin to the block's warps (FastZ
// section 3.2: strips of an anti-diagonal computed side by side, the strip
// boundaries exchanged through memory).  A cell reads its three predecessors
// from the last two anti-diagonals, which the block keeps in a shared-memory
// ring indexed by target row modulo the ring size; the anti-diagonal's
// maximum (earliest row on ties) and live range are combined across the warps
// once per anti-diagonal, in the same barrier that publishes its cells.  When
// a band is wider than the ring, the two anti-diagonals still read move to a
// per-block global scratch indexed by row and the sweep continues there, with
// all three buffers in it.  Liveness
// follows the y-drop rule as written: dead cells hold NEG in S, I and D.
// With windows of up to SB_MAX_LEN bases the block also stages both windows'
// bases in shared memory (2 bits each, 16 to a word, loaded once per
// extension), so a cell reads its two bases there instead of from global
// memory.
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int CW = 8;               // warps per block
constexpr int CT = CW * 32;         // threads per block
constexpr int RING_MAX = 2048;      // rows of the shared-memory ring at most
constexpr int32_t SB_MAX_LEN = 4080;  // windows staged in shared memory up to this length (3 blocks per SM)

// Words of staged bases per window (window positions 0 .. max_len, 16 to a word).
__host__ __device__ inline int32_t sb_words(int32_t max_len) { return max_len / 16 + 1; }

// Ring rows for windows of up to max_len rows: a power of two holding a whole
// window when it fits RING_MAX.
__host__ __device__ inline int32_t ring_rows(int32_t max_len) {
  int32_t c = 64;
  while (c < max_len + 1 && c < RING_MAX) c <<= 1;
  return c;
}

__device__ __forceinline__ uint32_t base_at(const uint8_t* __restrict__ s, uint64_t len, int64_t g0, int dir,
                                            int64_t w) {
  const int64_t g = g0 + dir * w;
  if (g < 0 || (uint64_t)g >= len) return 0u;
  return ((uint32_t)__ldg(s + (g >> 2)) >> ((g & 3) * 2)) & 3u;
}

// Candidate band of an anti-diagonal already computed: the rows written
// [blo, bhi] (dead ones hold NEG), the live rows [llo, lhi], and which of the
// three buffers holds it.
struct Band {
  int32_t blo, bhi, llo, lhi;
  int k;
};

// Sweep state shared by every thread of the block (each keeps its own copy;
// all copies follow the same block-wide values).
struct WideState {
  Band b1, b2;                      // anti-diagonals dn - 1 and dn - 2
  int32_t dn;                       // next anti-diagonal
  int32_t best, bi, bj, d_last, wrun, wbest;
};

// Buffer k's component c (0 S, 1 I, 2 D) at row i: buf[(3 k + c) stride + (i & mask)].
template <bool SMEM>
struct Bufs {
  int32_t* buf;
  int32_t stride, mask;
  __device__ __forceinline__ int32_t* at(int k, int c, int32_t i) const {
    return buf + (3 * k + c) * stride + (i & mask);
  }
};

// Anti-diagonals from s.dn on, until the sweep ends (true) or, in the ring, a
// band wider than the ring (false: s.dn is the anti-diagonal still to do).
template <bool TRACE, bool SMEM, bool SB>
__device__ bool wide_run(const Params& p, const Window& w, WideState& s, const Bufs<SMEM>& B, int32_t ring,
                         int32_t d_stop, uint32_t W, uint8_t* tbase, int32_t* lo_arr, const int32_t* s_sub,
                         const uint32_t* sb_t, const uint32_t* sb_q, int4 (*red)[CW], uint32_t& cnt, int tid,
                         int warp, int lane) {
  const int32_t m = w.m, n = w.n, oe = p.oe, e = p.e;
  for (; s.dn <= m + n; ++s.dn) {
    const int32_t dn = s.dn;
    if (dn > d_stop) return true;
    const Band& b1 = s.b1;
    const Band& b2 = s.b2;
    int32_t lo = 0x7fffffff, hi = -0x7fffffff;
    if (b1.lhi >= b1.llo) { lo = b1.llo; hi = b1.lhi + 1; }
    if (b2.lhi >= b2.llo) { lo = imin(lo, b2.llo + 1); hi = imax(hi, b2.lhi + 1); }
    lo = imax(lo, imax(0, dn - n));
    hi = imin(hi, imin(m, dn));
    if (lo > hi) return true;
    if (SMEM && hi - lo + 1 > ring) return false;
    const int kc = 3 - b1.k - b2.k;
    const int32_t T = threshold(s.best, p.ydrop);
    int32_t mx = NEG, mi = 0x7fffffff, a_lo = 0x7fffffff, a_hi = -1;
    // (the strip loop's bound is uniform within a warp, so every lane takes
    // part in the shuffle that pairs trace codes)
    for (int32_t c = lo + 32 * warp; c <= hi; c += CT) {
      const int32_t i = c + lane;
      const bool act = i <= hi;
      const int32_t j = dn - i;
      int32_t sl = NEG, il = NEG, su = NEG, du = NEG, sd = NEG;
      if (act) {
        if (j >= 1 && i >= b1.blo && i <= b1.bhi) { sl = *B.at(b1.k, 0, i); il = *B.at(b1.k, 1, i); }
        if (i >= 1 && i - 1 >= b1.blo && i - 1 <= b1.bhi) { su = *B.at(b1.k, 0, i - 1); du = *B.at(b1.k, 2, i - 1); }
        if (i >= 1 && j >= 1 && i - 1 >= b2.blo && i - 1 <= b2.bhi) sd = *B.at(b2.k, 0, i - 1);
      }
      const int32_t Iv = j >= 1 ? imax(il - e, sl - oe) : NEG;
      const int32_t Dv = i >= 1 ? imax(du - e, su - oe) : NEG;
      int32_t G = NEG;
      if (act && i >= 1 && j >= 1) {
        const uint32_t tb = SB ? (sb_t[i >> 4] >> (2 * (i & 15))) & 3u : base_at(p.t2, p.t_len, w.tg0, w.dir, i);
        const uint32_t qb = SB ? (sb_q[j >> 4] >> (2 * (j & 15))) & 3u : base_at(p.q2, p.q_len, w.qg0, w.dir, j);
        G = sd + s_sub[tb * 4 + qb];
      }
      const int32_t S = imax(G, imax(Iv, Dv));
      const bool alive = act && S >= T;
      if (act) {
        *B.at(kc, 0, i) = alive ? S : NEG;
        *B.at(kc, 1, i) = alive ? Iv : NEG;
        *B.at(kc, 2, i) = alive ? Dv : NEG;
      }
      if (alive) {
        ++cnt;
        if (S > mx) { mx = S; mi = i; }
        a_lo = imin(a_lo, i);
        a_hi = imax(a_hi, i);
      }
      if (TRACE) {
        // rows lo + 2u and lo + 2u + 1 sit in lanes of the same warp (strips
        // start at lo + 32 k)
        const uint32_t code = (G == S ? 0u : (Iv == S ? 1u : 2u)) | (j >= 1 && Iv == sl - oe ? 4u : 0u) |
                              (i >= 1 && Dv == su - oe ? 8u : 0u);
        const uint32_t hi4 = __shfl_down_sync(FULL, code, 1);
        const uint32_t u = (uint32_t)(i - lo);
        if (act && !(lane & 1) && u < W) tbase[(uint64_t)dn * (W / 2) + (u >> 1)] = (uint8_t)(code | (hi4 << 4));
      }
    }
    {
      const int32_t wm = __reduce_max_sync(FULL, mx);
      const uint32_t wi = __reduce_min_sync(FULL, (mx == wm && mx != NEG) ? (uint32_t)mi : 0xffffffffu);
      const uint32_t wlo = __reduce_min_sync(FULL, (uint32_t)a_lo);
      const int32_t whi = (int32_t)__reduce_max_sync(FULL, (uint32_t)(a_hi + 1)) - 1;
      if (lane == 0) red[dn & 1][warp] = make_int4(wm, (int32_t)wi, (int32_t)wlo, whi);
    }
    // publishes this anti-diagonal's cells and the warps' partial results
    // (red alternates by parity: a warp writing anti-diagonal dn + 1's entry
    // cannot overwrite one that a slower warp is still reading)
    __syncthreads();
    int32_t wm = NEG, nlo = 0x7fffffff, nhi = -1;
    uint32_t wi = 0xffffffffu;
#pragma unroll
    for (int k = 0; k < CW; ++k) {
      const int4 r = red[dn & 1][k];
      if (r.x > wm) { wm = r.x; wi = (uint32_t)r.y; }
      else if (r.x == wm && (uint32_t)r.y < wi) wi = (uint32_t)r.y;
      nlo = imin(nlo, r.z);
      nhi = imax(nhi, r.w);
    }
    s.b2 = s.b1;
    s.b1 = Band{lo, hi, nlo, nhi, kc};
    s.wrun = imax(s.wrun, hi - lo + 1);
    if (wm != NEG) {
      s.d_last = dn;
      if (wm > s.best) { s.best = wm; s.bi = (int32_t)wi; s.bj = dn - s.bi; s.wbest = s.wrun; }
    }
    if (TRACE && tid == 0) lo_arr[dn] = lo;
  }
  return true;
}

template <bool TRACE, bool SB>
__device__ void wide_ext(const Params& p, const WorkArgs& wa, uint32_t ext, uint32_t idx, int tid, int32_t* ring_buf,
                         int32_t ring, int32_t* gbuf, int32_t cap, const int32_t* s_sub, uint32_t* sb_t, uint32_t* sb_q,
                         int4 (*red)[CW], unsigned long long* s_sum) {
  const int warp = tid >> 5, lane = tid & 31;
  const Window w = make_window(p, ext);
  ExtRec* R = wa.rec + ext;
  if (!w.requested) {
    if (!TRACE && tid == 0) {
      ExtRec z = {};
      *R = z;
    }
    return;
  }
  int32_t d_stop = 0x7fffffff;
  uint32_t W = 0;
  uint8_t* tbase = nullptr;
  int32_t* lo_arr = nullptr;
  if (TRACE) {
    d_stop = R->i_end + R->j_end;
    W = R->width;
    tbase = wa.trace + (wa.trace_off[idx] - wa.trace_sub);
    lo_arr = reinterpret_cast<int32_t*>(tbase + trace_lo_offset(W, d_stop));
    if (tid == 0) lo_arr[0] = 0;
  }
  // anti-diagonal 0: the origin alone, S = 0
  WideState s;
  s.b1 = Band{0, 0, 0, 0, 0};
  s.b2 = Band{1, 0, 1, 0, 2};
  s.dn = 1;
  s.best = 0; s.bi = 0; s.bj = 0; s.d_last = 0; s.wrun = 1; s.wbest = 1;
  uint32_t cnt = tid == 0 ? 1u : 0u;
  const Bufs<true> RB{ring_buf, ring, ring - 1};
  if (tid == 0) { *RB.at(0, 0, 0) = 0; *RB.at(0, 1, 0) = NEG; *RB.at(0, 2, 0) = NEG; }
  if (SB) {
    // word k: window positions 16 k .. 16 k + 15 (row or column i at bits 2 (i % 16))
    for (int32_t k = tid; k <= w.m / 16; k += CT) sb_t[k] = fetch16(p.t2, p.t_len, w.tg0, w.dir, 16 * (int64_t)k);
    for (int32_t k = tid; k <= w.n / 16; k += CT) sb_q[k] = fetch16(p.q2, p.q_len, w.qg0, w.dir, 16 * (int64_t)k);
  }
  __syncthreads();
  if (!wide_run<TRACE, true, SB>(p, w, s, RB, ring, d_stop, W, tbase, lo_arr, s_sub, sb_t, sb_q, red, cnt, tid,
                                 warp, lane)) {
    // the band outgrew the ring: move the two previous anti-diagonals (the
    // only ones still read) to the global scratch, rows at their own index
    const Bufs<false> GB{gbuf, cap, 0x7fffffff};
    const Band bs[2] = {s.b1, s.b2};
    for (int q = 0; q < 2; ++q)
      for (int32_t i = bs[q].blo + tid; i <= bs[q].bhi; i += CT)
#pragma unroll
        for (int c = 0; c < 3; ++c) *GB.at(bs[q].k, c, i) = *RB.at(bs[q].k, c, i);
    __syncthreads();
    wide_run<TRACE, false, SB>(p, w, s, GB, cap, d_stop, W, tbase, lo_arr, s_sub, sb_t, sb_q, red, cnt, tid, warp,
                               lane);
  }
  // live cells: warp sums, then thread 0 adds the warps' (the barrier also
  // ends every read of the ring before the next extension writes it)
  const unsigned long long ws = __reduce_add_sync(FULL, cnt);
  if (lane == 0) s_sum[warp] = ws;
  __syncthreads();
  if (tid == 0) {
    unsigned long long tot = 0;
    for (int k = 0; k < CW; ++k) tot += s_sum[k];
    if (TRACE) {
      atomicAdd(wa.exec_total, tot);
      atomicAdd(wa.exec_live, tot);
    } else {
      ExtRec o;
      o.score = s.best; o.i_end = s.bi; o.j_end = s.bj; o.d_last = s.d_last;
      o.live = tot; o.path = 0; o.flags = FZ_FLAG_DONE | FZ_FLAG_WIDE; o.npath = 0;
      o.m = w.m; o.n = w.n; o.width = (uint32_t)((s.wbest + 31) & ~31); o.ckpt = 0;
      *R = o;
      atomicAdd(wa.live_total, tot);
    }
  }
  __syncthreads();   // (s_sum is rewritten by the next extension)
}

template <bool TRACE, bool SB>
__global__ void __launch_bounds__(CT) k_wide(Params p, WorkArgs wa) {
  // dynamic shared memory: 9 x ring rows (S, I, D of three anti-diagonals),
  // then (SB) the target window's and the query window's staged bases
  extern __shared__ int32_t s_ring[];
  __shared__ int32_t s_sub[16];
  __shared__ int4 s_red[2][CW];
  __shared__ unsigned long long s_sum[CW];
  __shared__ uint32_t s_idx;
  const int tid = threadIdx.x;
  if (tid < 16) s_sub[tid] = p.sub[tid];
  const int32_t ring = ring_rows(p.max_len);
  uint32_t* sb_t = reinterpret_cast<uint32_t*>(s_ring + 9 * ring);
  uint32_t* sb_q = sb_t + sb_words(p.max_len);
  int32_t* gbuf = wa.scratch + (uint64_t)blockIdx.x * wa.scratch_stride;
  const int32_t cap = (int32_t)(wa.scratch_stride / 9);
  for (;;) {
    if (tid == 0) s_idx = atomicAdd(wa.counter, 1u);
    __syncthreads();
    const uint32_t idx = s_idx;
    __syncthreads();                               // (s_idx is rewritten next round)
    const uint32_t nw = TRACE ? wa.n_work : *wa.wide_count;
    if (idx >= nw) break;
    if (TRACE) {
      // executor segment (wide-band extensions have only the origin segment)
      const uint4 sg = wa.seg[idx];
      const uint32_t ext = wa.list[sg.x];
      if (!(wa.rec[ext].flags & FZ_FLAG_WIDE)) continue;
      wide_ext<TRACE, SB>(p, wa, ext, sg.x, tid, s_ring, ring, gbuf, cap, s_sub, sb_t, sb_q, s_red, s_sum);
    } else {
      wide_ext<TRACE, SB>(p, wa, wa.list[idx], idx, tid, s_ring, ring, gbuf, cap, s_sub, sb_t, sb_q, s_red, s_sum);
    }
  }
}

size_t ring_bytes(int32_t max_len) { return (size_t)9 * ring_rows(max_len) * sizeof(int32_t); }

bool staged(int32_t max_len) { return max_len <= SB_MAX_LEN; }

// Dynamic shared memory of a launch: the ring, and the staged bases when the
// windows are short enough.
size_t wide_smem(int32_t max_len) {
  return ring_bytes(max_len) + (staged(max_len) ? 2 * (size_t)sb_words(max_len) * sizeof(uint32_t) : 0);
}

const void* kernel_of(bool trace, bool sb) {
  if (trace) return sb ? reinterpret_cast<const void*>(k_wide<true, true>) : reinterpret_cast<const void*>(k_wide<true, false>);
  return sb ? reinterpret_cast<const void*>(k_wide<false, true>) : reinterpret_cast<const void*>(k_wide<false, false>);
}

}  // namespace

uint64_t wide_scratch_elems(int32_t max_len) { return 9ull * (uint64_t)(max_len + 1); }

int wide_blocks_per_sm(int32_t max_len) {
  // every variant may take the largest dynamic shared memory, so that
  // contexts with other window caps can launch too
  const int limit = (int)(ring_bytes(RING_MAX) + 2 * (size_t)sb_words(SB_MAX_LEN) * sizeof(uint32_t));
  for (int t = 0; t < 2; ++t)
    for (int b = 0; b < 2; ++b)
      if (cudaFuncSetAttribute(kernel_of(t, b), cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess)
        return 0;
  int best = 0;
  for (int t = 0; t < 2; ++t) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel_of(t, staged(max_len)), CT, wide_smem(max_len)) !=
        cudaSuccess)
      return 0;
    best = t ? (nb < best ? nb : best) : nb;
  }
  return best;
}

cudaError_t launch_inspect_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  if (staged(p.max_len)) k_wide<false, true><<<grid, CT, wide_smem(p.max_len), st>>>(p, wa);
  else k_wide<false, false><<<grid, CT, wide_smem(p.max_len), st>>>(p, wa);
  return cudaGetLastError();
}

cudaError_t launch_execute_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  if (staged(p.max_len)) k_wide<true, true><<<grid, CT, wide_smem(p.max_len), st>>>(p, wa);
  else k_wide<true, false><<<grid, CT, wide_smem(p.max_len), st>>>(p, wa);
  return cudaGetLastError();
}

}  // namespace fz
