// Register-window anti-diagonal sweep: inspector and executor (sm_103a).
//
// One warp owns one extension at a time.  Lane l holds K consecutive rows of
// the current anti-diagonal, rows b + l*K .. b + l*K + K-1 (a 32*K-row window
// with base b), with per row: h = S - o - e of the current anti-diagonal, h of
// the previous one (diagonal source), I, D, the substitution row of its
// target base and the query selector of its column.  Stepping d -> d+1 either
// keeps the base (rows gain one query column; data of the row above comes
// from lane l-1 by shuffle) or moves it up by one row once row b is dead (the
// row above each row is then the same slot of the previous step; data of the
// row below comes from lane l+1).  Only the window's edges exchange values,
// three shuffles per step, so scores never leave registers (FastZ section
// 3.2's use-and-discard ring, in the anti-diagonal layout of its section 2.2).
//
// Y-drop: a cell is live when S >= best - ydrop, best being the maximum over
// completed anti-diagonals (kept in a warp-uniform register after a warp max
// reduction per step).  Only S is cleared on a pruned cell: I and D of a dead
// cell are below the threshold and can never make a later cell live, and no
// traceback path goes through them, so scores, ends and paths are those of
// the strict recurrence.
//
// The executor is the same sweep stopped at the inspector's best cell's
// anti-diagonal; it replays every threshold and window decision and stores a
// 4-bit direction code per cell (FastZ section 3.1.3 stores the S/I/D choices
// in 2+1+1 bits).
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int WARPS = 4;

struct Reservoir {          // warp-uniform stream of bases
  uint32_t cur;             // the next bases, 2 bits each, below a marker bit
  uint32_t nxt;             // the 16 bases after them (prefetched)
  int64_t next;             // window index of the first base after nxt's 15
};

// cur holds 15 bases and a marker bit above them; when only the marker is
// left the next 15 come from nxt, and nxt is fetched again.
__device__ __forceinline__ void res_init(Reservoir& r, const uint8_t* s, uint64_t len, int64_t g0, int dir,
                                         int64_t first) {
  r.cur = (fetch16(s, len, g0, dir, first) & 0x3fffffffu) | 0x40000000u;
  r.nxt = fetch16(s, len, g0, dir, first + 15);
  r.next = first + 30;
}

__device__ __forceinline__ uint32_t res_take(Reservoir& r, const uint8_t* s, uint64_t len, int64_t g0, int dir) {
  const uint32_t nx = __umulhi(r.cur, 1u << 30);              // cur >> 2 and
  const uint32_t b = (uint32_t)imad((int32_t)nx, -4, (int32_t)r.cur);   // cur & 3, on the FMA pipe
  r.cur = nx;
  if (r.cur == 1u) {
    r.cur = (r.nxt & 0x3fffffffu) | 0x40000000u;
    r.nxt = fetch16(s, len, g0, dir, r.next);
    r.next += 15;
  }
  return b;
}

// Eager traceback inside the 16x16 corner (FastZ section 3.1.2): recompute
// cells (i, j), i, j <= 16, with the sweep's thresholds, lane = row, then walk
// back from (bi, bj).  Returns the walk as 2-bit ops, first op = last column.
__device__ __noinline__ void eager_corner(const Params& p, const Window& w, int lane, const int32_t* sT,
                             uint8_t* tile, const int32_t* s_sub, int32_t bi, int32_t bj,
                             uint64_t& path, uint32_t& npath, uint32_t* err) {
  const int32_t dstar = bi + bj;
  const int i = lane;
  const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, 1);
  const uint32_t qw = fetch16(p.q2, p.q_len, w.qg0, w.dir, 1);
  const int tb = i >= 1 ? (int)((tw >> (2 * ((i - 1) & 15))) & 3u) : 0;
  const int32_t oe = p.oe, e = p.e;
  int32_t Sp = i == 0 ? 0 : NEG, Ip = NEG, Dp = NEG, Spp = NEG;
  for (int d = 1; d <= dstar; ++d) {
    const int j = d - i;
    int32_t su = __shfl_up_sync(FULL, Sp, 1);
    int32_t du = __shfl_up_sync(FULL, Dp, 1);
    int32_t sd = __shfl_up_sync(FULL, Spp, 1);
    if (lane == 0) { su = NEG; du = NEG; sd = NEG; }
    const int32_t Ic = j >= 1 ? imax(Ip - e, Sp - oe) : NEG;
    const int32_t Dc = i >= 1 ? imax(du - e, su - oe) : NEG;
    int32_t G = NEG;
    if (i >= 1 && j >= 1 && j <= EAGER_N) G = sd + s_sub[tb * 4 + (int)((qw >> (2 * (j - 1))) & 3u)];
    const int32_t S = imax(G, imax(Ic, Dc));
    const bool valid = j >= 0 && j <= w.n && i <= w.m && i <= EAGER_N && j <= EAGER_N;
    const bool alive = valid && S >= sT[d];
    if (valid) {
      const uint32_t sc = G == S ? 0u : (Ic == S ? 1u : 2u);
      const uint32_t io = (j >= 1 && Ic == Sp - oe) ? 4u : 0u;
      const uint32_t dop = (i >= 1 && Dc == su - oe) ? 8u : 0u;
      tile[i * (EAGER_N + 1) + j] = (uint8_t)(sc | io | dop);
    }
    Spp = Sp;
    Sp = alive ? S : NEG;
    Ip = alive ? Ic : NEG;
    Dp = alive ? Dc : NEG;
  }
  __syncwarp();
  uint64_t code = 0;
  uint32_t k = 0;
  if (lane == 0) {
    int ci = bi, cj = bj, st = 0;
    int guard = 4 * EAGER_N + 4;
    while ((ci > 0 || cj > 0) && k < 2 * EAGER_N && --guard > 0) {
      const uint32_t c = tile[ci * (EAGER_N + 1) + cj];
      if (st == 0) {
        const uint32_t sc = c & 3u;
        if (sc == 0 && ci > 0 && cj > 0) { ++k; --ci; --cj; }   // op M = 0
        else if (sc == 1 && cj > 0) st = 1;
        else if (sc == 2 && ci > 0) st = 2;
        else { atomicOr(err, 8u); break; }
      } else if (st == 1) {
        if (cj <= 0) { atomicOr(err, 8u); break; }
        code |= 1ull << (2 * k); ++k;
        st = (c & 4u) ? 0 : 1;
        --cj;
      } else {
        if (ci <= 0) { atomicOr(err, 8u); break; }
        code |= 2ull << (2 * k); ++k;
        st = (c & 8u) ? 0 : 2;
        --ci;
      }
    }
  }
  path = __shfl_sync(FULL, code, 0);
  npath = __shfl_sync(FULL, k, 0);
  __syncwarp();
}

// Register state of one lane: up to KS consecutive rows of the window.
template <int KS>
struct LaneState {
  int32_t H[KS], HP[KS], I[KS], D[KS];
  uint32_t MR[KS];
  uint32_t QP[KS / 2];
};

struct StepIn {
  int32_t Th;          // threshold on h = S - o - e for the new anti-diagonal
  int32_t vhi, vlo;    // edge mode: slot r is inside the window iff vlo <= r <= vhi
  int32_t oe, ne, c1;
  int32_t one;         // 1 (Params::one)
  uint32_t qb;         // NOSHIFT: query base entering lane 0
  uint32_t mr_new;     // SHIFT: substitution row entering lane 31
};

// Direction code of a cell, added into nibble r of the lane's codes: bits 0-1
// the source of S (0 diagonal, 1 I, 2 D, in that order of preference; from the
// DPX predicates, cell_max), bit 2
// set when I opens from h on the left, bit 3 when D opens from h above.  I >= h
// and D >= h_up always, so "opens" is "h - I is not negative": the sign bit of
// h - I, taken with a high multiply, is the complement of bit 2 (likewise for
// D).  The nibble is then 12 + S choice - 4 (I extends) - 8 (D extends), added
// with multiply-adds into two 32-bit words (rows 0-7 and 8-15); the caller
// starts both words at 12 in every nibble it stores, so each nibble's sum is
// its code in 0..15 and the words hold the codes once all rows are added.
template <int KA>
__device__ __forceinline__ void packed_code(uint32_t (&packed)[2], int r, uint32_t sc, int32_t Ic, int32_t Dc,
                                            int32_t hl, int32_t hu, int32_t one) {
  // (one is a runtime 1: the products stay multiply-adds on the FMA pipe)
  const uint32_t ie = __umulhi((uint32_t)imad(Ic, -one, hl), 2u);     // I extends
  const uint32_t de = __umulhi((uint32_t)imad(Dc, -one, hu), 2u);     // D extends
  const uint32_t nib = (uint32_t)imad((int32_t)de, -8, imad((int32_t)ie, -4, (int32_t)sc));
  packed[r >> 3] = (uint32_t)imad((int32_t)nib, (int32_t)(1u << (4 * (r & 7))), (int32_t)packed[r >> 3]);
}

// S of a cell and, for the executor, the source of S as the DPX predicates
// give it: __vibmax_s32(a, b, &p) returns max(a, b) with p = (a >= b) (a wins
// a tie; measured on the GB300), so the diagonal wins over I and D and I over
// D, the traceback's order of preference.  sc: 0 diagonal, 1 I, 2 D.
template <bool TRACE>
__device__ __forceinline__ int32_t cell_max(int32_t G, int32_t Ic, int32_t Dc, uint32_t& sc) {
  if (!TRACE) return __vimax3_s32(G, Ic, Dc);
  bool i_over_d, diag;
  const int32_t id = __vibmax_s32(Ic, Dc, &i_over_d);
  const int32_t S = __vibmax_s32(G, id, &diag);
  sc = diag ? 0u : (i_over_d ? 1u : 2u);
  return S;
}

// Word w of a lane's packed codes before any row is added: 12 in each of the
// nibbles the lane stores (rows 0..KA-1).
template <int KA>
__host__ __device__ constexpr uint32_t packed_base(int w) {
  return (KA >= 8 * (w + 1)) ? 0xccccccccu : (KA <= 8 * w ? 0u : (0xccccccccu >> (32 - 4 * (KA - 8 * w))));
}

// One anti-diagonal step over the first KA slots of every lane (a 32*KA-row
// window).  Returns the lane max of the pruned h; cnt counts live cells;
// packed receives the direction codes in TRACE mode.
template <int KS, int KA, bool TRACE, bool SHIFT, bool EDGE>
__device__ __forceinline__ int32_t step(LaneState<KS>& L, const StepIn& in, int lane, uint32_t& cnt,
                                        uint32_t (&packed)[2]) {
  static_assert(KA <= KS && KA % 2 == 0, "active slots");
  constexpr int KH = KA / 2;
  int32_t lm = NEG;
  if (!SHIFT) {
    const int32_t dtop = __viaddmax_s32(L.D[KA - 1], in.ne, L.H[KA - 1]);
    int32_t dc_top = __shfl_up_sync(FULL, dtop, 1);
    int32_t hp_top = __shfl_up_sync(FULL, L.HP[KA - 1], 1);
    uint32_t qs_top = __shfl_up_sync(FULL, __umulhi(L.QP[KH - 1], 65536u), 1);
    int32_t hu_top = 0;
    if (TRACE) hu_top = __shfl_up_sync(FULL, L.H[KA - 1], 1);
    if (lane == 0) { dc_top = NEG; hp_top = NEG; qs_top = 0x4440u | in.qb; hu_top = NEG; }
#pragma unroll
    for (int k = KH - 1; k >= 1; --k) L.QP[k] = __funnelshift_l(L.QP[k - 1], L.QP[k], 16);
    L.QP[0] = (L.QP[0] << 16) | qs_top;
#pragma unroll
    for (int r = KA - 1; r >= 0; --r) {
      const int32_t hl = L.H[r];
      const int32_t Ic = __viaddmax_s32(L.I[r], in.ne, hl);
      const int32_t Dc = r ? __viaddmax_s32(L.D[r - 1], in.ne, L.H[r - 1]) : dc_top;
      const int32_t hp = r ? L.HP[r - 1] : hp_top;
      const uint32_t sel = (r & 1) ? __umulhi(L.QP[r >> 1], 65536u) : L.QP[r >> 1];
      const int32_t G = imad((int32_t)prmt(L.MR[r], 0u, sel), in.one, hp);   // hp carries + o + e - 128
      uint32_t sc = 0;
      const int32_t S = cell_max<TRACE>(G, Ic, Dc, sc);
      const int32_t hn = imad(S, in.one, -in.oe);
      bool alive = hn >= in.Th;
      if (EDGE) alive = alive && r <= in.vhi && r >= in.vlo;
      if (TRACE) {
        const int32_t hu = r ? L.H[r - 1] : hu_top;
        packed_code<KA>(packed, r, sc, Ic, Dc, hl, hu, in.one);
      }
      L.HP[r] = imad(hl, in.one, in.c1);   // next step's diagonal source, offset by o + e - 128
      L.H[r] = alive ? hn : NEG;
      L.I[r] = Ic;
      L.D[r] = Dc;
      if ((r & 1) == 0) lm = __vimax3_s32(lm, L.H[r], L.H[r + 1]);   // rows r, r+1 are both new
      cnt += alive ? 1u : 0u;
    }
  } else {
    const int32_t itop = __viaddmax_s32(L.I[0], in.ne, L.H[0]);
    int32_t ic_top = __shfl_down_sync(FULL, itop, 1);
    int32_t h_top = __shfl_down_sync(FULL, L.H[0], 1);
    uint32_t mr_top = __shfl_down_sync(FULL, L.MR[0], 1);
    if (lane == 31) { ic_top = NEG; h_top = NEG; mr_top = in.mr_new; }
#pragma unroll
    for (int r = 0; r < KA - 1; ++r) L.MR[r] = L.MR[r + 1];
    L.MR[KA - 1] = mr_top;
#pragma unroll
    for (int r = 0; r < KA; ++r) {
      const int32_t hl = r < KA - 1 ? L.H[r + 1] : h_top;
      const int32_t Ic = r < KA - 1 ? __viaddmax_s32(L.I[r + 1], in.ne, L.H[r + 1]) : ic_top;
      const int32_t hu = L.H[r];
      const int32_t Dc = __viaddmax_s32(L.D[r], in.ne, hu);
      const int32_t hp = L.HP[r];
      const uint32_t sel = (r & 1) ? __umulhi(L.QP[r >> 1], 65536u) : L.QP[r >> 1];
      const int32_t G = imad((int32_t)prmt(L.MR[r], 0u, sel), in.one, hp);   // hp carries + o + e - 128
      uint32_t sc = 0;
      const int32_t S = cell_max<TRACE>(G, Ic, Dc, sc);
      const int32_t hn = imad(S, in.one, -in.oe);
      bool alive = hn >= in.Th;
      if (EDGE) alive = alive && r <= in.vhi && r >= in.vlo;
      if (TRACE) packed_code<KA>(packed, r, sc, Ic, Dc, hl, hu, in.one);
      L.HP[r] = imad(hl, in.one, in.c1);
      L.H[r] = alive ? hn : NEG;
      L.I[r] = Ic;
      L.D[r] = Dc;
      if (r & 1) lm = __vimax3_s32(lm, L.H[r - 1], L.H[r]);           // rows r-1, r are both new
      cnt += alive ? 1u : 0u;
    }
  }
  return lm;
}

// Lane l's KA direction codes of one anti-diagonal: nibbles l*KA .. l*KA+KA-1
// of the row (KA/2 bytes; 16-bit stores when they stay aligned).
template <int KA>
__device__ __forceinline__ void store_codes(uint8_t* row, int lane, const uint32_t (&pk)[2]) {
  const uint64_t packed = ((uint64_t)pk[1] << 32) | pk[0];
  uint8_t* dst = row + lane * (KA / 2);
  if (KA % 4 == 0) {
#pragma unroll
    for (int k = 0; k < KA / 4; ++k) reinterpret_cast<uint16_t*>(dst)[k] = (uint16_t)(packed >> (16 * k));
  } else {
#pragma unroll
    for (int k = 0; k < KA / 2; ++k) dst[k] = (uint8_t)(packed >> (8 * k));
  }
}

// Per-warp shared buffer used to re-lay the window out when its size changes.
template <int KS>
struct Relay {
  int32_t H[32 * KS], HP[32 * KS], I[32 * KS], D[32 * KS];
  uint8_t t[32 * KS], q[32 * KS];
};

// Changing the window from kold to knew active slots per lane keeps its base
// row b: row b+u moves from lane u/kold, slot u%kold to lane u/knew, slot
// u%knew, through the per-warp shared buffer.  relay_store writes the rows
// out; relay_load reads rows 0 .. rows_old-1 back (rows that did not exist
// before are dead; their target bases and query bases, column d - row, are
// read from memory).  When shrinking the caller guarantees the dropped rows
// are dead.  A checkpoint restore stages its rows with ck_stage and then
// takes the same relay_load.
template <int KS>
__device__ __forceinline__ void relay_store(const LaneState<KS>& L, int kold, int lane, Relay<KS>* rb,
                                            const uint32_t* s_mrow) {
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    if (r < kold) {
      const int u = lane * kold + r;
      rb->H[u] = L.H[r];
      rb->HP[u] = L.HP[r];
      rb->I[u] = L.I[r];
      rb->D[u] = L.D[r];
      uint32_t t = 0;
      for (uint32_t k = 3; k > 0; --k) t = (s_mrow[k] == L.MR[r]) ? k : t;   // base whose row this is
      if (s_mrow[0] == L.MR[r]) t = 0;
      rb->t[u] = (uint8_t)t;
      rb->q[u] = (uint8_t)(((r & 1) ? (L.QP[r >> 1] >> 16) : L.QP[r >> 1]) & 3u);
    }
  }
  __syncwarp();
}

template <int KS>
__device__ __forceinline__ void relay_load(LaneState<KS>& L, int rows_old, int knew, int32_t b, int32_t d,
                                           int lane, Relay<KS>* rb, const Params& p, const Window& w,
                                           const uint32_t* s_mrow) {
  const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)b + (int64_t)lane * knew);
  const uint32_t qw = fetch16(p.q2, p.q_len, w.qg0, w.dir, (int64_t)d - b - (int64_t)lane * knew - 15);
  uint32_t sel[KS];
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    sel[r] = 0x4440u;
    if (r < knew) {
      const int u = lane * knew + r;
      if (u < rows_old) {
        L.H[r] = rb->H[u];
        L.HP[r] = rb->HP[u];
        L.I[r] = rb->I[u];
        L.D[r] = rb->D[u];
        L.MR[r] = s_mrow[rb->t[u]];
        sel[r] = 0x4440u | rb->q[u];
      } else {
        L.H[r] = NEG; L.HP[r] = NEG; L.I[r] = NEG; L.D[r] = NEG;
        L.MR[r] = s_mrow[(tw >> (2 * r)) & 3u];
        sel[r] = 0x4440u | ((qw >> (2 * (15 - r))) & 3u);   // column d - (b + u)
      }
    }
  }
#pragma unroll
  for (int k = 0; k < KS / 2; ++k) L.QP[k] = sel[2 * k] | (sel[2 * k + 1] << 16);
  __syncwarp();
}

// ---- window checkpoints (layout in fz_dev.cuh) ----

// Sweep state after anti-diagonal d kept in a checkpoint header.
struct CkScalars {
  int32_t b, d, best, bi, bj, d_last;
};

// Writes the state after anti-diagonal d (all KS slots of every lane) to a new
// slot linked to `head`; returns the new head (slot + 1), or `head` unchanged
// when the pool is full.  cnt: this lane's live cells so far (lane 0 adds
// 2^32 cnt_hi).
template <int KS>
__device__ __forceinline__ uint32_t ck_write(const WorkArgs& wa, const LaneState<KS>& L, int lane, uint32_t head,
                                             const CkScalars& cs, uint32_t cnt, uint32_t cnt_hi,
                                             const int32_t* sT) {
  uint32_t slot = 0;
  if (lane == 0) slot = atomicAdd(wa.ckpt_used, 1u);
  slot = __shfl_sync(FULL, slot, 0);
  if (slot >= wa.ckpt_cap) return head;
  int32_t* c = wa.ckpt + (uint64_t)slot * CK_SLOT_WORDS;
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    c[CK_HDR + r * 32 + lane] = L.H[r];
    c[CK_HDR + CK_WIN_MAX + r * 32 + lane] = L.HP[r];
    c[CK_HDR + 2 * CK_WIN_MAX + r * 32 + lane] = L.I[r];
    c[CK_HDR + 3 * CK_WIN_MAX + r * 32 + lane] = L.D[r];
  }
  c[CK_T + lane] = sT[lane];
  c[CK_CNT + lane] = (int32_t)cnt;
  if (lane == 0) {
    c[CK_T + 32] = sT[32];
    c[CK_D] = cs.d; c[CK_B] = cs.b; c[CK_K] = KS; c[CK_BEST] = cs.best; c[CK_BI] = cs.bi; c[CK_BJ] = cs.bj;
    c[CK_DLAST] = cs.d_last; c[CK_FLAGS] = 0; c[CK_PREV] = (int32_t)head;
    c[CK_CNT_HI] = (int32_t)cnt_hi;
  }
  return slot + 1;
}

// Loads a checkpoint into a KS-row-per-lane window (KS >= the writer's K; rows
// the writer did not hold are dead) and rebuilds each row's substitution row
// and query selector from the sequences: row b + u has target base b + u and
// sits at column d - (b + u).
template <int KS>
__device__ __forceinline__ void ck_load(LaneState<KS>& L, const int32_t* c, int lane, const Params& p,
                                        const Window& w, const uint32_t* s_mrow, CkScalars& cs) {
  cs.b = c[CK_B]; cs.d = c[CK_D]; cs.best = c[CK_BEST]; cs.bi = c[CK_BI]; cs.bj = c[CK_BJ];
  cs.d_last = c[CK_DLAST];
  const int ks = c[CK_K];
  const int rows_src = 32 * ks;
  const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)cs.b + (int64_t)lane * KS);
  const uint32_t qw = fetch16(p.q2, p.q_len, w.qg0, w.dir, (int64_t)cs.d - cs.b - (int64_t)lane * KS - 15);
  uint32_t sel[KS];
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    const int u = lane * KS + r;
    L.H[r] = NEG; L.HP[r] = NEG; L.I[r] = NEG; L.D[r] = NEG;
    if (u < rows_src) {
      const int sl = u / ks, sr = u - sl * ks;
      const int pos = sr * 32 + sl;
      L.H[r] = c[CK_HDR + pos];
      L.HP[r] = c[CK_HDR + CK_WIN_MAX + pos];
      L.I[r] = c[CK_HDR + 2 * CK_WIN_MAX + pos];
      L.D[r] = c[CK_HDR + 3 * CK_WIN_MAX + pos];
    }
    L.MR[r] = s_mrow[(tw >> (2 * r)) & 3u];
    sel[r] = 0x4440u | ((qw >> (2 * (15 - r))) & 3u);
  }
#pragma unroll
  for (int k = 0; k < KS / 2; ++k) L.QP[k] = sel[2 * k] | (sel[2 * k + 1] << 16);
}

// Lanes whose rows hold a live cell at d (from h) and at d - 1 (from the
// previous anti-diagonal's h, kept offset by o + e - 128: dead is near NEG).
template <int KS>
__device__ __forceinline__ void ck_live_lanes(const LaneState<KS>& L, uint32_t& now, uint32_t& prev) {
  bool a = false, q = false;
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    a = a || L.H[r] > NEG / 2;
    q = q || L.HP[r] > NEG / 2;
  }
  now = __ballot_sync(FULL, a);
  prev = __ballot_sync(FULL, q);
}

// Stages a checkpoint's rows in the relay buffer for relay_load, with each
// row's target base and query base (column d - row), and returns the live row
// bounds at d (from h) and d - 1 (from the previous anti-diagonal's h, kept
// offset by o + e - 128: dead is near NEG) as absolute rows, or NOROW values.
template <int KS>
__device__ __forceinline__ int ck_stage(Relay<KS>* rb, const int32_t* c, int lane, const Params& p, const Window& w,
                                        int32_t& hi_c, int32_t& lo_c, int32_t& hi_p, int32_t& lo_p) {
  constexpr int32_t NOROW_HI = -0x3fffffff, NOROW_LO = 0x3fffffff;
  const int32_t b = c[CK_B], d = c[CK_D];
  const int ks = c[CK_K];
  const int rows = imin(32 * ks, 32 * KS);
  const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)b + 16 * lane);
  const uint32_t qw = fetch16(p.q2, p.q_len, w.qg0, w.dir, (int64_t)d - b - 16 * lane - 15);
  int32_t hc = NOROW_HI, lc = NOROW_LO, hp = NOROW_HI, lp = NOROW_LO;
#pragma unroll 4
  for (int k = 0; k < 16; ++k) {
    const int u = 16 * lane + k;
    if (u < rows) {
      const int sl = u / ks, pos = (u - sl * ks) * 32 + sl;
      const int32_t h = c[CK_HDR + pos], hq = c[CK_HDR + CK_WIN_MAX + pos];
      rb->H[u] = h;
      rb->HP[u] = hq;
      rb->I[u] = c[CK_HDR + 2 * CK_WIN_MAX + pos];
      rb->D[u] = c[CK_HDR + 3 * CK_WIN_MAX + pos];
      rb->t[u] = (uint8_t)((tw >> (2 * k)) & 3u);
      rb->q[u] = (uint8_t)((qw >> (2 * (15 - k))) & 3u);
      if (h > NEG / 2) { hc = imax(hc, b + u); lc = imin(lc, b + u); }
      if (hq > NEG / 2) { hp = imax(hp, b + u); lp = imin(lp, b + u); }
    }
  }
  hi_c = __reduce_max_sync(FULL, hc);
  lo_c = __reduce_min_sync(FULL, lc);
  hi_p = __reduce_max_sync(FULL, hp);
  lo_p = __reduce_min_sync(FULL, lp);
  __syncwarp();
  return rows;
}

// ---- executor: the replay with a lean step loop per window size ----
//
// A segment replays the inspector's sweep from the origin or from a
// checkpoint up to d_stop with KA active rows per lane.  The step loop for one
// KA carries only what the replay needs: the threshold (from the best score),
// row b's liveness and the top lane's; it leaves when the segment ends or when
// the band may reach past the top of the KA-row window, and the caller re-lays
// the window out two rows per lane wider.
//
// Away from the window's edges and while the top lane is dead the steps run
// in fixed pairs, a step that keeps the base and then one that moves it up
// when row b is dead, as in the inspector's pair sweep (one register layout
// per pair instead of a join of two every step).  The base then may trail the
// shift-by-one base, but only while row b is dead; a step that keeps the base
// with the top lane live is taken alone, and only when row b is live, so the
// base is the shift-by-one base there.  A window of KS rows per lane never
// needs to grow: keeping the base with row b live leaves the window at or
// above the inspector's window of the next anti-diagonal (the inspector's base
// never passes the shift-by-one base either), which held every live cell.
struct ExecState {
  int32_t b, d, best, T;
  uint32_t cnt;              // live cells this lane replayed
  bool rowb_alive, top, top_prev;
  Reservoir qr, tr;
};

// One replay step to anti-diagonal s.d + 1 and its bookkeeping.
template <int KS, int KA, bool SHIFT, bool EDGE>
__device__ __forceinline__ void exec_step(LaneState<KS>& L, ExecState& s, StepIn& in, const Params& p,
                                          const Window& w, int lane, const uint32_t* s_mrow, uint8_t* tbase,
                                          int32_t* lo_arr) {
  constexpr int32_t WMAX = 32 * KS;
  const int32_t dn = s.d + 1;
  const int32_t bn = s.b + (SHIFT ? 1 : 0);
  in.Th = s.T - in.oe;
  uint32_t packed[2] = {packed_base<KA>(0), packed_base<KA>(1)};
  if (EDGE) {
    const int32_t rowbase = bn + lane * KA;
    in.vhi = w.m - rowbase;
    in.vlo = dn - w.n - rowbase;
  }
  if (!SHIFT) in.qb = res_take(s.qr, p.q2, p.q_len, w.qg0, w.dir);
  else in.mr_new = s_mrow[res_take(s.tr, p.t2, p.t_len, w.tg0, w.dir)];
  const int32_t lm = step<KS, KA, true, SHIFT, EDGE>(L, in, lane, s.cnt, packed);
  store_codes<KA>(tbase + (uint64_t)dn * (WMAX / 2), lane, packed);
  const int32_t wm = __reduce_max_sync(FULL, lm);
  const bool edge_lane = (lane == 0 && L.H[0] >= in.Th) || (lane == 31 && lm >= in.Th);
  const uint32_t bits = __ballot_sync(FULL, edge_lane);
  if (wm + in.oe > s.best) {                       // the replay needs only the threshold
    s.best = wm + in.oe;
    s.T = threshold(s.best, p.ydrop);
  }
  if (lane == 0) lo_arr[dn] = bn;
  s.rowb_alive = bits & 1u;
  s.top_prev = s.top && !SHIFT;
  s.top = (bits >> 31) != 0u;
  s.b = bn;
  s.d = dn;
}

template <int KS, int KA>
__device__ __forceinline__ bool exec_loop(LaneState<KS>& L, ExecState& s, StepIn& in, const Params& p,
                                          const Window& w, int lane, const uint32_t* s_mrow, uint8_t* tbase,
                                          int32_t* lo_arr, int32_t d_stop) {
  constexpr int32_t WIN = 32 * KA;
  const int32_t m = w.m, n = w.n;
  for (;;) {
    if (s.d >= d_stop) return false;
    // steps that cannot touch the window's edges (the base grows by at most
    // one row per step)
    const int32_t d_fast = imin(d_stop, s.d + imin(m - WIN - s.b, s.b - s.d + n));
    if (d_fast > s.d && !s.top && !s.top_prev) {
      for (;;) {
        exec_step<KS, KA, false, false>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr);
        if (s.rowb_alive || s.d == d_fast) break;
        exec_step<KS, KA, true, false>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr);
        if (s.top || s.d == d_fast) break;
      }
      continue;
    }
    // one step of the shift-by-one rule, with edge masks
    const bool shift = !s.rowb_alive;
    if (KA < KS && !shift && (s.top || s.top_prev) && s.b + WIN <= m) return true;   // grow
    if (!shift) exec_step<KS, KA, false, true>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr);
    else exec_step<KS, KA, true, true>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr);
  }
}

template <int KS>
__device__ void run_exec(const Params& p, const WorkArgs& wa, uint32_t ext, uint4 sg, int lane,
                         const uint32_t* s_mrow, Relay<KS>* rb) {
  static_assert(KS % 2 == 0 && KS <= 16, "one 16-base fetch per lane");
  constexpr int32_t WMAX = 32 * KS;
  const Window w = make_window(p, ext);
  const ExtRec* R = wa.rec + ext;
  if (!w.requested) return;
  const int32_t dstar = R->i_end + R->j_end;
  const int32_t d_stop = (int32_t)sg.z;
  uint8_t* tbase = wa.trace + (wa.trace_off[sg.x] - wa.trace_sub);
  int32_t* lo_arr = reinterpret_cast<int32_t*>(tbase + trace_lo_offset(WMAX, dstar));
  StepIn in;
  in.oe = p.oe;
  in.ne = -p.e;
  in.c1 = p.oe - 128;
  in.one = p.one;
  ExecState s;
  LaneState<KS> L;
  int ka = 4;
  if (sg.y == 0u) {
    // origin: 4 rows per lane to start with
    const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)lane * 4);
#pragma unroll
    for (int r = 0; r < KS; ++r) {
      L.MR[r] = s_mrow[r < 4 ? (tw >> (2 * r)) & 3u : 0u];
      L.H[r] = NEG; L.HP[r] = NEG; L.I[r] = NEG; L.D[r] = NEG;
    }
#pragma unroll
    for (int k = 0; k < KS / 2; ++k) L.QP[k] = 0x44404440u;
    if (lane == 0) L.H[0] = -p.oe;                   // origin: S(0,0) = 0
    if (lane == 0) lo_arr[0] = 0;
    s.b = 0; s.d = 0; s.best = 0;
    s.rowb_alive = true;
  } else {
    // checkpoint: the smallest window (even rows per lane, at least 4) whose
    // top lane holds no live cell of the last two anti-diagonals
    const int32_t* c = wa.ckpt + (uint64_t)(sg.y - 1u) * CK_SLOT_WORDS;
    int32_t hi_c, lo_c, hi_p, lo_p;
    const int rows = ck_stage<KS>(rb, c, lane, p, w, hi_c, lo_c, hi_p, lo_p);
    s.b = c[CK_B]; s.d = c[CK_D]; s.best = c[CK_BEST];
    const int32_t span = imax(hi_c, hi_p) - s.b;     // highest live row above the base
    while (ka < KS && 31 * ka <= span) ka += 2;
    relay_load<KS>(L, rows, ka, s.b, s.d, lane, rb, p, w, s_mrow);
    s.rowb_alive = lo_c == s.b;
  }
  s.T = threshold(s.best, p.ydrop);
  s.cnt = 0;
  s.top = false;
  s.top_prev = false;
  res_init(s.qr, p.q2, p.q_len, w.qg0, w.dir, (int64_t)s.d + 1 - s.b);   // query columns entering at row b
  res_init(s.tr, p.t2, p.t_len, w.tg0, w.dir, (int64_t)s.b + 32 * ka);  // target rows entering at the top
  for (;;) {
    bool grow;
    switch (ka) {
      case 4: grow = exec_loop<KS, 4>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      case 6: grow = exec_loop<KS, 6>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      case 8: grow = exec_loop<KS, 8>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      case 10: grow = exec_loop<KS, 10>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      case 12: grow = exec_loop<KS, (KS >= 12 ? 12 : KS)>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      case 14: grow = exec_loop<KS, (KS >= 14 ? 14 : KS)>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
      default: grow = exec_loop<KS, KS>(L, s, in, p, w, lane, s_mrow, tbase, lo_arr, d_stop); break;
    }
    if (!grow) break;
    // two more rows per lane: the old top lane's rows move down, lane 31's are new and dead
    relay_store<KS>(L, ka, lane, rb, s_mrow);
    relay_load<KS>(L, 32 * ka, ka + 2, s.b, s.d, lane, rb, p, w, s_mrow);
    ka += 2;
    res_init(s.tr, p.t2, p.t_len, w.tg0, w.dir, (int64_t)s.b + 32 * ka);
    s.top = false;
    s.top_prev = false;
  }
  uint64_t tot = s.cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  if (lane == 0) {
    atomicAdd(wa.exec_total, (unsigned long long)(d_stop - (int32_t)sg.w) * (unsigned long long)WMAX);
    atomicAdd(wa.exec_live, (unsigned long long)tot);
  }
}

// Inspector sweep with a fixed window of KS rows per lane.  The loop keeps
// only what the inspector needs per step:
//   * overflow: the top lane held a live cell at d or d-1 and the base stays;
//   * edge mode whenever rows beyond m or columns beyond n exist inside the
//     window (then every cell checks its bounds);
//   * liveness of the anti-diagonal from its maximum, row b's liveness and the
//     top lane's from one ballot;
//   * the threshold, recomputed only when the best score changes.
template <int KS>
__device__ void run_inspect(const Params& p, const WorkArgs& wa, uint32_t ext, int lane, int32_t* sT,
                            uint8_t* tile, const uint32_t* s_mrow, const int32_t* s_sub) {
  static_assert(KS % 2 == 0 && KS <= 16, "one 16-base fetch per lane");
  constexpr int32_t WIN = 32 * KS;
  const Window w = make_window(p, ext);
  ExtRec* R = wa.rec + ext;
  if (!w.requested) {
    if (lane == 0) {
      ExtRec z = {};
      *R = z;
    }
    return;
  }
  const int32_t m = w.m, n = w.n, oe = p.oe, mn = w.m + w.n;
  uint32_t cnt_hi_carry = 0;   // high word of a live count carried from a checkpoint
  LaneState<KS> L;
  {
    const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)lane * KS);
#pragma unroll
    for (int r = 0; r < KS; ++r) {
      L.MR[r] = s_mrow[(tw >> (2 * r)) & 3u];
      L.H[r] = NEG; L.HP[r] = NEG; L.I[r] = NEG; L.D[r] = NEG;
    }
#pragma unroll
    for (int k = 0; k < KS / 2; ++k) L.QP[k] = 0x44404440u;
    if (lane == 0) L.H[0] = -oe;                       // origin: S(0,0) = 0
  }
  int32_t b = 0, d = 0, best = 0, bi = 0, bj = 0, d_last = 0;
  bool live_prev = true, rowb_alive = true, top = false, top_prev = false;
  uint32_t cnt = lane == 0 ? 1u : 0u;
  // resume (the widest window, after an overflow): continue from the newest checkpoint
  uint32_t head = KS >= 16 && wa.resume && wa.ckpt ? R->ckpt : 0u;
  if constexpr (KS >= 16) if (head) {
    const int32_t* c = wa.ckpt + (uint64_t)(head - 1) * CK_SLOT_WORDS;
    CkScalars cs;
    ck_load<KS>(L, c, lane, p, w, s_mrow, cs);
    b = cs.b; d = cs.d; best = cs.best; bi = cs.bi; bj = cs.bj; d_last = cs.d_last;
    cnt = (uint32_t)c[CK_CNT + lane];
    if (lane == 0) cnt_hi_carry = (uint32_t)c[CK_CNT_HI];
    sT[lane] = c[CK_T + lane];
    if (lane == 0) sT[32] = c[CK_T + 32];
    uint32_t now, prev;
    ck_live_lanes<KS>(L, now, prev);
    live_prev = now != 0u;                          // the loop's live_prev is the live flag of d
    rowb_alive = __shfl_sync(FULL, L.H[0] > NEG / 2 ? 1 : 0, 0) != 0;
    top = (now >> 31) != 0u;
    top_prev = (prev >> 31) != 0u;                  // conservative: may only add an overflow
    __syncwarp();
  }
  if (!head) {
    // sT[d], d <= 32: the best score when it rose at anti-diagonal d (NEG: it
    // did not); the eager corner's thresholds are rebuilt from these
    sT[lane] = NEG;
    if (lane == 0) sT[32] = NEG;
    __syncwarp();
  }
  Reservoir qr, tr;
  res_init(qr, p.q2, p.q_len, w.qg0, w.dir, (int64_t)d + 1 - b);   // query columns entering at row b
  res_init(tr, p.t2, p.t_len, w.tg0, w.dir, (int64_t)b + WIN);     // target rows entering at the window top

  StepIn in;
  in.oe = oe;
  in.ne = -p.e;
  in.c1 = oe - 128;
  in.one = p.one;
  in.Th = threshold(best, p.ydrop) - oe;
  bool overflow = false;
  uint32_t no_codes[2] = {0u, 0u};   // direction codes are the executor's
  const uint32_t ck_mask = wa.ckpt ? (uint32_t)wa.ckpt_every - 1u : 0xffffffffu;

  // The step loop leaves at the end of the sweep, on an overflow, and at every
  // checkpoint boundary; the checkpoint writes stay out of the step loop.
  // Exits are tested once per step, after it, for the next step: the end of
  // the sweep (two empty anti-diagonals, or the window's last one), an
  // overflow (the base stays and the top lane is or was live), and every
  // checkpoint boundary; the checkpoint writes stay out of the step loop.
  int why = d + 1 > mn ? 2 : ((rowb_alive && (top || top_prev) && b + WIN <= m) ? 1 : 0);   // 0 boundary, 1 overflow, 2 end
  if (why == 0) {
    for (;;) {
      for (;;) {
        const int32_t dn = d + 1;
        const bool shift = !rowb_alive;
        const int32_t bn = b + (shift ? 1 : 0);
        const bool edge = bn + WIN - 1 > m || bn < dn - n;
        int32_t lm;
        if (!shift) {
          in.qb = res_take(qr, p.q2, p.q_len, w.qg0, w.dir);
          if (edge) {
            const int32_t rowbase = bn + lane * KS;
            in.vhi = m - rowbase;
            in.vlo = dn - n - rowbase;
            lm = step<KS, KS, false, false, true>(L, in, lane, cnt, no_codes);
          } else {
            lm = step<KS, KS, false, false, false>(L, in, lane, cnt, no_codes);
          }
        } else {
          in.mr_new = s_mrow[res_take(tr, p.t2, p.t_len, w.tg0, w.dir)];
          if (edge) {
            const int32_t rowbase = bn + lane * KS;
            in.vhi = m - rowbase;
            in.vlo = dn - n - rowbase;
            lm = step<KS, KS, false, true, true>(L, in, lane, cnt, no_codes);
          } else {
            lm = step<KS, KS, false, true, false>(L, in, lane, cnt, no_codes);
          }
        }
        const int32_t wm = __reduce_max_sync(FULL, lm);
        const bool edge_lane = (lane == 0 && L.H[0] >= in.Th) || (lane == 31 && lm >= in.Th);
        const uint32_t bits = __ballot_sync(FULL, edge_lane);
        const bool live = wm >= in.Th;
        if (wm + oe > best) {                                // implies live
          int rf = KS;
#pragma unroll
          for (int r = KS - 1; r >= 0; --r) rf = (L.H[r] == wm) ? r : rf;
          const uint32_t fm = __ballot_sync(FULL, rf < KS);
          const int Ln = __ffs(fm) - 1;
          const int rr = __shfl_sync(FULL, rf, Ln);
          bi = bn + Ln * KS + rr;
          bj = dn - bi;
          best = wm + oe;
          in.Th = threshold(best, p.ydrop) - oe;
          if (dn <= 2 * EAGER_N && lane == 0) sT[dn] = best;   // eager corner thresholds come from these
        }
        d_last = live ? dn : d_last;
        rowb_alive = bits & 1u;
        top_prev = top && !shift;      // the old top row is still the top row only if the base stayed
        top = (bits >> 31) != 0u;
        b = bn;
        d = dn;
        const bool end_ = (!live && !live_prev) || d + 1 > mn;
        live_prev = live;
        // (no overflow once the window reaches row m: no row lies beyond it)
        const bool ovf = rowb_alive && (top || top_prev) && b + WIN <= m;
        if (end_ || ovf || ((uint32_t)d & ck_mask) == 0u) {
          why = end_ ? 2 : (ovf ? 1 : 0);
          break;
        }
      }
      if (why != 0) break;
      // periodic checkpoint while the best cell is recent: executor segments
      // start from these
      if (d - (bi + bj) <= wa.ckpt_recent) {
        const CkScalars cs{b, d, best, bi, bj, d_last};
        head = ck_write<KS>(wa, L, lane, head, cs, cnt, cnt_hi_carry, sT);
      }
    }
  }
  if (why == 1) {
    overflow = true;   // the live band may grow past the window top
    if (wa.ckpt) {     // the wider window resumes here
      const CkScalars cs{b, d, best, bi, bj, d_last};
      head = ck_write<KS>(wa, L, lane, head, cs, cnt, cnt_hi_carry, sT);
    }
  }

  uint64_t tot = cnt;
  if (lane == 0) tot += (uint64_t)cnt_hi_carry << 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  if (overflow) {
    if (lane == 0) {
      ExtRec z = {};
      z.flags = FZ_FLAG_DONE | FZ_FLAG_WIDE;
      z.m = m;
      z.n = n;
      z.ckpt = head;
      *R = z;
      const uint32_t slot = atomicAdd(wa.ovf_count, 1u);   // retried with a wider window
      wa.ovf_list[slot] = ext;
    }
    return;
  }
  uint64_t path = 0;
  uint32_t npath = 0;
  uint32_t flags = FZ_FLAG_DONE;
  uint32_t width = WIN;
  if (bi <= EAGER_N && bj <= EAGER_N) {
    flags |= FZ_FLAG_EAGER;
    width = 0;
    if (bi + bj > 0) {
      // thresholds of anti-diagonals 1..32: from the best score over the
      // anti-diagonals before each (the origin scores 0)
      int32_t v = sT[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) v = imax(v, __shfl_up_sync(FULL, v, o));
      v = imax(v, 0);                                  // best over anti-diagonals 0 .. lane
      __syncwarp();
      sT[lane + 1] = threshold(v, p.ydrop);            // lane 31 writes sT[32]
      __syncwarp();
      eager_corner(p, w, lane, sT, tile, s_sub, bi, bj, path, npath, wa.err);
    }
  }
  if (lane == 0) {
    ExtRec o;
    o.score = best; o.i_end = bi; o.j_end = bj; o.d_last = d_last;
    o.live = tot; o.path = path; o.flags = flags; o.npath = npath;
    o.m = m; o.n = n; o.width = width; o.ckpt = head;
    *R = o;
    atomicAdd(wa.live_total, (unsigned long long)tot);
  }
}

// ---- 16-bit pair sweep: the first tier when scores fit (Params::pair_ok) ----
//
// The same 384-row window and steps as run_inspect<12>, with two rows in each
// 32-bit register as 16-bit values, so that every DPX instruction (the s16x2
// forms) advances two cells.  Values are stored relative to a base
// B = T - PMG, T being the prune threshold of the anti-diagonal being
// computed, and clamped at 0 (the relu forms):
//   * a live cell has S >= T, so its stored h = S - o - e - B >= PMG - o - e;
//     a pruned cell stores 0;
//   * any value below T acts like a dead one: a live cell's maximum comes from
//     a term at or above T, and a term of 0 (or a clamped one) stays below
//     T - (o + e + max M) > 0, so a dead cell never makes a later one live;
//   * when the best score rises, T rises by the same amount; the rise is kept
//     in the stored threshold until it passes the slack of the 16-bit range,
//     then every stored value moves down by it (clamped at 0).
// Stored values stay below ydrop + PMG + slack + 2 max|M| < 2^15 (checked when
// the context is created).  Results, live counts and checkpoints are those of the
// 32-bit sweep: checkpoints are written in its layout, so the 512-row tier and
// the executor resume from them unchanged.
constexpr int PK = K_TIER0 / 2;   // register pairs per lane at most (12 rows, a 384-row window)
constexpr int NP_SMALL = 4;       // pairs per lane of the small window (8 rows, 256 rows)
constexpr int32_t PMG = 2048;

// With NP active pairs (2 NP rows per lane), register p < NP of a lane holds
// its rows p (low half) and p + NP (high half).  The row above a pair is then
// the previous pair (both halves), so a step reads its neighbours without
// moving halves; only pair 0 combines the row above the lane (lane l-1's row
// 2 NP - 1) with the lane's own row NP - 1.
struct PairState {
  uint32_t H[PK];     // h = S - o - e
  uint32_t HP[PK];    // h of the previous anti-diagonal + (o + e): the diagonal source
  uint32_t I[PK], D[PK];
  uint32_t MR[2 * PK];  // substitution row of each row's target base (signed bytes), by row
  uint32_t SEL[PK];     // byte-permute selector: sign-extended scores of both rows' query bases
};

// Selector bytes of a row's query base q: as the low row of a pair (bytes q
// and sign of byte q of the first operand) and as the high row (bytes 4+q and
// its sign, second operand).
__device__ __forceinline__ uint32_t sel_lo(uint32_t q) { return 0x80u + 17u * q; }
__device__ __forceinline__ uint32_t sel_hi(uint32_t q) { return 0xc4u + 17u * q; }

__device__ __forceinline__ uint32_t lo16(uint32_t x) { return x & 0xffffu; }
__device__ __forceinline__ uint32_t hi16(uint32_t x) { return x >> 16; }
__device__ __forceinline__ uint32_t dup16(int32_t v) { return ((uint32_t)v & 0xffffu) * 0x10001u; }
template <int NP>
__device__ __forceinline__ uint32_t prow(const uint32_t (&X)[PK], int r) {
  return r < NP ? lo16(X[r]) : hi16(X[r - NP]);
}

// Live mask of a pair of new h values.  hn = S - (o + e) comes from a packed
// add, so a half lies in [-(o + e), 2^15) (two's complement); hn + lb2 as a
// packed add (lb2 = 0x8000 - threshold in both halves, 0 < threshold <= 8192 +
// 2048) sets bit 15 of a half exactly when 0 <= hn and hn >= threshold: a
// negative half wraps to 0x8000 - |hn| - threshold, below 0x8000.  The
// sign-replicating byte permute spreads that bit over the half.
__device__ __forceinline__ uint32_t live_mask(uint32_t hn, uint32_t lb2) { return prmt(__vadd2(hn, lb2), 0u, 0xbb99u); }

// Live cells from a sum of live masks (0xffff per live low half, 0xffff0000
// per live high half, mod 2^32): with n_lo, n_hi < 2^15 the low 16 bits give
// -n_lo and the rest n_lo - n_hi.
__device__ __forceinline__ uint32_t live_count(uint32_t s) {
  const uint32_t nlo = (0x10000u - (s & 0xffffu)) & 0xffffu;
  const int32_t diff = (int32_t)(int16_t)(uint16_t)((s + nlo) >> 16);
  return 2u * nlo - (uint32_t)diff;
}

// Lane max and live-mask sum over the pairs of a step, two pairs at a time
// (a 3-way max and a 3-input add).  q counts the pairs in the order they are
// computed: an even one is held back for the next, an odd one folds both,
// and with an odd count the last folds alone.
__device__ __forceinline__ void fold2(int q, bool last, uint32_t h, uint32_t live, uint32_t& hk,
                                      uint32_t& lk, uint32_t& lm2, uint32_t& live2) {
  if (q & 1) {
    live2 = live2 + lk + live;
    lm2 = q == 1 ? __vmaxs2(hk, h) : __vimax3_s16x2(lm2, hk, h);
  } else if (last) {
    live2 += live;
    lm2 = q == 0 ? h : __vmaxs2(lm2, h);
  } else {
    hk = h;
    lk = live;
  }
}

// Traced pair sweep: the four direction flags of both cells of pair p, from
// packed differences whose sign bit (bit 15 of a half) is the flag:
//   nd = g - S   < 0: S does not come from the diagonal
//   ni = I - S   < 0: S does not come from I (when not from the diagonal; a
//                     tie with D goes to I)
//   ie = hl - I  < 0: I extends (I > h of the cell to the left; a tie opens)
//   de = hu - D  < 0: D extends (D > h of the cell above; a tie opens)
// S >= g, I, D, I >= hl and D >= hu, and every value lies in (-2^15, 2^15)
// (g may be negative in lane 0's bottom row, which has no row above it), so
// each difference lies in (-2^15, 0] and its sign is exact.  The packed
// subtractions issue on the FMA pipe, which the DPX maxima, byte permutes and
// logic ops of the cell leave less busy than the ALU pipe.  Two
// sign-replicating byte permutes turn the four words into bytes of 0 or 0xff,
// and two logic ops with a per-pair mask place them: acc[p / 4] byte 0 holds
// (nd, ie) of the low-half cell (row p) at bits 7 - 2 (p % 4) and
// 6 - 2 (p % 4), byte 1 its (ni, de), bytes 2 and 3 the same for the
// high-half cell (row p + NP).  (p is a constant once the caller's pair loop
// is unrolled.)
__device__ __forceinline__ void pair_flags(uint32_t (&acc)[2], int p, uint32_t g, uint32_t sv, uint32_t ic,
                                           uint32_t hl, uint32_t dc, uint32_t hu) {
  const uint32_t w1 = prmt(__vsub2(g, sv), __vsub2(ic, sv), 0xfbd9u);
  const uint32_t w2 = prmt(__vsub2(hl, ic), __vsub2(hu, dc), 0xfbd9u);
  const int q = p & 3;
  acc[p >> 2] |= (w1 & (0x80808080u >> (2 * q))) | (w2 & (0x40404040u >> (2 * q)));
}

// One step of the pair sweep with NP active pairs; returns the pair-wise max
// of the new h (both halves); live2 accumulates the live masks; with TR, acc
// receives the direction flags of every cell (pair_flags).
template <int NP, bool SHIFT, bool EDGE, bool TR>
__device__ __forceinline__ uint32_t pstep(PairState& L, uint32_t ne2, uint32_t noe2, uint32_t oe2, uint32_t lb2,
                                          int lane, uint32_t qb, uint32_t mr_new, int32_t vlo, int32_t vhi,
                                          uint32_t& live2, uint32_t (&acc)[2]) {
  uint32_t lm2 = 0, hk = 0, lk = 0;
  if (!SHIFT) {
    // above pair 0 (rows -1 and NP-1): lane l-1's row 2NP-1 (high half of its
    // pair NP-1) and the lane's own row NP-1
    const uint32_t hu = __shfl_up_sync(FULL, L.H[NP - 1], 1);
    const uint32_t du = __shfl_up_sync(FULL, L.D[NP - 1], 1);
    const uint32_t pu = __shfl_up_sync(FULL, L.HP[NP - 1], 1);
    uint32_t su = __shfl_up_sync(FULL, L.SEL[NP - 1], 1);
    if (lane == 0) su = sel_hi(qb) << 8;                            // row b's new column
    // The shuffled high half under the own low half; lane 0 has no row
    // above row b and takes the sign of its own byte 1 instead: 0 for h and
    // D (below 2^15), 0 or -1 for the diagonal source, which then stays far
    // below any live value like a dead cell's.
    const uint32_t fs = lane == 0 ? 0x54ddu : 0x5432u;
    const uint32_t ha0 = prmt(hu, L.H[NP - 1], fs);
    const uint32_t da0 = prmt(du, L.D[NP - 1], fs);
    const uint32_t pa0 = prmt(pu, L.HP[NP - 1], fs);
    const uint32_t sel0 = prmt(su, L.SEL[NP - 1], 0x0041u) + 0x43bcu;   // query roles swap halves
#pragma unroll
    for (int p = NP - 1; p >= 0; --p) {
      const uint32_t ha = p ? L.H[p - 1] : ha0;
      const uint32_t da = p ? L.D[p - 1] : da0;
      const uint32_t pa = p ? L.HP[p - 1] : pa0;
      const uint32_t sel = p ? L.SEL[p - 1] : sel0;               // each row takes the next query base
      const uint32_t ic = __viaddmax_s16x2_relu(L.I[p], ne2, L.H[p]);
      const uint32_t dc = __viaddmax_s16x2_relu(da, ne2, ha);
      const uint32_t g = __vadd2(pa, prmt(L.MR[p], L.MR[p + NP], sel));
      const uint32_t sv = __vimax3_s16x2_relu(g, ic, dc);
      if (TR) pair_flags(acc, p, g, sv, ic, L.H[p], dc, ha);
      const uint32_t hn = __vadd2(sv, noe2);          // a dead half may go negative: live_mask
      uint32_t live = live_mask(hn, lb2);
      if (EDGE) {
        live &= ((p >= vlo && p <= vhi) ? 0xffffu : 0u) | ((p + NP >= vlo && p + NP <= vhi) ? 0xffff0000u : 0u);
      }
      const uint32_t h = hn & live;
      L.HP[p] = L.H[p] + oe2;                                       // no carry: h + o + e < 2^16
      L.H[p] = h;
      L.I[p] = ic;
      L.D[p] = dc;
      L.SEL[p] = sel;
      fold2(NP - 1 - p, p == 0, h, live, hk, lk, lm2, live2);
    }
  } else {
    // the base moves up a row: new row r is old row r + 1; new row 2NP-1 is
    // lane l+1's old row 0 (low half of its pair 0)
    const uint32_t hd = __shfl_down_sync(FULL, L.H[0], 1);
    const uint32_t id = __shfl_down_sync(FULL, L.I[0], 1);
    uint32_t md = __shfl_down_sync(FULL, L.MR[0], 1);
    if (lane == 31) md = mr_new;
    // old rows NP and 2NP; lane 31's row 2NP lies above the window: the sign
    // of its own byte 1 (h and I are below 2^15) makes it dead
    const uint32_t fs = lane == 31 ? 0x9932u : 0x5432u;
    const uint32_t hol = prmt(L.H[0], hd, fs);
    const uint32_t iol = prmt(L.I[0], id, fs);
#pragma unroll
    for (int r = 0; r < 2 * NP - 1; ++r) L.MR[r] = L.MR[r + 1];
    L.MR[2 * NP - 1] = md;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const uint32_t ho = p < NP - 1 ? L.H[p + 1] : hol;            // the row itself, one step back
      const uint32_t io = p < NP - 1 ? L.I[p + 1] : iol;
      const uint32_t ic = __viaddmax_s16x2_relu(io, ne2, ho);
      const uint32_t dc = __viaddmax_s16x2_relu(L.D[p], ne2, L.H[p]);
      const uint32_t g = __vadd2(L.HP[p], prmt(L.MR[p], L.MR[p + NP], L.SEL[p]));
      const uint32_t sv = __vimax3_s16x2_relu(g, ic, dc);
      if (TR) pair_flags(acc, p, g, sv, ic, ho, dc, L.H[p]);
      const uint32_t hn = __vadd2(sv, noe2);          // a dead half may go negative: live_mask
      uint32_t live = live_mask(hn, lb2);
      if (EDGE) {
        live &= ((p >= vlo && p <= vhi) ? 0xffffu : 0u) | ((p + NP >= vlo && p + NP <= vhi) ? 0xffff0000u : 0u);
      }
      const uint32_t h = hn & live;
      L.HP[p] = ho + oe2;
      L.H[p] = h;
      L.I[p] = ic;
      L.D[p] = dc;
      fold2(p, p == NP - 1, h, live, hk, lk, lm2, live2);
    }
  }
  return lm2;
}

// Checkpoint of the pair sweep after anti-diagonal d, in the 32-bit layout
// (rows u = K lane + r, K = 2 NP): h and I, D back in score space, dead as NEG.
template <int NP>
__device__ __forceinline__ void ck_fill_pair(int32_t* c, const PairState& L, int lane, uint32_t head,
                                             const CkScalars& cs, int32_t B, int32_t oe, uint32_t cnt,
                                             uint32_t cnt_hi, const int32_t* sT) {
  const int32_t c1 = oe - 128;
#pragma unroll
  for (int r = 0; r < 2 * NP; ++r) {
    const uint32_t h = prow<NP>(L.H, r);
    const uint32_t hp = prow<NP>(L.HP, r);
    const uint32_t iv = prow<NP>(L.I, r);
    const uint32_t dv = prow<NP>(L.D, r);
    c[CK_HDR + r * 32 + lane] = h ? (int32_t)h + B : NEG;
    c[CK_HDR + CK_WIN_MAX + r * 32 + lane] = ((int32_t)hp > oe ? (int32_t)hp - oe + B : NEG) + c1;
    c[CK_HDR + 2 * CK_WIN_MAX + r * 32 + lane] = iv ? (int32_t)iv + B : NEG;
    c[CK_HDR + 3 * CK_WIN_MAX + r * 32 + lane] = dv ? (int32_t)dv + B : NEG;
  }
  c[CK_T + lane] = sT[lane];
  c[CK_CNT + lane] = (int32_t)cnt;
  if (lane == 0) {
    c[CK_T + 32] = sT[32];
    c[CK_D] = cs.d; c[CK_B] = cs.b; c[CK_K] = 2 * NP; c[CK_BEST] = cs.best; c[CK_BI] = cs.bi; c[CK_BJ] = cs.bj;
    c[CK_DLAST] = cs.d_last; c[CK_FLAGS] = 0; c[CK_PREV] = (int32_t)head;
    c[CK_CNT_HI] = (int32_t)cnt_hi;
  }
}

template <int NP>
__device__ __forceinline__ uint32_t ck_write_pair(const WorkArgs& wa, const PairState& L, int lane, uint32_t head,
                                                  const CkScalars& cs, int32_t B, int32_t oe, uint32_t cnt,
                                                  uint32_t cnt_hi, const int32_t* sT) {
  uint32_t slot = 0;
  if (lane == 0) slot = atomicAdd(wa.ckpt_used, 1u);
  slot = __shfl_sync(FULL, slot, 0);
  if (slot >= wa.ckpt_cap) return head;
  ck_fill_pair<NP>(wa.ckpt + (uint64_t)slot * CK_SLOT_WORDS, L, lane, head, cs, B, oe, cnt, cnt_hi, sT);
  return slot + 1;
}

// Warp-uniform control state of the pair sweep.  Stored values are score
// minus B; T is the prune threshold, pend the part of its rises not yet
// moved out of the stored values, wbest2 the stored h of a cell scoring best
// in both halves.  A rise of the best score records its anti-diagonal
// (dbest).  The traced sweep locates the best cell lazily: the rise copies the
// window's h values to the warp's snapshot buffer (pair_after), and
// pair_best_row finds the cell's row when a checkpoint or the result needs
// it.  The plain sweep, whose rises are rare on short alignments, finds the
// row at once (bi).
struct PairCtl {
  int32_t b, d, best, dbest, d_last;
  int32_t bi;                // plain sweep: row of the best cell
  int32_t B, T, pend;
  uint32_t wbest2;
  uint32_t lb2;              // live_mask bias: 0x8000 - the stored threshold
  uint32_t live2;            // live masks summed since the last fold (live_count)
  uint32_t cnt;              // live cells of this lane (the 32-bit sweep's count)
  bool rowb_alive;           // row b is live at d
  bool top;                  // the window's top lane holds a live cell at d
};

// Snapshot buffer of a warp (shared memory): lane l's pair q at
// snap[32 q + l], then the stored maximum (-1 while the best cell is the
// origin) and the window, b | NP << 24.
constexpr int SNAP_WM = 32 * PK, SNAP_WIN = 32 * PK + 1, SNAP_WORDS = 32 * PK + 2;

// After each step: the anti-diagonal's best (warp max of the stored h), a
// rise of the best score (traced: with a snapshot of the window; plain: with
// the best cell's row), the last live anti-diagonal, and one ballot with row
// b's liveness (bit 0, lane 0) and the top lane's (bit 31, lane 31).
template <int NP, bool TR>
__device__ __forceinline__ uint32_t pair_after(PairState& L, PairCtl& c, uint32_t lm2, const Params& p, int lane,
                                               int32_t* sT, uint32_t m0, uint32_t m31, uint32_t* snap,
                                               uint32_t& wmd_out) {
  const int32_t oe = p.oe;
  // the lane max in both halves (a 32-bit compare of such values orders them
  // like their halves)
  const uint32_t lmd = __vmaxs2(lm2, prmt(lm2, 0u, 0x1032u));
  const uint32_t wmd = __reduce_max_sync(FULL, lmd);
  const uint32_t bits = __ballot_sync(FULL, ((L.H[0] & m0) | (lmd & m31)) != 0u);
  if (wmd > c.wbest2) {                     // implies a live cell (wbest2 > 0)
    const int32_t wm = (int32_t)lo16(wmd);
    if (TR) {
#pragma unroll
      for (int q = 0; q < NP; ++q) snap[32 * q + lane] = L.H[q];   // (each lane reads back only its own words)
      snap[SNAP_WM] = (uint32_t)wm;                                // (the same value from every lane)
      snap[SNAP_WIN] = (uint32_t)c.b | (NP << 24);
    } else {
      int rf = 2 * NP;
#pragma unroll
      for (int r = 2 * NP - 1; r >= 0; --r) rf = (int32_t)prow<NP>(L.H, r) == wm ? r : rf;
      const uint32_t fm = __ballot_sync(FULL, rf < 2 * NP);
      const int Ln = __ffs(fm) - 1;
      const int rr = __shfl_sync(FULL, rf, Ln);
      c.bi = c.b + Ln * 2 * NP + rr;
    }
    c.dbest = c.d;
    c.best = wm + oe + c.B;
    if (c.d <= 2 * EAGER_N && lane == 0) sT[c.d] = c.best;
    const int32_t Tn = threshold(c.best, p.ydrop);
    c.pend += Tn - c.T;
    c.T = Tn;
    if (c.pend > p.pair_slack) {
      const uint32_t dl = dup16(-c.pend);   // move every value down by the rise
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        L.H[q] = __viaddmax_s16x2_relu(L.H[q], dl, 0u);
        L.HP[q] = __viaddmax_s16x2_relu(L.HP[q], dl, 0u);
        L.I[q] = __viaddmax_s16x2_relu(L.I[q], dl, 0u);
        L.D[q] = __viaddmax_s16x2_relu(L.D[q], dl, 0u);
      }
      c.B += c.pend;
      c.pend = 0;
    }
    c.lb2 = dup16(0x8000 - (PMG - oe + c.pend));
    c.wbest2 = dup16(c.best - oe - c.B);
  }
  c.d_last = wmd != 0u ? c.d : c.d_last;
  wmd_out = wmd;
  return bits;
}

// Row of the best cell (the first cell in lane-then-row order holding the
// stored maximum of the snapshot; the origin while no rise was seen).  Warp
// collective.
template <int NP>
__device__ __forceinline__ int pair_snap_row(const uint32_t* snap, int lane, int32_t wm) {
  uint32_t H[PK];
#pragma unroll
  for (int q = 0; q < NP; ++q) H[q] = snap[32 * q + lane];
  int rf = 2 * NP;
#pragma unroll
  for (int r = 2 * NP - 1; r >= 0; --r) rf = (int32_t)prow<NP>(H, r) == wm ? r : rf;
  return rf;
}

template <bool TR>
__device__ __forceinline__ int32_t pair_best_row(const PairCtl& c, const uint32_t* snap, int lane) {
  if (!TR) return c.bi;
  const int32_t wm = (int32_t)snap[SNAP_WM];
  if (wm < 0) return 0;
  const uint32_t win = snap[SNAP_WIN];
  const int np = (int)(win >> 24);
  const int rf = np == NP_SMALL ? pair_snap_row<NP_SMALL>(snap, lane, wm) : pair_snap_row<PK>(snap, lane, wm);
  const uint32_t fm = __ballot_sync(FULL, rf < 2 * np);
  const int Ln = __ffs(fm) - 1;
  const int rr = __shfl_sync(FULL, rf, Ln);
  return (int32_t)(win & 0xffffffu) + Ln * 2 * np + rr;
}

// Per-warp shared buffer for changing the number of pairs per lane: the
// stored 16-bit values of up to 384 rows, row u at index u.
struct PairRelay {
  uint16_t H[64 * PK], HP[64 * PK], I[64 * PK], D[64 * PK];
};

template <int NP>
__device__ __forceinline__ void prelay_store(const PairState& L, int lane, PairRelay* rb) {
#pragma unroll
  for (int r = 0; r < 2 * NP; ++r) {
    const int u = 2 * NP * lane + r;
    rb->H[u] = (uint16_t)prow<NP>(L.H, r);
    rb->HP[u] = (uint16_t)prow<NP>(L.HP, r);
    rb->I[u] = (uint16_t)prow<NP>(L.I, r);
    rb->D[u] = (uint16_t)prow<NP>(L.D, r);
  }
  __syncwarp();
}

// Loads rows 0 .. rows_old-1 of the relay buffer into NP pairs per lane (rows
// beyond them are dead) and rebuilds every row's substitution row and query
// selector from the sequences: row b + u has target base b + u and, after
// anti-diagonal d, sits at column d - (b + u).
template <int NP>
__device__ __forceinline__ void prelay_load(PairState& L, int rows_old, const PairCtl& c, int lane,
                                            const PairRelay* rb, const Params& p, const Window& w,
                                            const uint32_t* s_mrow16) {
  const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)c.b + (int64_t)lane * 2 * NP);
  const uint32_t qw = fetch16(p.q2, p.q_len, w.qg0, w.dir, (int64_t)c.d - c.b - (int64_t)lane * 2 * NP - 15);
  const uint32_t oe = (uint32_t)p.oe;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int u0 = 2 * NP * lane + q, u1 = u0 + NP;
    const bool a0 = u0 < rows_old, a1 = u1 < rows_old;
    L.H[q] = (a0 ? rb->H[u0] : 0u) | ((a1 ? rb->H[u1] : 0u) << 16);
    L.HP[q] = (a0 ? rb->HP[u0] : oe) | ((a1 ? rb->HP[u1] : oe) << 16);
    L.I[q] = (a0 ? rb->I[u0] : 0u) | ((a1 ? rb->I[u1] : 0u) << 16);
    L.D[q] = (a0 ? rb->D[u0] : 0u) | ((a1 ? rb->D[u1] : 0u) << 16);
    L.SEL[q] = sel_lo((qw >> (2 * (15 - q))) & 3u) | (sel_hi((qw >> (2 * (15 - q - NP))) & 3u) << 8);
  }
#pragma unroll
  for (int r = 0; r < 2 * NP; ++r) L.MR[r] = s_mrow16[(tw >> (2 * r)) & 3u];
  __syncwarp();
}

// Lanes (from lane 0) that hold a live cell of anti-diagonal d or d - 1.
template <int NP>
__device__ __forceinline__ int pair_live_lanes(const PairState& L, uint32_t oe2) {
  uint32_t a = 0;
#pragma unroll
  for (int q = 0; q < NP; ++q) a |= L.H[q] | (L.HP[q] ^ oe2);
  const uint32_t bits = __ballot_sync(FULL, a != 0u);
  return bits ? 32 - __clz(bits) : 0;
}

// Per-warp trace of the traced pair sweep.  Anti-diagonal d's flags are row d
// of `rows` (256 bytes): with more than 4 pairs per lane, lane l's 8 bytes
// (pair_flags' acc[0], acc[1]) cover its 2 NP window rows b + 2 NP l ..
// b + 2 NP l + 2 NP - 1; with at most 4 pairs acc[1] is 0 and lane l stores
// only acc[0], as the l-th 32-bit word of the row (its first 128 bytes).
// hdr[d] = b | NP << 24 gives the window of that step.  runs: the walk's
// runs, in walk order.
struct TraceSlot {
  uint2* rows;
  int32_t* hdr;
  uint32_t* runs;
  int32_t* ring;     // wa.tring checkpoint slots (see ring_publish)
};

template <int NP>
__device__ __forceinline__ void trace_store(const TraceSlot& ts, const PairCtl& c, int lane, const uint32_t (&acc)[2]) {
  if (NP <= 4) reinterpret_cast<uint32_t*>(ts.rows)[(uint32_t)c.d * 64u + (uint32_t)lane] = acc[0];
  else ts.rows[(uint32_t)c.d * 32u + (uint32_t)lane] = make_uint2(acc[0], acc[1]);
  if (lane == 0) ts.hdr[c.d] = c.b | (NP << 24);
}

// Steps of the pair sweep with NP pairs per lane (a 64 NP-row window) from
// anti-diagonal c.d until the sweep ends (returns 2), the live band reaches
// the window's top lane while row b is live (1: the window must grow, or the
// extension overflows at 384 rows), or c.d reaches d_stop (0).
//
// Away from the window's edges the steps run in fixed pairs: a step that
// keeps the base, then one that moves it up a row.  A loop with one kind of
// step after the other needs no register moves between them, where a loop
// choosing the kind per step pays for both register layouts every step.  The
// pair ends after its first step when row b is live (the base cannot move:
// the next pair starts right away, inside the loop, since leaving and
// re-entering it costs more than a step), and the loop is left after the
// second step when the top lane is live (the next step is then taken alone).
// Keeping the base while row b is dead only leaves a dead row at the bottom,
// so every live cell stays inside the window; the base never passes the base
// of the shift-by-one rule, and the two agree whenever row b is live, which is
// when the window has to grow or the extension overflows — the same decisions
// as the shift-by-one rule.
//
// Steps that cannot touch the window's edges run without edge masks: the base
// grows by at most one row per step, so b + 64 NP <= m and b >= d - n hold
// for that many steps.  An overflow test of one step suffices: a cell beyond
// the window's top row at d needs that row live at d-1 (gap) or d-2
// (diagonal) with the base kept since, which the test of that step saw.
//
// With TR every step's direction flags go to the trace slot (trace_store).
template <int NP, bool TR>
__device__ __forceinline__ int pair_run(PairState& L, PairCtl& c, const Params& p, const Window& w, int lane,
                                     Reservoir& qr, Reservoir& tr, const uint32_t* s_mrow16, int32_t* sT,
                                     int32_t d_stop, uint32_t m0, uint32_t m31, const TraceSlot& ts,
                                     uint32_t* snap) {
  constexpr int32_t WIN = 64 * NP;
  const int32_t m = w.m, n = w.n, mn = w.m + w.n, oe = p.oe;
  const uint32_t ne2 = dup16(-p.e), noe2 = dup16(-oe), oe2 = dup16(oe);
  // the last anti-diagonal up to which steps cannot touch the window's edges;
  // it never decreases (d - b and b + n never do), so it is recomputed only
  // once reached
  int32_t d_fast = c.d;
  for (;;) {
    if (d_fast <= c.d) d_fast = imin(d_stop, c.d + imin(m - WIN - c.b, c.b - c.d + n));
    bool ovf;
    if (d_fast > c.d && !c.top) {
      uint32_t bits, wmd;
      for (;;) {
        {
          const uint32_t qb = res_take(qr, p.q2, p.q_len, w.qg0, w.dir);
          uint32_t acc[2] = {0u, 0u};
          const uint32_t lm2 = pstep<NP, false, false, TR>(L, ne2, noe2, oe2, c.lb2, lane, qb, 0u, 0, 0, c.live2, acc);
          ++c.d;
          if (TR) trace_store<NP>(ts, c, lane, acc);
          bits = pair_after<NP, TR>(L, c, lm2, p, lane, sT, m0, m31, snap, wmd);
        }
        if ((bits & 1u) || c.d == d_fast || wmd == 0u) {
          // row b live: the base stays and the next pair starts here, unless
          // the window must grow or overflows (the top lane is live too)
          if (bits != 1u || c.d == d_fast || wmd == 0u) break;
          continue;
        }
        {
          const uint32_t mr_new = s_mrow16[res_take(tr, p.t2, p.t_len, w.tg0, w.dir)];
          uint32_t acc[2] = {0u, 0u};
          const uint32_t lm2 = pstep<NP, true, false, TR>(L, ne2, noe2, oe2, c.lb2, lane, 0u, mr_new, 0, 0, c.live2, acc);
          ++c.b;
          ++c.d;
          if (TR) trace_store<NP>(ts, c, lane, acc);
          bits = pair_after<NP, TR>(L, c, lm2, p, lane, sT, m0, m31, snap, wmd);
        }
        if ((int32_t)bits < 0 || c.d == d_fast || wmd == 0u) break;
      }
      // (an anti-diagonal without a live cell leaves the pairs; two in a row end the sweep)
      c.rowb_alive = bits & 1u;
      c.top = (int32_t)bits < 0;
      if (c.d - c.d_last >= 2) return 2;
      if (c.rowb_alive && c.top) return 1;
      if (c.d >= d_stop) return 0;
      continue;
    } else {
      // one step of the shift-by-one rule, with edge masks: rows beyond m or
      // columns beyond n are dead
      const bool shift = !c.rowb_alive;
      const int32_t bn = c.b + (shift ? 1 : 0), dn = c.d + 1;
      const int32_t rowbase = bn + lane * 2 * NP;
      const int32_t vhi = m - rowbase, vlo = dn - n - rowbase;
      uint32_t lm2;
      uint32_t acc[2] = {0u, 0u};
      if (!shift) {
        const uint32_t qb = res_take(qr, p.q2, p.q_len, w.qg0, w.dir);
        lm2 = pstep<NP, false, true, TR>(L, ne2, noe2, oe2, c.lb2, lane, qb, 0u, vlo, vhi, c.live2, acc);
      } else {
        const uint32_t mr_new = s_mrow16[res_take(tr, p.t2, p.t_len, w.tg0, w.dir)];
        lm2 = pstep<NP, true, true, TR>(L, ne2, noe2, oe2, c.lb2, lane, 0u, mr_new, vlo, vhi, c.live2, acc);
      }
      c.b = bn;
      c.d = dn;
      if (TR) trace_store<NP>(ts, c, lane, acc);
      uint32_t wmd;
      const uint32_t bits = pair_after<NP, TR>(L, c, lm2, p, lane, sT, m0, m31, snap, wmd);
      c.rowb_alive = bits & 1u;
      c.top = (int32_t)bits < 0;
      // (no overflow once the window reaches row m: no row lies beyond it)
      ovf = (bits & 0x80000001u) == 0x80000001u && c.b + WIN <= m;
    }
    if (c.d - c.d_last >= 2 || c.d + 1 > mn) return 2;
    if (ovf) return 1;
    if (c.d >= d_stop) return 0;
  }
}

// ---- traced pair sweep: the walk ----
//
// Per-warp staging of 32 anti-diagonals of the trace: for anti-diagonal
// d0 - t (lane t) the window origin, the rows per lane and the flags of the
// lanes that hold rows i - t .. i (every row the walk can reach there from
// row i of d0: each step back lowers the row by at most one per
// anti-diagonal).  Those rows span at most 32 rows, i.e. at most 5 lanes of 8
// or more rows each.
constexpr int WALK_WORDS = 6;
struct WalkStage {
  uint2 w[32][WALK_WORDS];
  int32_t b[32], rpl[32], l0[32];
};

// Lane 0's run accumulation in walk order (runs (len << 4) | op; op 0 = M,
// 1 = I, 2 = D).
struct WalkRuns {
  uint32_t* dst;
  uint32_t cap, nr, op, len;
  bool bad;
  __device__ void push_n(uint32_t o, uint32_t n) {
    if (o == op) { len += n; return; }
    if (len) {
      if (nr >= cap) { bad = true; return; }
      dst[nr++] = (len << 4) | op;
    }
    op = o;
    len = n;
  }
  __device__ void flush() {
    if (!len) return;
    if (nr >= cap) { bad = true; return; }
    dst[nr++] = (len << 4) | op;
    len = 0;
  }
};

// The four direction flags of row `row` at staged anti-diagonal d0 - t
// (bit 0: S not from the diagonal, bit 1: not from I, bit 2: I extends, bit 3:
// D extends), or 0x10 when the row is not in the staged flags.
__device__ __forceinline__ uint32_t staged_flags(const WalkStage* sm, int t, int32_t row) {
  const int32_t rpl = sm->rpl[t], np = rpl >> 1;
  const int32_t u = row - sm->b[t];
  if (u < 0 || u >= 32 * rpl) return 0x10u;
  const int32_t l = rpl == 8 ? (u >> 3) : ((u * 2731) >> 15);   // u / rpl (rpl 8 or 12, u < 384)
  const int32_t r = u - l * rpl, k = l - sm->l0[t];
  if (k < 0 || k >= WALK_WORDS) return 0x10u;
  const uint2 wv = sm->w[t][k];
  const int32_t half = r >= np ? 1 : 0, pp = r - half * np;
  const uint32_t w32 = ((pp < 4 ? wv.x : wv.y) >> (16 * half)) << (2 * (pp & 3));
  return ((w32 >> 7) & 1u) | ((w32 >> 14) & 2u) | ((w32 >> 4) & 4u) | ((w32 >> 11) & 8u);
}

// Walks from the best cell (bi, bj) in state S back to the origin through the
// traced flags (the traceback rules of the oracle: in S the diagonal, then I,
// then D; in a gap state the gap opens when its flag says it does not extend;
// on row 0 only I moves remain, on column 0 only D moves).  The warp stages 32
// anti-diagonals of flags at a time in shared memory and then takes a whole
// run per round: in S, lane k looks at the k-th cell down the diagonal
// (anti-diagonal 2k further back), in I at the k-th cell to the left, in D at
// the k-th cell above, and one ballot gives where the run ends.  Writes the
// runs in walk order to ts.runs (at most cap) and returns their number, or
// 0xffffffff if the walk left the staged flags or the run buffer.
__device__ __noinline__ uint32_t trace_walk(const TraceSlot& ts, int32_t bi, int32_t bj, uint32_t cap, int lane,
                                            WalkStage* sm) {
  int32_t i = bi, j = bj, st = 0;
  WalkRuns wr;
  wr.dst = ts.runs; wr.cap = cap; wr.nr = 0; wr.op = 0xffu; wr.len = 0; wr.bad = false;
  bool bad = false;
  while (i > 0 && j > 0 && !bad) {
    // stage anti-diagonals d0 - t, t = lane: the rows i - t .. i
    const int32_t d0 = i + j;
    const int32_t dt = d0 - lane;
    if (dt >= 1) {
      const int32_t h = __ldcg(ts.hdr + dt);
      const int32_t b = h & 0xffffff, rpl = 2 * (h >> 24);
      const int32_t lo = imax(i - lane - b, 0), hi = imin(i - b, 32 * rpl - 1);
      const int32_t l0 = lo <= hi ? lo / rpl : 0;
      const int32_t l1 = lo <= hi ? hi / rpl : -1;
      sm->b[lane] = b;
      sm->rpl[lane] = rpl;
      sm->l0[lane] = l0;
#pragma unroll
      for (int k = 0; k < WALK_WORDS; ++k)
        if (l0 + k <= l1)
          sm->w[lane][k] = rpl <= 8 ? make_uint2(__ldcg(reinterpret_cast<const uint32_t*>(ts.rows) +
                                                        (uint32_t)dt * 64u + (uint32_t)(l0 + k)), 0u)
                                    : __ldcg(ts.rows + (uint32_t)dt * 32u + (uint32_t)(l0 + k));
    }
    __syncwarp();
    // The next two stages start near d0 - 32 and d0 - 64 (the walk leaves a
    // stage 32 or 33 anti-diagonals down): bring their headers and flag rows
    // to L2 while this stage's runs resolve, so that their staging loads do
    // not each wait for DRAM.  Only a row's first 128-byte line: with at most
    // 4 pairs per lane (nearly every traced step) the second holds no flags.
#pragma unroll
    for (int s = 1; s <= 2; ++s) {
      const int32_t dn = d0 - 32 * s - lane;
      if (dn >= 1) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ts.rows + (uint32_t)dn * 32u));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ts.hdr + dn));
      }
    }
    // runs inside the staged window (t = d0 - (i + j) <= 31)
    for (;;) {
      const int t = d0 - (i + j);
      if (i <= 0 || j <= 0 || t > 31) break;
      const int k = lane;
      uint32_t fl = 0;
      bool valid;
      if (st == 0) {
        valid = k < 16 && t + 2 * k <= 31 && i - k >= 1 && j - k >= 1;
        if (valid) fl = staged_flags(sm, t + 2 * k, i - k);
      } else if (st == 1) {
        valid = t + k <= 31 && j - k >= 1;
        if (valid) fl = staged_flags(sm, t + k, i);
      } else {
        valid = t + k <= 31 && i - k >= 1;
        if (valid) fl = staged_flags(sm, t + k, i - k);
      }
      // (lanes past the end of the run look at cells the walk does not reach,
      // which may lie outside the traced window: only the lane where the run
      // stops must hold a cell of it)
      const uint32_t eb = __ballot_sync(FULL, valid && (fl & 0x10u));
      const uint32_t vb = __ballot_sync(FULL, valid) & ~eb;
      if (st == 0) {
        // diagonal moves while the cell's S comes from the diagonal
        const uint32_t go = __ballot_sync(FULL, valid && !(fl & 0x11u));
        const uint32_t nib = __ballot_sync(FULL, (fl & 2u) != 0u);
        const int f = __ffs(~go) - 1;                   // 0..16
        if ((eb >> f) & 1u) { bad = true; break; }
        if (lane == 0 && f) wr.push_n(0u, (uint32_t)f);
        i -= f;
        j -= f;
        if ((vb >> f) & 1u) st = ((nib >> f) & 1u) ? 2 : 1;   // S from D, else from I (same cell)
      } else {
        // gap moves while the gap extends; the cell where it opens is the run's last
        const uint32_t go = __ballot_sync(FULL, valid && (fl & 0x10u) == 0u && (fl & (st == 1 ? 4u : 8u)));
        const int f = go == FULL ? 32 : __ffs(~go) - 1;  // 0..32
        if (f < 32 && ((eb >> f) & 1u)) { bad = true; break; }
        const bool opens = f < 32 && ((vb >> f) & 1u);
        const int n = opens ? f + 1 : f;
        if (lane == 0 && n) wr.push_n((uint32_t)st, (uint32_t)n);
        if (st == 1) j -= n;
        else i -= n;
        if (opens) st = 0;
        else if ((st == 1 && j == 0) || (st == 2 && i == 0)) bad = true;   // a gap cannot run off the matrix
      }
      bad = __shfl_sync(FULL, (bad || wr.bad) ? 1 : 0, 0) != 0;
      if (bad) break;
    }
    __syncwarp();
  }
  if (lane == 0 && !bad) {
    if (i == 0 && j > 0) {
      if (st == 2) bad = true;
      else wr.push_n(1u, (uint32_t)j);                     // row 0: I moves only
    } else if (j == 0 && i > 0) {
      if (st == 1) bad = true;
      else wr.push_n(2u, (uint32_t)i);                     // column 0: D moves only
    }
    wr.flush();
    bad = bad || wr.bad;
  }
  const uint32_t nr = __shfl_sync(FULL, bad ? 0xffffffffu : wr.nr, 0);
  __syncwarp();
  return nr;
}

// Changes the window from NPO to NPN pairs per lane, keeping base row b:
// rows move through the per-warp relay buffer.  When shrinking, the caller
// has checked that the dropped rows are dead at d and d - 1 (a cell above the
// new top can then only become live through the rows below it, which the
// overflow test watches).
template <int NPO, int NPN>
__device__ __forceinline__ void pair_resize(PairState& L, const PairCtl& c, int lane, PairRelay* rb,
                                            const Params& p, const Window& w, const uint32_t* s_mrow16,
                                            Reservoir& tr) {
  prelay_store<NPO>(L, lane, rb);
  prelay_load<NPN>(L, 64 * NPO, c, lane, rb, p, w, s_mrow16);
  res_init(tr, p.t2, p.t_len, w.tg0, w.dir, (int64_t)c.b + 64 * NPN);   // target rows entering at the new top
}

template <bool TR>
__device__ __forceinline__ uint32_t pair_ckpt(int np, const WorkArgs& wa, const PairState& L, int lane,
                                              uint32_t head, const PairCtl& c, int32_t oe, const int32_t* sT,
                                              const uint32_t* snap) {
  const int32_t bi = pair_best_row<TR>(c, snap, lane);
  const CkScalars cs{c.b, c.d, c.best, bi, c.dbest - bi, c.d_last};
  return np == NP_SMALL ? ck_write_pair<NP_SMALL>(wa, L, lane, head, cs, c.B, oe, c.cnt, 0u, sT)
                        : ck_write_pair<PK>(wa, L, lane, head, cs, c.B, oe, c.cnt, 0u, sT);
}

// Traced sweep: checkpoints go to a ring in the warp's trace slot (one every
// wa.tring_every anti-diagonals) instead of the shared pool, since no
// executor replays a traced extension.  Only when the extension overflows the
// 384-row window (it then continues untraced in the 512-row tier and the
// executor traces it) are they copied to the pool and linked (ring_publish),
// so that the executor splits its replay at them.
__device__ __forceinline__ void ring_ckpt(int np, const TraceSlot& ts, uint32_t k, const PairState& L, int lane,
                                          const PairCtl& c, int32_t oe, const int32_t* sT, const uint32_t* snap) {
  const int32_t bi = pair_best_row<true>(c, snap, lane);
  const CkScalars cs{c.b, c.d, c.best, bi, c.dbest - bi, c.d_last};
  int32_t* dst = ts.ring + (uint64_t)k * CK_SLOT_WORDS;
  if (np == NP_SMALL) ck_fill_pair<NP_SMALL>(dst, L, lane, 0u, cs, c.B, oe, c.cnt, 0u, sT);
  else ck_fill_pair<PK>(dst, L, lane, 0u, cs, c.B, oe, c.cnt, 0u, sT);
}

// Copies the n ring checkpoints (oldest first) to consecutive pool slots,
// each linked to the one before; returns the newest's slot + 1, or 0 when the
// pool has no room (the executor then replays from the origin).
__device__ __noinline__ uint32_t ring_publish(const WorkArgs& wa, const TraceSlot& ts, uint32_t n, int lane) {
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(wa.ckpt_used, n);
  base = __shfl_sync(FULL, base, 0);
  if ((uint64_t)base + n > wa.ckpt_cap) return 0u;
  for (uint32_t k = 0; k < n; ++k) {
    const int32_t* src = ts.ring + (uint64_t)k * CK_SLOT_WORDS;
    int32_t* dst = wa.ckpt + (uint64_t)(base + k) * CK_SLOT_WORDS;
    for (int w = lane; w < CK_SLOT_WORDS; w += 32) dst[w] = __ldcg(src + w);
    __syncwarp();
    if (lane == 0) dst[CK_PREV] = (int32_t)(k ? base + k : 0u);   // the previous entry's slot + 1
  }
  __syncwarp();
  return base + n;
}

// The pair sweep of one extension.  The window has two sizes: 256 rows (4
// pairs per lane) to start with, and 384 rows (6 pairs): it grows when the
// live band reaches the top lane of the small one while row b is live, and
// every 64 anti-diagonals the large one shrinks back when the rows live at d
// and d - 1 fit in the small one's first 30 lanes.  At 384 rows the same
// top-lane test is the first tier's overflow, as for a fixed 384-row window:
// the base row follows the same rule at both sizes, so the values, best
// cells, live counts and the overflow decision do not depend on the size.
//
// TR (the traced sweep): every step's direction flags go to the warp's trace
// slot, no periodic checkpoints are written (no executor replays this
// extension), and after the sweep the warp walks its best cell back to the
// origin (trace_walk) and puts the runs, in forward genomic order, in the
// traced-run arena; the record then carries FZ_XFLAG_TRACED with the runs'
// offset (path) and count (npath).  If the arena is full the record is left
// for the executor, which replays the sweep from the origin.
template <bool TR>
__device__ void run_inspect_pair(const Params& p, const WorkArgs& wa, uint32_t ext, int lane, int32_t* sT,
                                 uint8_t* tile, const uint32_t* s_mrow16, const int32_t* s_sub, PairRelay* rb,
                                 const TraceSlot& ts, WalkStage* wsm, uint32_t* snap) {
  constexpr int32_t WIN = 64 * PK;   // the first tier's largest window (the executor's row width)
  const Window w = make_window(p, ext);
  ExtRec* R = wa.rec + ext;
  if (!w.requested) {
    if (lane == 0) {
      ExtRec z = {};
      *R = z;
    }
    return;
  }
  const int32_t m = w.m, n = w.n, oe = p.oe, mn = w.m + w.n;
  PairCtl c;
  c.b = 0; c.d = 0; c.best = 0; c.dbest = 0; c.d_last = 0; c.bi = 0;
  if (lane == 0) snap[SNAP_WM] = 0xffffffffu;   // best cell: the origin
  c.T = threshold(0, p.ydrop);
  c.B = c.T - PMG;                          // stored value = score-space value - B
  // A rise of the threshold is first only added to the stored threshold
  // (pend); the values move down once pend passes the slack that the 16-bit
  // range leaves (Params::pair_slack).
  c.pend = 0;
  c.wbest2 = dup16(c.best - oe - c.B);
  c.lb2 = dup16(0x8000 - (PMG - oe));
  c.live2 = 0u;
  c.cnt = lane == 0 ? 1u : 0u;
  c.rowb_alive = true;
  c.top = false;
  const uint32_t oe2 = dup16(oe);
  const uint32_t m0 = lane == 0 ? 0xffffu : 0u;          // lane 0 reports row b,
  const uint32_t m31 = lane == 31 ? 0xffffffffu : 0u;    // lane 31 its rows (the window's top lane)
  int np = NP_SMALL;
  PairState L;
  {
    const uint32_t tw = fetch16(p.t2, p.t_len, w.tg0, w.dir, (int64_t)lane * 2 * NP_SMALL);
#pragma unroll
    for (int r = 0; r < 2 * PK; ++r) L.MR[r] = s_mrow16[(tw >> (2 * r)) & 3u];
#pragma unroll
    for (int q = 0; q < PK; ++q) {
      L.H[q] = 0u; L.HP[q] = oe2; L.I[q] = 0u; L.D[q] = 0u;
      L.SEL[q] = sel_lo(0) | (sel_hi(0) << 8);
    }
    if (lane == 0) L.H[0] = (uint32_t)(-oe - c.B) & 0xffffu;      // origin: S(0,0) = 0
  }
  uint32_t head = 0u;
  uint32_t nring = 0u;                      // traced: ring checkpoints written
  sT[lane] = NEG;
  if (lane == 0) sT[32] = NEG;
  __syncwarp();
  Reservoir qr, tr;
  res_init(qr, p.q2, p.q_len, w.qg0, w.dir, 1);
  res_init(tr, p.t2, p.t_len, w.tg0, w.dir, 64 * NP_SMALL);
  // the sweep stops every ex_mask + 1 anti-diagonals (at most 2048, so that
  // each half's live count stays below 2^15 for live_count) to fold the live
  // count and to write the checkpoints, and with the large window every 64
  // anti-diagonals to see whether the small one holds the band again
  const uint32_t ck_mask = wa.ckpt ? (uint32_t)wa.ckpt_every - 1u : 0xffffffffu;
  const uint32_t ex_mask = (wa.ckpt && wa.ckpt_every <= 2048) ? (uint32_t)wa.ckpt_every - 1u : 2047u;
  bool overflow = false;

  int why = c.d + 1 > mn ? 2 : 0;   // 0 boundary, 1 top lane live with the base kept, 2 end
  while (why != 2) {
    const uint32_t mask = np == PK ? (ex_mask & 63u) : ex_mask;
    const int32_t d_stop = (int32_t)(((uint32_t)c.d | mask) + 1u);
    why = np == PK ? pair_run<PK, TR>(L, c, p, w, lane, qr, tr, s_mrow16, sT, d_stop, m0, m31, ts, snap)
                   : pair_run<NP_SMALL, TR>(L, c, p, w, lane, qr, tr, s_mrow16, sT, d_stop, m0, m31, ts, snap);
    if (why != 0 || ((uint32_t)c.d & ex_mask) == 0u) {
      c.cnt += live_count(c.live2);
      c.live2 = 0u;
    }
    if (why == 2) break;
    if (why == 1) {
      if (np == PK) {
        overflow = true;   // the live band may grow past the 384-row window
        break;
      }
      pair_resize<NP_SMALL, PK>(L, c, lane, rb, p, w, s_mrow16, tr);
      np = PK;
      c.top = false;        // the new top lane's rows lay beyond the old window: dead
      continue;
    }
    if (!TR && ((uint32_t)c.d & ck_mask) == 0u && c.d - c.dbest <= wa.ckpt_recent)
      head = pair_ckpt<TR>(np, wa, L, lane, head, c, oe, sT, snap);
    if (TR && wa.ckpt && ((uint32_t)c.d & (wa.tring_every - 1u)) == 0u && nring < wa.tring) {
      ring_ckpt(np, ts, nring, L, lane, c, oe, sT, snap);
      ++nring;
    }
    if (np == PK) {
      const int lanes = pair_live_lanes<PK>(L, oe2);   // lanes with a live cell at d or d-1
      if (lanes * 2 * PK <= 60 * NP_SMALL) {
        pair_resize<PK, NP_SMALL>(L, c, lane, rb, p, w, s_mrow16, tr);
        np = NP_SMALL;
        c.top = false;      // rows 240 and up are dead at d and d - 1
      }
    }
  }
  if (overflow && wa.ckpt) {
    if (TR && nring) head = ring_publish(wa, ts, nring, lane);
    head = pair_ckpt<TR>(PK, wa, L, lane, head, c, oe, sT, snap);
  }

  uint64_t tot = c.cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  if (overflow) {
    if (lane == 0) {
      ExtRec z = {};
      z.flags = FZ_FLAG_DONE | FZ_FLAG_WIDE;
      z.m = m;
      z.n = n;
      z.ckpt = head;
      *R = z;
      const uint32_t slot = atomicAdd(wa.ovf_count, 1u);
      wa.ovf_list[slot] = ext;
    }
    return;
  }
  const int32_t best = c.best, bi = pair_best_row<TR>(c, snap, lane), bj = c.dbest - bi;
  uint64_t path = 0;
  uint32_t npath = 0;
  uint32_t flags = FZ_FLAG_DONE;
  uint32_t width = WIN;
  if (bi <= EAGER_N && bj <= EAGER_N) {
    flags |= FZ_FLAG_EAGER;
    width = 0;
    if (bi + bj > 0) {
      int32_t v = sT[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) v = imax(v, __shfl_up_sync(FULL, v, o));
      v = imax(v, 0);
      __syncwarp();
      sT[lane + 1] = threshold(v, p.ydrop);
      __syncwarp();
      eager_corner(p, w, lane, sT, tile, s_sub, bi, bj, path, npath, wa.err);
    }
  } else if (TR) {
    const uint32_t nr = trace_walk(ts, bi, bj, (uint32_t)(bi + bj), lane, wsm);
    if (nr == 0xffffffffu) {
      if (lane == 0) atomicOr(wa.err, 0x20u);      // (the executor still traces it)
    } else {
      unsigned long long off = 0;
      if (lane == 0) off = atomicAdd(wa.truns_used, (unsigned long long)nr);
      off = __shfl_sync(FULL, off, 0);
      if (off + nr <= wa.truns_cap) {
        const bool right = (ext & 1u) == 0u;       // right side: genomic order is the walk reversed
        for (uint32_t k = (uint32_t)lane; k < nr; k += 32) wa.truns[off + k] = __ldcg(ts.runs + (right ? nr - 1 - k : k));
        path = off;
        npath = nr;
        flags |= FZ_XFLAG_TRACED;
        width = 0;
      }
    }
  }
  if (lane == 0) {
    ExtRec o;
    o.score = best; o.i_end = bi; o.j_end = bj; o.d_last = c.d_last;
    o.live = tot; o.path = path; o.flags = flags; o.npath = npath;
    o.m = m; o.n = n; o.width = width; o.ckpt = head;
    *R = o;
    atomicAdd(wa.live_total, (unsigned long long)tot);
    if (TR) atomicAdd(wa.traced_live, (unsigned long long)tot);
  }
}

// The first inspector tier as the pair sweep.  TR: the traced sweep over the
// extensions predicted long (list[0 .. *n_work_dev)); otherwise the plain
// sweep (with list_base_dev set: over list[*list_base_dev .. n_work)).
template <bool TR>
__global__ void __launch_bounds__(WARPS * 32, 4) k_pair(Params p, WorkArgs wa) {
  __shared__ int32_t s_T[WARPS][2 * EAGER_N + 2];
  __shared__ uint8_t s_tile[WARPS][(EAGER_N + 1) * (EAGER_N + 1)];
  __shared__ PairRelay s_relay[WARPS];
  __shared__ WalkStage s_walk[TR ? WARPS : 1];
  __shared__ uint32_t s_snap[WARPS][SNAP_WORDS];
  __shared__ uint32_t s_mrow16[4];
  __shared__ int32_t s_sub[16];
  if (threadIdx.x < 4) s_mrow16[threadIdx.x] = p.mrow16[threadIdx.x];
  if (threadIdx.x < 16) s_sub[threadIdx.x] = p.sub[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TraceSlot ts{};
  if (TR) {
    const uint32_t gw = blockIdx.x * WARPS + warp;
    if (gw >= wa.tslots) return;                   // (warp-uniform; no block barrier follows)
    uint8_t* base = wa.tpool + (uint64_t)gw * wa.tslot_bytes;
    ts.rows = reinterpret_cast<uint2*>(base);
    ts.hdr = reinterpret_cast<int32_t*>(base + (uint64_t)wa.tslot_rows * 256u);
    ts.runs = reinterpret_cast<uint32_t*>(base + (uint64_t)wa.tslot_rows * 260u);
    ts.ring = reinterpret_cast<int32_t*>(base + (uint64_t)wa.tslot_rows * 264u);
  }
  const uint32_t lbase = wa.list_base_dev ? *wa.list_base_dev : 0u;
  const uint32_t nw = wa.n_work_dev ? *wa.n_work_dev : wa.n_work - lbase;
  for (;;) {
    uint32_t idx = 0;
    if (lane == 0) idx = atomicAdd(wa.counter, 1u);
    idx = __shfl_sync(FULL, idx, 0);
    if (idx >= nw) break;
    const uint32_t ext = wa.list ? wa.list[lbase + idx] : lbase + idx;
    run_inspect_pair<TR>(p, wa, ext, lane, s_T[warp], s_tile[warp], s_mrow16, s_sub, &s_relay[warp], ts,
                         &s_walk[TR ? warp : 0], s_snap[warp]);
  }
}

// MINB: resident blocks per SM the register budget is fitted to.
template <int K, bool TRACE, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB) k_extend(Params p, WorkArgs wa) {
  __shared__ int32_t s_T[WARPS][2 * EAGER_N + 2];
  __shared__ uint8_t s_tile[WARPS][(EAGER_N + 1) * (EAGER_N + 1)];
  __shared__ uint32_t s_mrow[4];
  __shared__ int32_t s_sub[16];
  __shared__ Relay<TRACE ? K : 2> s_relay[WARPS];
  if (threadIdx.x < 4) s_mrow[threadIdx.x] = p.mrow[threadIdx.x];
  if (threadIdx.x < 16) s_sub[threadIdx.x] = p.sub[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (;;) {
    uint32_t idx = 0;
    if (lane == 0) idx = atomicAdd(wa.counter, 1u);
    idx = __shfl_sync(FULL, idx, 0);
    const uint32_t nw = wa.n_work_dev ? *wa.n_work_dev : wa.n_work;
    if (idx >= nw) break;
    if (TRACE) {
      // executor segment; only the extensions this window size inspected
      const uint4 sg = wa.seg[idx];
      const uint32_t ext = wa.list[sg.x];
      const ExtRec& r = wa.rec[ext];
      if ((r.flags & FZ_FLAG_WIDE) || r.width != (uint32_t)(32 * K)) continue;
      run_exec<K>(p, wa, ext, sg, lane, s_mrow, reinterpret_cast<Relay<K>*>(&s_relay[warp]));
    } else {
      const uint32_t ext = wa.list ? wa.list[idx] : idx;
      run_inspect<K>(p, wa, ext, lane, s_T[warp], s_tile[warp], s_mrow, s_sub);
    }
  }
}

}  // namespace

// Two register windows: 384 rows (K = 12, fitted to 4 blocks of 4 warps per
// SM) holds the live band of typical y-drop extensions; extensions whose band
// could outgrow it are retried with 512 rows (K = 16), then the wide path.
constexpr int KA = K_TIER0, KB = K_TIER1;

int fast_window_rows(int tier) { return 32 * (tier == 0 ? KA : KB); }

cudaError_t launch_inspect_fast(int tier, const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  if (tier == 0 && p.pair_ok) k_pair<false><<<grid, WARPS * 32, 0, st>>>(p, wa);
  else if (tier == 0) k_extend<KA, false, 4><<<grid, WARPS * 32, 0, st>>>(p, wa);
  else k_extend<KB, false, 1><<<grid, WARPS * 32, 0, st>>>(p, wa);
  return cudaGetLastError();
}

cudaError_t launch_inspect_traced(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  k_pair<true><<<grid, WARPS * 32, 0, st>>>(p, wa);
  return cudaGetLastError();
}

int traced_blocks_per_sm() {
  int nb = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_pair<true>, WARPS * 32, 0);
  return nb > 0 ? nb : 1;
}

cudaError_t launch_execute_fast(int tier, const Params& p, const WorkArgs& wa, int grid, cudaStream_t st) {
  if (tier == 0) k_extend<KA, true, 4><<<grid, WARPS * 32, 0, st>>>(p, wa);
  else k_extend<KB, true, 1><<<grid, WARPS * 32, 0, st>>>(p, wa);
  return cudaGetLastError();
}

int extend_fast_blocks_per_sm(int tier, bool trace, bool pair) {
  int nb = 0;
  if (tier == 0 && !trace && pair) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_pair<false>, WARPS * 32, 0);
  } else if (tier == 0) {
    if (trace) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_extend<KA, true, 4>, WARPS * 32, 0);
    else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_extend<KA, false, 4>, WARPS * 32, 0);
  } else {
    if (trace) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_extend<KB, true, 1>, WARPS * 32, 0);
    else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_extend<KB, false, 1>, WARPS * 32, 0);
  }
  return nb > 0 ? nb : 1;
}

}  // namespace fz
