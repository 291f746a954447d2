// Device-side definitions shared by the fz kernels (sm_103a).
#pragma once

#include <cstdint>

#include "fz.h"

namespace fz {

constexpr int32_t NEG = -(1 << 30);       // dead / missing score
constexpr int32_t TFLOOR = -(1 << 29);    // lowest threshold: every reachable cell is above it
constexpr unsigned FULL = 0xffffffffu;
constexpr int EAGER_N = 16;               // eager traceback corner: i*, j* <= 16
constexpr int K_TIER0 = 12, K_TIER1 = 16; // rows per lane of the two register windows (384, 512 rows)
// ExtRec flag (internal, never in an fz_result): traced by the inspector's
// traced sweep; path = first run in the traced-run arena, npath = runs
constexpr uint32_t FZ_XFLAG_TRACED = 1u << 16;

// Per-extension record written by the inspector, read by binning, the
// executor and the traceback.
struct ExtRec {
  int32_t score, i_end, j_end, d_last;    // best S, its cell, last anti-diagonal with a live cell
  uint64_t live;                          // live cells of the sweep
  uint64_t path;                          // eager traceback: ops walking back, 2 bits each;
                                          // traced: first run in the traced-run arena
  uint32_t flags;                         // FZ_FLAG_*
  uint32_t npath;                         // ops in path
  int32_t m, n;                           // window sizes
  uint32_t width;                         // executor trace row width (cells), 0 = no executor
  uint32_t ckpt;                          // newest window checkpoint + 1 (0 = none)
};
static_assert(sizeof(ExtRec) == 56, "ExtRec layout");

struct Params {
  const uint8_t* t2;
  const uint8_t* q2;
  uint64_t t_len, q_len;
  const fz_seed* seeds;
  uint32_t n_seeds;
  int32_t o, e, oe;
  int32_t ydrop;          // >= 0, or FZ_YDROP_INF
  int32_t max_len;
  int32_t one;            // 1, opaque to the compiler (see imad)
  uint32_t mrow[4];       // fast path: byte q of mrow[t] = sub[t][q] + 128
  uint32_t mrow16[4];     // 16-bit pair path: byte q of mrow16[t] = sub[t][q] (signed)
  int32_t pair_ok;        // 1: the inspector's first tier keeps two 16-bit rows per register
  int32_t pair_slack;     // pair sweep: threshold rise kept before the stored values move
  int32_t trace_all;      // work order: predict every extension long (traced sweep for all)
  int32_t sub[16];
};

// Where one-sided extension `ext` (= 2 * seed + side, side 0 right, 1 left)
// reads its bases: window index w (1-based) sits at genomic position
// g0 + dir * w in each sequence.
struct Window {
  int64_t tg0, qg0;
  int dir;
  int32_t m, n;
  bool requested;
};

__device__ __forceinline__ Window make_window(const Params& p, uint32_t ext) {
  Window w;
  const fz_seed s = p.seeds[ext >> 1];
  const bool left = ext & 1u;
  w.requested = (s.side & (left ? FZ_SIDE_LEFT : FZ_SIDE_RIGHT)) != 0;
  const uint64_t tp = s.t_pos < p.t_len ? s.t_pos : p.t_len;
  const uint64_t qp = s.q_pos < p.q_len ? s.q_pos : p.q_len;
  const uint64_t ta = left ? tp : p.t_len - tp;
  const uint64_t qa = left ? qp : p.q_len - qp;
  w.m = (int32_t)(ta < (uint64_t)p.max_len ? ta : (uint64_t)p.max_len);
  w.n = (int32_t)(qa < (uint64_t)p.max_len ? qa : (uint64_t)p.max_len);
  w.dir = left ? -1 : 1;
  w.tg0 = left ? (int64_t)tp : (int64_t)tp - 1;
  w.qg0 = left ? (int64_t)qp : (int64_t)qp - 1;
  if (!w.requested) { w.m = 0; w.n = 0; }
  return w;
}

// 16 bases of a window starting at window index w: base w+k at bits 2k.
// Positions outside the sequence read as 0 (callers never score them).  The
// 16 bases span 5 bytes of the packed sequence; they are taken with two
// aligned 8-byte loads when both lie inside the sequence's bytes and the
// sequence is 8-byte aligned (device allocations are), else byte by byte.
__device__ __forceinline__ uint32_t fetch16(const uint8_t* __restrict__ s, uint64_t len, int64_t g0,
                                            int dir, int64_t w) {
  const int64_t lo = dir > 0 ? g0 + w : g0 - w - 15;   // lowest genomic position covered
  const int64_t b0 = lo >> 2;                           // floor division
  const int sh = (int)(lo & 3) * 2;
  const int64_t nbytes = (int64_t)((len + 3) >> 2);
  const int64_t a = b0 & ~int64_t(7);                   // aligned 8-byte word holding byte b0
  uint32_t fw;                                          // genomic lo .. lo+15, forward
  if (b0 >= 0 && a + 16 <= nbytes && ((uintptr_t)s & 7u) == 0u) {
    const uint64_t* q = reinterpret_cast<const uint64_t*>(s + a);
    const uint64_t w0 = __ldg(q), w1 = __ldg(q + 1);
    const int bs = 8 * (int)(b0 - a) + sh;              // bit offset of base lo in w1:w0, 0..62
    fw = (uint32_t)(bs ? (w0 >> bs) | (w1 << (64 - bs)) : w0);
  } else {
    uint64_t v = 0;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int64_t bi = b0 + k;
      const uint32_t byte = (bi >= 0 && bi < nbytes) ? (uint32_t)__ldg(s + bi) : 0u;
      v |= (uint64_t)byte << (8 * k);
    }
    fw = (uint32_t)(v >> sh);
  }
  if (dir > 0) return fw;
  const uint32_t r = __brev(fw);                        // reverse the order of the 2-bit fields
  return ((r >> 1) & 0x55555555u) | ((r & 0x55555555u) << 1);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// a * b + c as an integer multiply-add.  With b = Params::one (a runtime 1)
// the compiler keeps the multiply-add, which issues on the FMA pipe and
// leaves the ALU pipe (DPX max, byte permute, compares) to the rest of a cell.
__device__ __forceinline__ int32_t imad(int32_t a, int32_t b, int32_t c) {
  int32_t d;
  asm("mad.lo.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int32_t imax(int32_t a, int32_t b) { return a > b ? a : b; }
__device__ __forceinline__ int32_t imin(int32_t a, int32_t b) { return a < b ? a : b; }

// Prune threshold for an anti-diagonal from the best score of the completed
// ones.  ydrop = INF (or huge) clamps to TFLOOR, below every reachable score.
__device__ __forceinline__ int32_t threshold(int32_t best, int32_t ydrop) {
  if (ydrop < 0) return TFLOOR;
  const int64_t t = (int64_t)best - (int64_t)ydrop;
  return t < (int64_t)TFLOOR ? TFLOOR : (int32_t)t;
}

// Window checkpoint: the register-window sweep's complete state after one
// anti-diagonal, so that a sweep can resume there (a wider window after an
// overflow, or an executor segment).  One slot of CK_SLOT_WORDS int32:
//   header (CK_HDR words): anti-diagonal d, base row b, rows per lane K of the
//     writer, best score and its cell, last live anti-diagonal, flags, the
//     previous checkpoint of the same extension (+1, 0 = none), the high word
//     of lane 0's live-cell count, thresholds of anti-diagonals 0..32 (eager
//     corner), each lane's live-cell count so far;
//   then h, h of the previous anti-diagonal + (o + e - 128), I and D of the
//     window rows, CK_WIN_MAX words each, row u = lane * K + r stored at
//     r * 32 + lane (coalesced per slot).
// Target and query bases of each row are functions of (b, d) and are not stored.
constexpr int CK_HDR = 96;
constexpr int CK_WIN_MAX = 512;
constexpr int CK_SLOT_WORDS = CK_HDR + 4 * CK_WIN_MAX;   // 8,576 bytes
enum CkHdr : int {
  CK_D = 0, CK_B = 1, CK_K = 2, CK_BEST = 3, CK_BI = 4, CK_BJ = 5, CK_DLAST = 6, CK_FLAGS = 7,
  CK_PREV = 8, CK_CNT_HI = 11,
  CK_T = 12,     // CK_T .. CK_T + 32: thresholds
  CK_CNT = 48    // CK_CNT .. CK_CNT + 31: per-lane live-cell counts
};

// Trace arena layout of one executor extension: (d_end + 1) rows of `width`
// 4-bit cells (row d covers rows lo[d] .. lo[d] + width - 1 of anti-diagonal
// d), then (d_end + 1) int32 row origins.  Cell code: bits 0-1 S choice
// (0 diag, 1 I, 2 D), bit 2 I opens here, bit 3 D opens here.
// Every size is a multiple of 16 bytes, so each extension's base (a prefix sum
// of sizes) stays 16-byte aligned for the executor's 8-byte stores.
__host__ __device__ __forceinline__ uint64_t trace_lo_offset(uint32_t width, int32_t d_end) {
  const uint64_t rows = (uint64_t)d_end + 1;
  return (rows * (uint64_t)(width / 2) + 15) & ~uint64_t(15);
}
__host__ __device__ __forceinline__ uint64_t trace_bytes(uint32_t width, int32_t d_end) {
  const uint64_t rows = (uint64_t)d_end + 1;
  return trace_lo_offset(width, d_end) + ((rows * 4 + 15) & ~uint64_t(15));
}

}  // namespace fz
