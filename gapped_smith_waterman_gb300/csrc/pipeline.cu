// Device-side length binning, scans and CIGAR emission (sm_103a).
//
// Binning follows FastZ section 3.3: an extension whose best cell (i*, j*) lies
// outside the 16x16 eager corner goes to the smallest bin whose box contains it,
// boxes 512, 2048, 8192, 32768 (the paper's four) and 131072 (one more 4x step,
// as the paper allows).  The paper sorts on the host; here a block-local
// histogram and scatter build the executor's work list on the device, largest
// bin first so that the longest extensions start first.
#include <cuda_runtime.h>

#include <algorithm>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int TB = 256;

__device__ __forceinline__ uint32_t bin_of(int32_t i, int32_t j) {
  const int32_t mx = imax(i, j);
  return mx <= 512 ? 1u : mx <= 2048 ? 2u : mx <= 8192 ? 3u : mx <= 32768 ? 4u : 5u;
}

// Bin 1 is laid out by the best cell's anti-diagonal i + j (<= 1024), in 16
// buckets of 64, longest first: one thread walks each of its extensions, and a
// warp of walks of like length waits less for its longest one.
__device__ __forceinline__ uint32_t sub_of(int32_t i, int32_t j) {
  const int32_t b = (i + j) >> 6;
  return 15u - (uint32_t)(b > 15 ? 15 : b);
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

// ---- inspector order: likely long extensions first ----
//
// The inspector's warps take extensions from one work counter, so one long
// extension taken near the end of the batch sets the kernel's tail.  FastZ
// section 3.3 balances its executors by sorting on the inspected length; the
// inspector has no length yet, so it is predicted: lane k of a warp looks at
// the window's k-th 32-base block (bases 32k+1 .. 32k+32 of both sequences,
// k < 16) and calls it homologous when some diagonal offset of -8..8 (indels
// so far) matches at least 24 of the 32 bases; the key is the number of
// homologous blocks, and the work list runs from the highest key down.  Only
// the order of the work changes, never a result.
//
// The same pass predicts which extensions align far beyond the first 512
// bases, for the traced sweep (the inspector that also stores direction codes
// and walks its own best cell back, so that no executor replays it): one of
// the blocks 8..15 is homologous at some diagonal offset of -40..40 (the
// wider range follows the indels of a long alignment).  Predicted extensions
// get key 17 + count and so come first in the work list; the first *n_long
// entries of the list are exactly them.  A wrong prediction costs time only:
// both sweeps and the executor compute the same records.
constexpr int ORDER_BASE = 17;
constexpr int ORDER_KEYS = 2 * ORDER_BASE;
constexpr int LATE_FIRST = 8, LATE_OFF = 40;
constexpr int LATE_WORDS = (32 + 2 * LATE_OFF + 15) / 16 + 1;   // 16-base query words around a block

__device__ __forceinline__ uint32_t same_bases(uint32_t a, uint32_t b) {
  const uint32_t z = ~(a ^ b);
  return __popc(z & (z >> 1) & 0x55555555u);   // 2-bit fields that are equal
}

__global__ void k_order_key(Params p, uint32_t n_ext, uint8_t* key, uint32_t* hist) {
  __shared__ uint32_t h[ORDER_KEYS];
  if (threadIdx.x < ORDER_KEYS) h[threadIdx.x] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint32_t ext = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (ext < n_ext) {                                // warp-uniform
    const Window w = make_window(p, ext);
    uint32_t homologous = 0, late = 0;
    if (lane < 16 && w.requested && 32 * lane + 32 <= w.m && 32 * lane + 32 <= w.n) {
      const int64_t b0 = 32 * lane + 1;
      const uint32_t t0 = fetch16(p.t2, p.t_len, w.tg0, w.dir, b0);
      const uint32_t t1 = fetch16(p.t2, p.t_len, w.tg0, w.dir, b0 + 16);
      const uint32_t q0 = fetch16(p.q2, p.q_len, w.qg0, w.dir, b0 - 8);
      const uint32_t q1 = fetch16(p.q2, p.q_len, w.qg0, w.dir, b0 + 8);
      const uint32_t q2 = fetch16(p.q2, p.q_len, w.qg0, w.dir, b0 + 24);
      uint32_t best = 0;
#pragma unroll
      for (int s = 0; s <= 16; ++s) {               // query offset s - 8
        const uint32_t a0 = s < 16 ? __funnelshift_r(q0, q1, 2 * s) : q1;
        const uint32_t a1 = s < 16 ? __funnelshift_r(q1, q2, 2 * s) : q2;
        const uint32_t c = same_bases(t0, a0) + same_bases(t1, a1);
        best = c > best ? c : best;
      }
      homologous = best >= 24u ? 1u : 0u;
      if (lane >= LATE_FIRST) {
        // offsets -40..40: query bases b0 - 40 .. b0 + 71 in 16-base words
        uint32_t qw[LATE_WORDS + 1];
#pragma unroll
        for (int k = 0; k < LATE_WORDS; ++k) qw[k] = fetch16(p.q2, p.q_len, w.qg0, w.dir, b0 - LATE_OFF + 16 * k);
        qw[LATE_WORDS] = 0u;
        uint32_t lb = 0;
#pragma unroll
        for (int o = 0; o <= 2 * LATE_OFF; ++o) {       // query offset o - LATE_OFF
          const int wi = o >> 4, sh = o & 15;
          const uint32_t a0 = sh ? __funnelshift_r(qw[wi], qw[wi + 1], 2 * sh) : qw[wi];
          const uint32_t a1 = sh ? __funnelshift_r(qw[wi + 1], qw[wi + 2], 2 * sh) : qw[wi + 1];
          const uint32_t c = same_bases(t0, a0) + same_bases(t1, a1);
          lb = c > lb ? c : lb;
        }
        late = lb >= 24u ? 1u : 0u;
      }
    }
    const uint32_t k = __popc(__ballot_sync(FULL, homologous != 0u)) +
                       ((__ballot_sync(FULL, late != 0u) || p.trace_all) ? (uint32_t)ORDER_BASE : 0u);
    if (lane == 0) {
      key[ext] = (uint8_t)k;
      atomicAdd(&h[k], 1u);
    }
  }
  __syncthreads();
  if (threadIdx.x < ORDER_KEYS && h[threadIdx.x]) atomicAdd(&hist[threadIdx.x], h[threadIdx.x]);
}

// list[start(key) + rank] = ext, start(key) = extensions with a higher key;
// ranks are taken per block in shared memory, then one range per key and block
__global__ void k_order_scatter(uint32_t n_ext, const uint8_t* key, const uint32_t* hist, uint32_t* cursor,
                                uint32_t* list, uint32_t* n_long, uint32_t min_long) {
  __shared__ uint32_t start[ORDER_KEYS], count[ORDER_KEYS], base[ORDER_KEYS];
  if (threadIdx.x < ORDER_KEYS) count[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    uint32_t acc = 0;
    for (int k = ORDER_KEYS - 1; k >= 0; --k) {
      start[k] = acc;
      acc += hist[k];
      // predicted long: keys 17..33; too few to fill the traced sweep's warps
      // several times over leave them to the plain sweep and the executor
      // (the traced launch would last as long as its longest extension)
      // (or when they are at least half of the batch: then the plain sweep has
      // little left to do after it either)
      if (k == ORDER_BASE && blockIdx.x == 0 && n_long)
        *n_long = (acc >= min_long || 2ull * acc >= (uint64_t)n_ext) ? acc : 0u;
    }
  }
  __syncthreads();
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t k = 0, rank = 0;
  if (x < n_ext) {
    k = key[x];
    rank = atomicAdd(&count[k], 1u);
  }
  __syncthreads();
  if (threadIdx.x < ORDER_KEYS && count[threadIdx.x]) base[threadIdx.x] = atomicAdd(&cursor[threadIdx.x], count[threadIdx.x]);
  __syncthreads();
  if (x < n_ext) list[start[k] + base[k] + rank] = x;
}

__global__ void k_classify(PipeArgs a) {
  __shared__ uint32_t h[8], hs[16];
  if (threadIdx.x < 8) h[threadIdx.x] = 0;
  if (threadIdx.x < 16) hs[threadIdx.x] = 0;
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
        } else if (r.flags & FZ_XFLAG_TRACED) {
          atomicAdd(&h[6], 1u);                    // traced in the inspector: no executor
        } else {
          bin = bin_of(r.i_end, r.j_end);
          atomicAdd(&h[bin], 1u);
          if (bin == 1u) atomicAdd(&hs[sub_of(r.i_end, r.j_end)], 1u);
        }
      }
    }
    a.ext_bin[x] = bin;
    a.cig_cap[x] = cap;
  }
  __syncthreads();
  if (threadIdx.x < 8 && h[threadIdx.x]) atomicAdd(&a.bin_count[threadIdx.x], h[threadIdx.x]);
  if (threadIdx.x < 16 && hs[threadIdx.x]) atomicAdd(&a.sub_count[threadIdx.x], hs[threadIdx.x]);
}

// cursor[k] = first executor slot of bin k; bins are laid out 5, 4, 3, 2, 1
__global__ void k_bin_starts(PipeArgs a) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    uint32_t c = 0;
    for (int k = 5; k >= 1; --k) {
      a.bin_cursor[k] = c;
      if (k == 1)
        for (int s = 0; s < 16; ++s) {
          a.sub_cursor[s] = c;
          c += a.sub_count[s];
        }
      else
        c += a.bin_count[k];
    }
    a.bin_cursor[0] = c;   // executor items
  }
}

__global__ void k_scatter(PipeArgs a) {
  // slots 2..5: bins 2..5; slots 8..23: bin 1's length buckets
  __shared__ uint32_t cnt[24], base[24];
  if (threadIdx.x < 24) cnt[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t bin = 0, slot = 0, local_pos = 0;
  ExtRec r;
  if (x < a.n_ext) {
    bin = a.ext_bin[x];
    if (bin) {
      r = a.rec[x];
      slot = bin == 1u ? 8u + sub_of(r.i_end, r.j_end) : bin;
      local_pos = atomicAdd(&cnt[slot], 1u);
    }
  }
  __syncthreads();
  if (threadIdx.x >= 2 && threadIdx.x < 24 && (threadIdx.x <= 5 || threadIdx.x >= 8) && cnt[threadIdx.x])
    base[threadIdx.x] = atomicAdd(threadIdx.x >= 8 ? &a.sub_cursor[threadIdx.x - 8] : &a.bin_cursor[threadIdx.x],
                                  cnt[threadIdx.x]);
  __syncthreads();
  if (x < a.n_ext && bin) {
    const uint32_t pos = base[slot] + local_pos;
    a.exec_list[pos] = x;
    a.exec_pos[x] = pos;
    a.trace_sz[pos] = trace_bytes(r.width, r.i_end + r.j_end);
  }
}

// ---- executor segments ----
constexpr int CHAIN_MAX = 1 << 22;   // bound on a chain walk (a chain never holds a cycle)

// An executor extension is replayed in segments: from the origin to its first
// checkpoint, between consecutive checkpoints, and from its last checkpoint
// before the best cell's anti-diagonal d* to d*.  Checkpoints are linked
// newest first, so anti-diagonals decrease along a chain.
// Executor tier of an extension: 0 = 384-row window, 1 = 512-row window, 2 = wide band.
__device__ __forceinline__ int exec_tier(const ExtRec& r) {
  return (r.flags & FZ_FLAG_WIDE) ? 2 : (r.width == 32u * K_TIER0 ? 0 : 1);
}

// nseg holds three arrays of n_max counts, one per tier: item pos counts in
// its tier's array (0 in the others), so that each tier's segments form one
// list after a scan of its array.
__global__ void k_seg_count(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                            const int32_t* ck, uint64_t* nseg) {
  const uint32_t pos = blockIdx.x * blockDim.x + threadIdx.x;
  if (pos >= n_max) return;
  nseg[pos] = 0;
  nseg[n_max + pos] = 0;
  nseg[2ull * n_max + pos] = 0;
  if (pos >= *n_exec) return;
  const ExtRec r = rec[exec_list[pos]];
  const int32_t dstar = r.i_end + r.j_end;
  uint64_t cnt = 1;
  uint32_t h = ck ? r.ckpt : 0u;
  for (int guard = 0; h && guard < CHAIN_MAX; ++guard) {
    const int32_t* c = ck + (uint64_t)(h - 1) * CK_SLOT_WORDS;
    if (c[CK_D] < dstar) ++cnt;
    h = (uint32_t)c[CK_PREV];
  }
  nseg[(uint64_t)exec_tier(r) * n_max + pos] = cnt;
}

// seg = {position, start checkpoint + 1 (0 = origin), last anti-diagonal,
// first anti-diagonal}; tier t's segments start at seg + base[t]
__global__ void k_seg_fill(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                           const int32_t* ck, const uint64_t* seg_off, uint4* seg, uint64_t base1, uint64_t base2) {
  const uint32_t pos = blockIdx.x * blockDim.x + threadIdx.x;
  if (pos >= n_max || pos >= *n_exec) return;
  const ExtRec r = rec[exec_list[pos]];
  const int tier = exec_tier(r);
  const int32_t dstar = r.i_end + r.j_end;
  uint64_t at = (tier == 0 ? 0 : (tier == 1 ? base1 : base2)) + seg_off[(uint64_t)tier * n_max + pos];
  int32_t end = dstar;
  uint32_t h = ck ? r.ckpt : 0u;
  for (int guard = 0; h && guard < CHAIN_MAX; ++guard) {
    const int32_t* c = ck + (uint64_t)(h - 1) * CK_SLOT_WORDS;
    const int32_t dc = c[CK_D];
    if (dc < dstar) {
      seg[at++] = make_uint4(pos, h, (uint32_t)end, (uint32_t)dc);
      end = dc;
    }
    h = (uint32_t)c[CK_PREV];
  }
  seg[at] = make_uint4(pos, 0u, (uint32_t)end, 0u);
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

// A whole scan in one block (small arrays): chunks of SCAN_E elements in
// order, each scanned in the block and offset by the total of those before.
__global__ void __launch_bounds__(SCAN_T) k_scan_small(uint64_t* d, uint32_t n, uint64_t* total_out) {
  __shared__ uint64_t wt[32];
  uint64_t carry = 0;
  for (uint32_t c = 0; c < n; c += SCAN_E) {
    const uint32_t i0 = c + 2 * threadIdx.x;
    const uint64_t a = i0 < n ? d[i0] : 0, b = i0 + 1 < n ? d[i0 + 1] : 0;
    uint64_t total;
    const uint64_t ex = block_excl_scan(a + b, wt, total);
    if (i0 < n) d[i0] = carry + ex;
    if (i0 + 1 < n) d[i0 + 1] = carry + ex + a;
    carry += total;
    __syncthreads();                               // (wt is reused by the next chunk)
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
  __device__ void push_n(uint32_t o, uint32_t n) {   // n >= 1 ops of one kind
    if (o == op) { len += n; return; }
    flush();
    op = o;
    len = n;
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
  if (!(r.flags & FZ_FLAG_EAGER)) return;       // executor extension: k_emit_exec; traced: k_emit_traced
  const uint64_t off = a.cig_off[x];
  const uint64_t cap = cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub);
  RunWriter wr;
  wr.init(a.cigar, off, cap, (x & 1u) == 0u);
  for (uint32_t k = 0; k < r.npath; ++k) wr.push((uint32_t)(r.path >> (2 * k)) & 3u);
  wr.flush();
  if (wr.overflow) atomicOr(a.err, 16u);
  write_out(a.out + x, r, wr.nruns ? wr.first() : (uint32_t)off, wr.nruns, 0);
}

// Extensions the traced sweep walked: a warp per extension copies its runs
// (already in forward genomic order) from the traced-run arena to its CIGAR
// slot, where the run writer would have put them (right side: the slot's
// end, left side: its start), and writes its record with its size bin.
__global__ void k_emit_traced(EmitArgs a) {
  const uint32_t x = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (x >= a.n_ext) return;
  const ExtRec r = a.rec[x];
  if (!(r.flags & FZ_FLAG_DONE) || !(r.flags & FZ_XFLAG_TRACED) || a.local) return;
  const uint64_t off = a.cig_off[x];
  const uint64_t cap = cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub);
  const uint32_t nr = r.npath;
  if (nr > cap) {
    if (lane == 0) {
      atomicOr(a.err, 16u);
      write_out(a.out + x, r, (uint32_t)off, 0, bin_of(r.i_end, r.j_end));
    }
    return;
  }
  const uint64_t dst = (x & 1u) == 0u ? off + cap - nr : off;
  for (uint32_t k = lane; k < nr; k += 32) a.cigar[dst + k] = a.truns[r.path + k];
  if (lane == 0) write_out(a.out + x, r, (uint32_t)dst, nr, bin_of(r.i_end, r.j_end));
}

// One executor extension's walk state and trace rows.
struct Walk {
  const uint8_t* base;       // rows of W/2 bytes, anti-diagonal 0 first
  const int32_t* lo;         // row origin per anti-diagonal
  uint64_t bytes;            // size of this extension's trace block
  uint32_t W;
  int32_t i, j, st;
};

__device__ __forceinline__ void walk_init(const EmitArgs& a, uint32_t pos, const ExtRec& r, Walk& w) {
  const int32_t dend = r.i_end + r.j_end;
  w.W = r.width;
  w.base = a.trace + (a.trace_off[pos] - a.trace_sub);
  w.lo = reinterpret_cast<const int32_t*>(w.base + trace_lo_offset(w.W, dend));
  w.bytes = trace_bytes(w.W, dend);
  w.i = r.i_end;
  w.j = r.j_end;
  w.st = 0;
}

// One step of the walk from the code c of the current cell; returns false
// (with an error bit set) on an impossible code.
__device__ __forceinline__ bool walk_step(Walk& w, uint32_t c, RunWriter& wr, uint32_t* err) {
  if (w.st == 0) {
    const uint32_t sc = c & 3u;
    if (sc == 0) { wr.push(0); --w.i; --w.j; }
    else if (sc == 3) { atomicOr(err, 2u); return false; }
    else w.st = (int)sc;
  } else if (w.st == 1) {
    wr.push(1);
    w.st = (c & 4u) ? 0 : 1;
    --w.j;
  } else {
    wr.push(2);
    w.st = (c & 8u) ? 0 : 2;
    --w.i;
  }
  return true;
}

__device__ __forceinline__ void emit_done(const EmitArgs& a, uint32_t x, const ExtRec& r, RunWriter& wr,
                                          uint64_t off, int64_t guard) {
  if (guard <= 0) atomicOr(a.err, 4u);
  wr.flush();
  if (wr.overflow) atomicOr(a.err, 16u);
  write_out(a.out + x, r, wr.nruns ? wr.first() : (uint32_t)off, wr.nruns, a.local ? 0u : bin_of(r.i_end, r.j_end));
}

// Thread per extension: each step reads the row origin and the code byte.
__device__ void walk_thread(const EmitArgs& a, uint32_t pos) {
  const uint32_t x = a.exec_list[pos];
  const ExtRec r = a.rec[x];
  Walk w;
  walk_init(a, pos, r, w);
  const uint64_t off = a.cig_off[x];
  RunWriter wr;
  wr.init(a.cigar, off, cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub), (x & 1u) == 0u);
  int64_t guard = 2 * (int64_t)(r.i_end + r.j_end) + 4;
  while ((w.i > 0 || w.j > 0) && --guard > 0) {
    if (w.i < 0 || w.j < 0) { atomicOr(a.err, 1u); break; }
    const int32_t d = w.i + w.j;
    const int32_t u = w.i - w.lo[d];
    if (u < 0 || (uint32_t)u >= w.W) { atomicOr(a.err, 1u); break; }
    const uint32_t c = (w.base[(uint64_t)d * (w.W / 2) + (uint32_t)(u >> 1)] >> (4 * (u & 1))) & 15u;
    // The walk visits one row per step, going down in d: pull the row it will
    // reach PF anti-diagonals later (around where the path should be) and the
    // row origins further ahead into L2.  Addresses stay inside this
    // extension's rows.
    constexpr int32_t PF = 12;
    if (d >= PF) {
      const int32_t dp = d - PF;
      int32_t up = w.i - PF / 2 - w.lo[dp];
      up = up < 0 ? 0 : ((uint32_t)up >= w.W ? (int32_t)w.W - 1 : up);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(w.base + (uint64_t)dp * (w.W / 2) + (uint32_t)(up >> 1)));
      if (d >= 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(w.lo + (d - 64)));
    }
    if (!walk_step(w, c, wr, a.err)) break;
  }
  emit_done(a, x, r, wr, off, guard);
}

// Warp per extension, for long walks.  From the walker's cell (i, d = i + j)
// the next 32 anti-diagonals d, d-1, ..., d-31 can only be met in rows
// i-t .. i of anti-diagonal d-t (each step lowers i by at most the drop in d),
// at most 32 nibbles.  Lane t loads that row segment (5 aligned words) and the
// row origin into shared memory; lane 0 then walks through them, and the warp
// reloads once the walk leaves the 32 anti-diagonals.  A cell outside the
// loaded segment (only possible on a corrupt trace) is read from global memory.
constexpr int SEG_W = 5;

__device__ void walk_warp(const EmitArgs& a, uint32_t pos, int lane, uint32_t (*seg)[SEG_W], int32_t* seg_off,
                          int32_t* seg_lo) {
  const uint32_t x = a.exec_list[pos];
  const ExtRec r = a.rec[x];
  Walk w;
  walk_init(a, pos, r, w);
  const uint64_t off = a.cig_off[x];
  RunWriter wr;
  wr.init(a.cigar, off, cigar_cap(r.i_end, r.j_end, a.oe, a.max_sub), (x & 1u) == 0u);
  int64_t guard = 2 * (int64_t)(r.i_end + r.j_end) + 4;
  const uint32_t rowb = w.W / 2;
  const uintptr_t blk_lo = reinterpret_cast<uintptr_t>(w.base);
  const uintptr_t blk_hi = blk_lo + w.bytes;               // loads stay below this
  bool run = true;
  while (run) {
    // anchor of this batch, broadcast from the walker
    const int32_t iA = __shfl_sync(FULL, w.i, 0);
    const int32_t dA = __shfl_sync(FULL, w.i + w.j, 0);
    const int32_t dt = dA - lane;
    if (dt >= 0) {
      const int32_t lot = w.lo[dt];
      int32_t u0 = iA - lane - lot;
      u0 = u0 < 0 ? 0 : ((uint32_t)u0 >= w.W ? (int32_t)w.W - 1 : u0);
      const uintptr_t row = blk_lo + (uint64_t)dt * rowb;
      uintptr_t a0 = (row + (uint32_t)(u0 >> 1)) & ~uintptr_t(3);
      const uintptr_t amax = (blk_hi - 4 * SEG_W) & ~uintptr_t(3);
      if (a0 > amax) a0 = amax;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a0);
#pragma unroll
      for (int k = 0; k < SEG_W; ++k) seg[lane][k] = src[k];
      seg_off[lane] = (int32_t)(a0 - row);                  // byte offset of the segment in its row
      seg_lo[lane] = lot;
      // The next batch starts about 32 anti-diagonals lower and at most 33
      // rows lower: pull its row origins and, with this row's origin as the
      // guess, its row segments into L2 while lane 0 walks this batch.
      const int32_t dq = dt - 32;
      if (dq >= 0) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(w.lo + dq));
        int32_t uq = iA - 16 - lane - lot;
        uq = uq < 0 ? 0 : ((uint32_t)uq >= w.W ? (int32_t)w.W - 1 : uq);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(w.base + (uint64_t)dq * rowb + (uint32_t)(uq >> 1)));
      }
    }
    __syncwarp();
    // Walk this batch with the whole warp.  The walker's state (i, j, st) is
    // the same in every lane; lane k looks at the k-th cell of a run in the
    // current state's direction (diagonal in S, left in I, up in D), and one
    // ballot gives the run of moves that stays in the state.  Cells outside
    // the staged segments end a run; the walker's own cell is read from global
    // memory when it is not staged.
    for (;;) {
      if (!(w.i > 0 || w.j > 0)) { run = false; break; }
      if (--guard <= 0) { run = false; break; }
      if (w.i < 0 || w.j < 0) { if (lane == 0) atomicOr(a.err, 1u); run = false; break; }
      const int32_t t = dA - (w.i + w.j);
      if (t >= 32) break;                                   // left the loaded anti-diagonals
      int32_t ci, cj, ct;
      if (w.st == 0) { ci = w.i - lane; cj = w.j - lane; ct = t + 2 * lane; }
      else if (w.st == 1) { ci = w.i; cj = w.j - lane; ct = t + lane; }
      else { ci = w.i - lane; cj = w.j; ct = t + lane; }
      uint32_t c = 0;
      bool known = false, band = true;
      if (ct < 32 && ci >= 0 && cj >= 0) {
        const int32_t u = ci - seg_lo[ct];
        band = u >= 0 && (uint32_t)u < w.W;
        if (band) {
          const int32_t b = (u >> 1) - seg_off[ct];
          if (b >= 0 && b < 4 * SEG_W) {
            c = ((seg[ct][b >> 2] >> (8 * (b & 3))) >> (4 * (u & 1))) & 15u;
            known = true;
          } else if (lane == 0) {
            c = (w.base[(uint64_t)(w.i + w.j) * rowb + (uint32_t)(u >> 1)] >> (4 * (u & 1))) & 15u;
            known = true;
          }
        }
      }
      if (!__shfl_sync(FULL, band ? 1 : 0, 0)) { if (lane == 0) atomicOr(a.err, 1u); run = false; break; }
      const uint32_t c0 = __shfl_sync(FULL, c, 0);
      if (w.st == 0) {
        const uint32_t diag = __ballot_sync(FULL, known && (c & 3u) == 0u && ci >= 1 && cj >= 1);
        const int n = __ffs(~diag) - 1;                     // leading diagonal moves (-1: all 32)
        const int k = n < 0 ? 32 : n;
        if (k > 0) {
          if (lane == 0) wr.push_n(0, (uint32_t)k);
          w.i -= k;
          w.j -= k;
          continue;
        }
        const uint32_t sc = c0 & 3u;
        if (sc == 3u || sc == 0u) { if (lane == 0) atomicOr(a.err, sc == 3u ? 2u : 1u); run = false; break; }
        w.st = (int)sc;
      } else {
        // a run of gap moves: every cell pushes the gap op; the cell whose code
        // says the gap opens there returns the walk to S
        const uint32_t bit = w.st == 1 ? 4u : 8u;
        const bool valid = known && (w.st == 1 ? cj >= 1 : ci >= 1);
        const uint32_t vm = __ballot_sync(FULL, valid);
        const uint32_t om = __ballot_sync(FULL, valid && (c & bit) != 0u);
        const int nv = __ffs(~vm) - 1;
        const int nvalid = nv < 0 ? 32 : nv;                // cells from the walker's that can be used
        if (nvalid == 0) { if (lane == 0) atomicOr(a.err, 1u); run = false; break; }
        const int f = __ffs(om) - 1;                         // first opening cell, or -1
        const int k = (f >= 0 && f < nvalid) ? f + 1 : nvalid;
        if (lane == 0) wr.push_n((uint32_t)w.st, (uint32_t)k);
        if (w.st == 1) w.j -= k; else w.i -= k;
        if (f >= 0 && f < nvalid) w.st = 0;
      }
    }
    __syncwarp();
  }
  if (lane == 0) emit_done(a, x, r, wr, off, guard);
}

// ---- packing the CIGAR runs for a host copy ----
// The arena holds one slot per extension sized by cigar_cap; most slots are
// partly used.  For a copy to the host the runs are packed in extension order.
__global__ void k_cig_lens(const fz_result* out, uint32_t n, uint64_t* lens) {
  const uint32_t x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x < n) lens[x] = out[x].cigar_len;
}

// warp per extension: copy its runs to their packed offset and repoint the record
__global__ void k_cig_pack(fz_result* out, uint32_t n, const uint64_t* poff, const uint32_t* src, uint32_t* dst) {
  const uint32_t x = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (x >= n) return;
  const uint32_t len = out[x].cigar_len, from = out[x].cigar_off;
  const uint64_t to = poff[x];
  for (uint32_t k = lane; k < len; k += 32) dst[to + k] = src[(uint64_t)from + k];
  __syncwarp();
  if (lane == 0) out[x].cigar_off = (uint32_t)to;
}

// ---- two-sided alignments (fz_combine) ----
// runs of seed k's combined CIGAR: both sides' runs, one fewer when the two
// runs meeting at the anchor are the same operation
__device__ __forceinline__ uint32_t comb_runs(const fz_result& rr, const fz_result& rl, const uint32_t* cig,
                                              bool& merge) {
  const uint32_t nl = (rl.flags & FZ_FLAG_DONE) ? rl.cigar_len : 0u;
  const uint32_t nr = (rr.flags & FZ_FLAG_DONE) ? rr.cigar_len : 0u;
  merge = nl && nr && (cig[(uint64_t)rl.cigar_off + nl - 1] & 15u) == (cig[rr.cigar_off] & 15u);
  return nl + nr - (merge ? 1u : 0u);
}

__global__ void k_comb_lens(const fz_result* res, uint32_t n_seeds, const uint32_t* cig, uint64_t* lens) {
  const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n_seeds) return;
  bool merge;
  lens[k] = comb_runs(res[2 * k], res[2 * k + 1], cig, merge);
}

// warp per seed: the left runs, then the right runs; the two runs that meet at
// the anchor become one when they are the same operation
__global__ void k_comb(const fz_seed* seeds, uint32_t n_seeds, const fz_result* res, const uint32_t* cig,
                       const uint64_t* off, uint32_t* out_cig, fz_alignment* aln) {
  const uint32_t k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (k >= n_seeds) return;
  const fz_seed sd = seeds[k];
  const fz_result rr = res[2 * k], rl = res[2 * k + 1];
  const bool hr = (rr.flags & FZ_FLAG_DONE) != 0u, hl = (rl.flags & FZ_FLAG_DONE) != 0u;
  const uint32_t nl = hl ? rl.cigar_len : 0u, nr = hr ? rr.cigar_len : 0u;
  const uint64_t o = off[k];
  bool merge;
  const uint32_t total = comb_runs(rr, rl, cig, merge);
  const uint32_t first_r = nr ? cig[rr.cigar_off] : 0u;
  for (uint32_t q = lane; q < nl; q += 32) {
    uint32_t v = cig[(uint64_t)rl.cigar_off + q];
    if (merge && q == nl - 1) v += first_r & ~15u;     // add the right run's length
    out_cig[o + q] = v;
  }
  const uint32_t skip = merge ? 1u : 0u;
  for (uint32_t q = lane + skip; q < nr; q += 32) out_cig[o + nl + q - skip] = cig[(uint64_t)rr.cigar_off + q];
  if (lane == 0) {
    fz_alignment a;
    a.score = (hr ? rr.score : 0) + (hl ? rl.score : 0);
    a.cigar_len = total;
    a.t_start = sd.t_pos - (uint64_t)(hl ? rl.t_end : 0);
    a.q_start = sd.q_pos - (uint64_t)(hl ? rl.q_end : 0);
    a.t_end = sd.t_pos + (uint64_t)(hr ? rr.t_end : 0);
    a.q_end = sd.q_pos + (uint64_t)(hr ? rr.q_end : 0);
    a.cigar_off = o;
    aln[k] = a;
  }
}

// Blocks [0, long_blocks): one warp per item of [exec_begin, exec_split), the
// long walks (the executor list holds the largest bins first).  The other
// blocks: one thread per item of [exec_split, exec_end).
constexpr int EMIT_T = 128;

__global__ void __launch_bounds__(EMIT_T) k_emit_exec(EmitArgs a) {
  __shared__ uint32_t seg[EMIT_T / 32][32][SEG_W];
  __shared__ int32_t seg_off[EMIT_T / 32][32], seg_lo[EMIT_T / 32][32];
  if (blockIdx.x < a.long_blocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t nw = a.long_blocks * (EMIT_T / 32);
    for (uint32_t pos = a.exec_begin + blockIdx.x * (EMIT_T / 32) + warp; pos < a.exec_split; pos += nw)
      walk_warp(a, pos, lane, seg[warp], seg_off[warp], seg_lo[warp]);
    return;
  }
  const uint32_t pos = a.exec_split + (blockIdx.x - a.long_blocks) * EMIT_T + threadIdx.x;
  if (pos < a.exec_end) walk_thread(a, pos);
}

}  // namespace

cudaError_t launch_order(const Params& p, uint32_t n_ext, uint8_t* key, uint32_t* hist, uint32_t* cursor,
                         uint32_t* list, uint32_t* n_long, uint32_t min_long, cudaStream_t st) {
  if (n_ext == 0) return cudaSuccess;
  const uint32_t gk = (uint32_t)(((uint64_t)n_ext * 32 + TB - 1) / TB);
  k_order_key<<<gk, TB, 0, st>>>(p, n_ext, key, hist);
  k_order_scatter<<<(n_ext + TB - 1) / TB, TB, 0, st>>>(n_ext, key, hist, cursor, list, n_long, min_long);
  return cudaGetLastError();
}

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

uint32_t scan_launch_count(uint32_t n) {
  const uint32_t nb = (n + SCAN_E - 1) / SCAN_E;
  return nb == 0 ? 0u : (nb <= 16 ? 1u : 3u);
}

cudaError_t launch_scan_u64(uint64_t* data, uint32_t n, uint64_t* block_tmp, uint64_t* total, cudaStream_t st) {
  const uint32_t nb = (n + SCAN_E - 1) / SCAN_E;
  if (nb == 0) {
    cudaMemsetAsync(total, 0, sizeof(uint64_t), st);
    return cudaGetLastError();
  }
  if (nb <= 16) {                                  // up to 32,768 elements: one launch
    k_scan_small<<<1, SCAN_T, 0, st>>>(data, n, total);
    return cudaGetLastError();
  }
  k_scan1<<<nb, SCAN_T, 0, st>>>(data, n, block_tmp);
  k_scan2<<<1, SCAN_T, 0, st>>>(block_tmp, nb, total);
  k_scan3<<<nb, SCAN_T, 0, st>>>(data, n, block_tmp);
  return cudaGetLastError();
}

cudaError_t launch_seg_count(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                             const int32_t* ckpt, uint64_t* nseg, cudaStream_t st) {
  if (n_max) k_seg_count<<<(n_max + TB - 1) / TB, TB, 0, st>>>(rec, exec_list, n_max, n_exec, ckpt, nseg);
  return cudaGetLastError();
}

cudaError_t launch_seg_fill(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                            const int32_t* ckpt, const uint64_t* seg_off, uint4* seg, uint64_t base1, uint64_t base2,
                            cudaStream_t st) {
  if (n_max)
    k_seg_fill<<<(n_max + TB - 1) / TB, TB, 0, st>>>(rec, exec_list, n_max, n_exec, ckpt, seg_off, seg, base1, base2);
  return cudaGetLastError();
}

cudaError_t launch_emit_direct(const EmitArgs& a, cudaStream_t st) {
  const uint32_t g = (a.n_ext + TB - 1) / TB;
  if (g) k_emit_direct<<<g, TB, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_emit_traced(const EmitArgs& a, cudaStream_t st) {
  const uint64_t threads = (uint64_t)a.n_ext * 32;
  if (a.n_ext) k_emit_traced<<<(uint32_t)((threads + TB - 1) / TB), TB, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_cig_lens(const fz_result* out, uint32_t n, uint64_t* lens, cudaStream_t st) {
  if (n) k_cig_lens<<<(n + TB - 1) / TB, TB, 0, st>>>(out, n, lens);
  return cudaGetLastError();
}

cudaError_t launch_cig_pack(fz_result* out, uint32_t n, const uint64_t* poff, const uint32_t* src, uint32_t* dst,
                            cudaStream_t st) {
  const uint64_t threads = (uint64_t)n * 32;
  if (n) k_cig_pack<<<(uint32_t)((threads + TB - 1) / TB), TB, 0, st>>>(out, n, poff, src, dst);
  return cudaGetLastError();
}

cudaError_t launch_comb_lens(const fz_result* res, uint32_t n_seeds, const uint32_t* cig, uint64_t* lens,
                             cudaStream_t st) {
  if (n_seeds) k_comb_lens<<<(n_seeds + TB - 1) / TB, TB, 0, st>>>(res, n_seeds, cig, lens);
  return cudaGetLastError();
}

cudaError_t launch_comb(const fz_seed* seeds, uint32_t n_seeds, const fz_result* res, const uint32_t* cig,
                        const uint64_t* off, uint32_t* out_cig, fz_alignment* aln, cudaStream_t st) {
  const uint64_t threads = (uint64_t)n_seeds * 32;
  if (n_seeds) k_comb<<<(uint32_t)((threads + TB - 1) / TB), TB, 0, st>>>(seeds, n_seeds, res, cig, off, out_cig, aln);
  return cudaGetLastError();
}

cudaError_t launch_emit_exec(EmitArgs a, uint32_t long_end, int sms, cudaStream_t st) {
  a.exec_split = long_end < a.exec_begin ? a.exec_begin : (long_end > a.exec_end ? a.exec_end : long_end);
  const uint32_t n_long = a.exec_split - a.exec_begin, n_short = a.exec_end - a.exec_split;
  const uint32_t warps = EMIT_T / 32;
  const uint32_t cap = (uint32_t)(sms > 0 ? sms : 1) * 16;  // warp blocks: at most 16 per SM
  a.long_blocks = n_long ? std::min<uint32_t>((n_long + warps - 1) / warps, cap) : 0u;
  const uint32_t g = a.long_blocks + (n_short + EMIT_T - 1) / EMIT_T;
  if (g) k_emit_exec<<<g, EMIT_T, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fz
