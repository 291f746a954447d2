// Batched edit distance and dynamic time warping on the DPX instructions
// (sm_103a).  The DPX intrinsics article names both as the other dynamic
// programs its instructions serve (section 1.3: a minimum over three sources
// plus an add) and times them (section 4.1: edit distance 1024 x 1024 over
// 512 pairs, DTW 800 x 800 over 256 pairs).
//
// Edit distance (unit costs, 2-bit DNA):
//   D(i,0) = i, D(0,j) = j,
//   D(i,j) = min(min(D(i-1,j), D(i,j-1)) + 1, D(i-1,j-1) + [a_i != b_j])
//          = viaddmin(left, 1, viaddmin(up, 1, diag + mismatch))
// DTW (int32 samples, cell cost c = |x_i - y_j|):
//   D(0,0) = 0, D(i,0) = D(0,j) = infinity,
//   D(i,j) = c + min(D(i-1,j), D(i,j-1), D(i-1,j-1))
//          = viaddmin(left, c, min(up, diag) + c)
//
// One warp per pair, the local fill's wavefront: the b (column) sequence is
// cut into strips of 32 * KC columns; in a strip lane l owns KC consecutive
// columns and works on row i = tau - l + 1 at step tau, so a step needs only
// the value of the column left of its block (from lane l-1 by shuffle, one
// step old: the same row) and that column's value one row up (two steps
// old).  Lane 31 keeps the strip's last column per row in shared memory for
// the next strip's lane 0.  The a (row) element enters at lane 0 and moves
// one lane per step with the wavefront.
#include <cuda_runtime.h>

#include "fz_dev.cuh"
#include "fz_kernels.h"

namespace fz {

namespace {

constexpr int DW = 2;                  // warps per block
constexpr int KC = 32;                 // columns per lane
constexpr int SWD = 32 * KC;           // strip width
constexpr int32_t DINF = 1 << 30;      // DTW: no path (interior values stay below 2^30)
constexpr int32_t DP_BAD = -2;         // result of a pair beyond the limits

template <bool DTW>
struct Seqs {
  const void* a;                       // uint8_t 2-bit packed bases, or int32 samples
  const void* b;
  uint64_t a_len, b_len;
};

// Element k (0-based) of the pair's a or b slice: a base code, or a sample.
template <bool DTW>
__device__ __forceinline__ int32_t elem(const void* s, uint64_t len, uint64_t pos) {
  if (DTW) return pos < len ? __ldg(static_cast<const int32_t*>(s) + pos) : 0;
  return (int32_t)(fetch16(static_cast<const uint8_t*>(s), len, (int64_t)pos - 1, 1, 1) & 3u);
}

template <bool DTW>
__global__ void __launch_bounds__(DW * 32) k_dp(Seqs<DTW> sq, const fz_pair* pairs, uint32_t n_pairs,
                                                int32_t* out) {
  __shared__ int32_t s_spill[DW][FZ_DP_MAX_LEN + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t k = blockIdx.x * DW + warp;
  if (k >= n_pairs) return;                       // (warp-uniform; no block barrier follows)
  const fz_pair pr = pairs[k];
  const int32_t m = (int32_t)pr.a_len, n = (int32_t)pr.b_len;
  if (pr.a_len > FZ_DP_MAX_LEN || pr.b_len > FZ_DP_MAX_LEN || pr.a_pos + pr.a_len > sq.a_len ||
      pr.b_pos + pr.b_len > sq.b_len) {
    if (lane == 0) out[k] = DP_BAD;
    return;
  }
  if (m == 0 || n == 0) {
    if (lane == 0) out[k] = DTW ? (m == 0 && n == 0 ? 0 : -1) : m + n;
    return;
  }
  int32_t* sp = s_spill[warp];
  bool bad = false;                               // a DTW sample outside [-32767, 32767]
  int32_t result = 0;
  const int32_t nstrips = (n + SWD - 1) / SWD;
  for (int32_t s = 0; s < nstrips; ++s) {
    const int32_t c0 = s * SWD + lane * KC + 1;   // first column of this lane (1-based)
    int32_t col[KC];                              // column element: base code or sample
    int32_t dc[KC];                               // D of the lane's columns, previous row
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      const int32_t c = c0 + q;
      int32_t v = 0;
      if (c <= n) v = elem<DTW>(sq.b, sq.b_len, pr.b_pos + (uint64_t)(c - 1));
      if (DTW && (v < -32767 || v > 32767)) bad = true;
      col[q] = v;
      dc[q] = DTW ? DINF : c;                     // row 0
    }
    // edit: byte t of prof[q] is 1 unless t is the column's base (mismatch flags)
    uint32_t prof[KC];
    if (!DTW) {
#pragma unroll
      for (int q = 0; q < KC; ++q) prof[q] = 0x01010101u & ~(0xffu << (8 * col[q]));
    }
    // row 0: every lane starts with D(0, its last column), so that the next
    // lane's first step finds D(0, c0 - 1) as its diagonal; lane 0 starts
    // with D(0, c0 - 1) itself (D(0,0) = 0)
    int32_t left_out = DTW ? DINF : c0 + KC - 1;
    int32_t hh_prev = DTW ? (s == 0 ? 0 : DINF) : SWD * s;
    int32_t a_cur = 0;
    const bool last = s == nstrips - 1;
    for (int32_t tau = 0; tau < m + 31; ++tau) {
      const int32_t i = tau - lane + 1;
      int32_t hh = __shfl_up_sync(FULL, left_out, 1);     // D(i, c0 - 1)
      int32_t ab = __shfl_up_sync(FULL, a_cur, 1);        // row i's element
      if (lane == 0) {
        if (i >= 1 && i <= m) {
          ab = elem<DTW>(sq.a, sq.a_len, pr.a_pos + (uint64_t)(i - 1));
          if (DTW && (ab < -32767 || ab > 32767)) bad = true;
          hh = s == 0 ? (DTW ? DINF : i) : sp[i];
        }
      }
      if (i >= 1 && i <= m) {
        int32_t left = hh, diag = hh_prev;
#pragma unroll
        for (int q = 0; q < KC; ++q) {
          const int32_t up = dc[q];
          int32_t v;
          // Only the cell to the left is on the lane's dependent chain: the
          // minimum over the other two sources is formed off it, and one
          // add-min joins the left one (the same values: min is associative,
          // and no sum nears 2^31)
          if (DTW) {
            const int32_t d = ab - col[q];
            const int32_t c = d < 0 ? -d : d;
            v = __viaddmin_s32(left, c, min(up, diag) + c);
          } else {
            const int32_t x = (int32_t)prmt(prof[q], 0u, 0x4440u | (uint32_t)ab);
            v = __viaddmin_s32(left, 1, __viaddmin_s32(up, 1, diag + x));
          }
          diag = up;
          dc[q] = v;
          left = v;
        }
        left_out = left;
        if (lane == 31 && !last) sp[i] = left;
        if (i == m && last && n >= c0 && n < c0 + KC) {
#pragma unroll
          for (int q = 0; q < KC; ++q)
            if (c0 + q == n) result = dc[q];
        }
      }
      hh_prev = hh;
      a_cur = ab;
    }
    __syncwarp();
  }
  const uint32_t owner = (uint32_t)(((n - 1) % SWD) / KC);   // lane holding column n in the last strip
  result = __shfl_sync(FULL, result, owner);
  bad = __any_sync(FULL, bad);
  if (lane == 0) out[k] = bad ? DP_BAD : result;
}

template <bool DTW>
fz_status launch_dp(const void* a, uint64_t a_len, const void* b, uint64_t b_len, const fz_pair* pairs,
                    uint32_t n_pairs, int32_t* out, void* stream) {
  if (n_pairs == 0) return FZ_OK;
  if (!pairs || !out || (a_len && !a) || (b_len && !b)) return FZ_ERR_ARG;
  if (n_pairs > 0x7fffffffu) return FZ_ERR_ARG;
  if (cudaPeekAtLastError() != cudaSuccess) return FZ_ERR_CUDA;   // an earlier error is the caller's
  Seqs<DTW> sq{a, b, a_len, b_len};
  const uint32_t grid = (n_pairs + DW - 1) / DW;
  k_dp<DTW><<<grid, DW * 32, 0, static_cast<cudaStream_t>(stream)>>>(sq, pairs, n_pairs, out);
  return cudaGetLastError() == cudaSuccess ? FZ_OK : FZ_ERR_CUDA;
}

}  // namespace

}  // namespace fz

extern "C" fz_status fz_edit_distance_batch(const uint8_t* d_a2, uint64_t a_bases, const uint8_t* d_b2,
                                            uint64_t b_bases, const fz_pair* d_pairs, uint32_t n_pairs,
                                            int32_t* d_dist, void* cuda_stream) {
  return fz::launch_dp<false>(d_a2, a_bases, d_b2, b_bases, d_pairs, n_pairs, d_dist, cuda_stream);
}

extern "C" fz_status fz_dtw_batch(const int32_t* d_x, uint64_t x_len, const int32_t* d_y, uint64_t y_len,
                                  const fz_pair* d_pairs, uint32_t n_pairs, int32_t* d_cost, void* cuda_stream) {
  return fz::launch_dp<true>(d_x, x_len, d_y, y_len, d_pairs, n_pairs, d_cost, cuda_stream);
}
