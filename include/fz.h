/*
 * fz -- batched gapped seed extension on one GB300 (sm_103a).  C ABI.
 *
 * The method is the gapped extension stage of seed-and-extend whole-genome
 * alignment: from each seed anchor, a one-sided affine-gap (S/I/D) dynamic
 * program with y-drop pruning, followed by a traceback of the best cell
 * (FastZ: Accelerating Gapped Whole Genome Alignment on GPUs, sections 2.1,
 * 2.2 and 3.1-3.4).  A second mode runs an unpruned, zero-floored local fill
 * that returns the best score and its cell (the local recurrence of the DPX
 * intrinsics article, section 1.1, with affine gaps).
 *
 * Recurrence, for window cells (i, j) (i indexes the target, j the query):
 *   I(i,j) = max(I(i,j-1) - e, S(i,j-1) - o - e)
 *   D(i,j) = max(D(i-1,j) - e, S(i-1,j) - o - e)
 *   S(i,j) = max(S(i-1,j-1) + M[t_i][q_j], I(i,j), D(i,j))
 * with S(0,0) = 0; a gap of k bases costs o + k*e.  Anti-diagonals d = i + j
 * are swept in order; a cell on d is pruned when S < best - ydrop, best being
 * the maximum S over live cells of anti-diagonals < d; a cell with no live
 * predecessor is dead; the sweep ends when two consecutive anti-diagonals hold
 * no live cell.  The result is the maximum live S (ties: smallest i + j, then
 * smallest i) and the traceback from it (ties: diagonal > I > D; a gap opens
 * rather than extends on a tie).
 *
 * All device pointers are caller-owned device memory unless stated; every
 * call is asynchronous on the given CUDA stream except where a host read-back
 * is documented.  No function throws; errors are status codes, and
 * fz_last_error() gives a one-line message for the context.
 */
#ifndef FZ_H
#define FZ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fz_ctx fz_ctx;

typedef enum {
    FZ_OK = 0,
    FZ_ERR_ARG = 1,     /* invalid argument (null, out of range, capacity too small) */
    FZ_ERR_OOM = 2,     /* device or host allocation failed; nothing leaked */
    FZ_ERR_CUDA = 3,    /* a CUDA runtime call failed */
    FZ_ERR_DEVICE = 4   /* a kernel reported an internal check failure */
} fz_status;

typedef enum {
    FZ_EXTEND = 0,      /* one-sided y-drop extension with traceback */
    FZ_LOCAL = 1        /* unpruned local fill, score and end cell only */
} fz_mode;

#define FZ_YDROP_INF (-1)   /* ydrop value meaning "never prune" */
#define FZ_SIDE_RIGHT 1u
#define FZ_SIDE_LEFT 2u
#define FZ_SIDE_BOTH 3u
#define FZ_MAX_LEN_LIMIT (1 << 20)

/* result flags */
#define FZ_FLAG_DONE 1u         /* extension was requested and computed */
#define FZ_FLAG_EAGER 2u        /* end cell inside the 16x16 corner: traced in the inspector */
#define FZ_FLAG_WIDE 4u         /* live band wider than the register window: general path */
#define FZ_FLAG_BIN_SHIFT 4     /* bits 4..7: executor bin 1..5 (0 = none) */

/* One seed anchor.  Right side: window t[t_pos ..], q[q_pos ..] (t[t_pos] is
 * window index 1).  Left side: window read backwards from t[t_pos-1],
 * q[q_pos-1].  Bases of the anchor itself are not scored. */
typedef struct {
    uint64_t t_pos, q_pos;
    uint32_t side;          /* FZ_SIDE_RIGHT, FZ_SIDE_LEFT or FZ_SIDE_BOTH */
} fz_seed;                  /* 24 bytes */

/* One per seed and side: out[2k] = right, out[2k+1] = left of seed k. */
typedef struct {
    int32_t score;          /* best live S (>= 0); 0 if not requested */
    int32_t t_end, q_end;   /* i*, j*: target / query bases consumed from the anchor */
    uint32_t cigar_off;     /* first run in the CIGAR arena */
    uint32_t cigar_len;     /* runs; each run is (len << 4) | op, op 0 = M, 1 = I, 2 = D,
                               in forward genomic order (right: anchor outward;
                               left: leftmost base first) */
    uint32_t flags;         /* FZ_FLAG_* */
} fz_result;                /* 24 bytes */

typedef struct {
    uint64_t live_cells;    /* live cells of all inspector sweeps (EXTEND) or m*n cells (LOCAL) */
    uint64_t exec_cells;    /* executor trace cells: anti-diagonals replayed x trace row width
                               (register-window path; live cells on the wide path) */
    uint32_t eager;         /* extensions traced back inside the inspector */
    uint32_t bin[5];        /* executor bins: max(i*, j*) <= 512, 2048, 8192, 32768, 131072
                               (eager + bins + traced = extensions) */
    uint32_t extensions;    /* one-sided extensions computed */
    uint32_t wide;          /* extensions that ran on the general (wide band) path */
    uint64_t trace_bytes;   /* executor direction-bit arena used */
    uint64_t cigar_runs;    /* CIGAR arena runs used */
    uint32_t launches;      /* kernels launched by the last batch */
    uint32_t profiled;      /* 1 if phase_ms holds device times (fz_set_profiling) */
    float phase_ms[6];      /* device time per phase: 0 inspector (register window;
                               after the traced sweep when that ran, see traced_ms),
                               1 inspector (wide band), 2 binning + scans, 3 executor,
                               4 CIGAR emission, 5 whole batch */
    uint32_t retried;       /* extensions whose live band outgrew the first register
                               window and resumed in the 512-row one */
    uint64_t exec_live_cells;   /* live cells the executor replayed (anti-diagonals
                               1 .. i* + j* of each executor extension) */
    uint32_t traced;        /* extensions traced back by the inspector's traced sweep
                               (predicted long; no executor replay) */
    float traced_ms;        /* device time of the work order and the traced sweep when
                               profiling (then phase_ms[0] excludes it) */
    uint64_t traced_live_cells;  /* live cells of the traced sweep (part of live_cells) */
} fz_stats;

/*
 * Create a context.  sub: 4x4 substitution scores, row = target base, column =
 * query base, order A, C, G, T (host memory, copied).  gap_open >= 0,
 * gap_extend >= 1, ydrop >= 0 or FZ_YDROP_INF, 1 <= max_len <= FZ_MAX_LEN_LIMIT
 * (window cap per side).  |score| bounds: max(|sub|, gap_open + gap_extend) *
 * (2 * max_len + 1) must stay below 2^28 (int32 DP without wrap-around).
 * The context owns its device scratch and arenas; the calling thread's current
 * device is used.  Each call also sets the library's general-band kernels'
 * dynamic shared-memory limit (a process-wide function attribute), always to
 * the same value whatever max_len, so contexts with different window caps
 * coexist.  Returns FZ_ERR_ARG on a bad parameter, FZ_ERR_OOM or
 * FZ_ERR_CUDA when the device refuses an allocation or a call (*out = NULL).
 */
fz_status fz_create(fz_ctx** out, const int32_t sub[16], int32_t gap_open, int32_t gap_extend,
                    int32_t ydrop, int32_t max_len, fz_mode mode);

/*
 * Extend every seed.  d_target2 / d_query2: 2-bit packed sequences (A=0, C=1,
 * G=2, T=3; base k at bits 2*(k%4) of byte k/4), t_len / q_len bases.
 * d_seeds: n_seeds anchors (t_pos <= t_len, q_pos <= q_len).  d_out: 2*n_seeds
 * results.  *d_cigar receives the device address of the context-owned CIGAR
 * arena (valid until the next call on this context or fz_destroy); LOCAL mode
 * emits no CIGAR.
 *
 * Stream use: kernels run on cuda_stream (a cudaStream_t; NULL = legacy
 * default stream).  EXTEND mode reads a few counters back to the host once per
 * call (to size the executor and CIGAR arenas), so it returns after the
 * inspector has finished; the executor and traceback are still asynchronous.
 * The inputs must stay valid until the stream has passed this call's work.
 */
fz_status fz_extend_batch(fz_ctx* ctx, const uint8_t* d_target2, uint64_t t_len,
                          const uint8_t* d_query2, uint64_t q_len, const fz_seed* d_seeds,
                          uint32_t n_seeds, fz_result* d_out, const uint32_t** d_cigar,
                          void* cuda_stream);

/*
 * Same computation from HOST buffers: copies the packed sequences and seeds to
 * context-owned device memory, runs fz_extend_batch, copies the results to
 * h_out (2*n_seeds) and the CIGAR runs to h_cigar, and synchronises the
 * stream before returning.  The runs are packed: extension x's runs are
 * h_cigar[h_out[x].cigar_off .. + h_out[x].cigar_len), extensions in order, and
 * *cigar_used is the number of runs written (the device entry's arena instead
 * keeps one worst-case slot per extension).  h_cigar may be NULL when
 * cigar_cap is 0.  If the CIGAR needs more than cigar_cap runs, the results
 * are still written, *cigar_used holds the size needed and FZ_ERR_ARG is
 * returned.  Host buffers may be pageable; page-locked buffers copy faster.
 */
fz_status fz_extend_batch_host(fz_ctx* ctx, const uint8_t* h_target2, uint64_t t_len,
                               const uint8_t* h_query2, uint64_t q_len, const fz_seed* h_seeds,
                               uint32_t n_seeds, fz_result* h_out, uint32_t* h_cigar,
                               uint64_t cigar_cap, uint64_t* cigar_used, void* cuda_stream);

/* One two-sided alignment per seed (fz_combine). */
typedef struct {
    int32_t score;          /* right score + left score */
    uint32_t cigar_len;     /* runs in the combined CIGAR */
    uint64_t t_start, q_start;   /* first aligned base: t_pos - left t_end, q_pos - left q_end */
    uint64_t t_end, q_end;       /* one past the last: t_pos + right t_end, q_pos + right q_end */
    uint64_t cigar_off;     /* first run in the combined CIGAR arena */
} fz_alignment;             /* 48 bytes */

/*
 * Combine the two one-sided results of every seed into one alignment (FastZ,
 * section 3.1.2: LASTZ joins the left and right extensions of a seed before it
 * filters the alignments).  The pages give no formula; this is the plain one:
 *   score = right score + left score (the anchor is a point between the two
 *           windows and scores nothing);
 *   span  = [t_pos - left t_end, t_pos + right t_end) and the same on the query;
 *   CIGAR = the left side's runs, then the right side's, both in forward genomic
 *           order, with the two runs that meet at the anchor merged into one
 *           when they are the same operation.
 * A side that was not requested (or is empty) contributes score 0, no bases and
 * no runs.
 * d_seeds: the n_seeds anchors given to fz_extend_batch; d_res: its 2*n_seeds
 * results; d_cigar: its CIGAR arena (device memory, caller- or context-owned,
 * unchanged; required for an EXTEND context, may be NULL for a LOCAL one,
 * whose results have no runs).  d_aln: n_seeds records (device, caller-owned).  *d_aln_cigar
 * receives the device address of the context-owned combined CIGAR arena,
 * packed in seed order and valid until the next fz_combine or fz_extend_batch
 * on this context, or fz_destroy.  Reads 8 bytes back to size that arena (so
 * it synchronises with cuda_stream once); the rest is asynchronous.
 * Errors: FZ_ERR_ARG for a NULL context or NULL pointers with n_seeds > 0.
 * Device memory: the combined arena grows as needed (FZ_ERR_OOM if it cannot).
 */
fz_status fz_combine(fz_ctx* ctx, const fz_seed* d_seeds, uint32_t n_seeds, const fz_result* d_res,
                     const uint32_t* d_cigar, fz_alignment* d_aln, const uint32_t** d_aln_cigar,
                     void* cuda_stream);

/* Counters of the last completed batch (synchronises the context's last stream). */
fz_status fz_get_stats(fz_ctx* ctx, fz_stats* out);

/*
 * Per-phase device timing: when on, each batch records CUDA events on its
 * stream around its phases and fz_get_stats() fills phase_ms.  Off by default
 * (events add a little host work per batch).
 */
fz_status fz_set_profiling(fz_ctx* ctx, int on);

/* One-line description of the last error on this context ("" if none). */
const char* fz_last_error(fz_ctx* ctx);

/* Frees all device memory of the context.  NULL is ignored. */
void fz_destroy(fz_ctx* ctx);

/*
 * Local fill without any allocation.  The papers this library follows have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory at run time -- for example code running under a caching
 * allocator or a host framework that forbids cudaMalloc/cudaFree on its hot
 * path, or a process that must not grow its footprint after start-up -- and so
 * cannot create an fz_ctx (a context owns device buffers and pinned memory).
 *
 * Computes exactly what fz_extend_batch computes for a FZ_LOCAL context with
 * the same sub / gap_open / gap_extend / max_len: one fz_result per seed and
 * side (score, t_end, q_end, flags; no CIGAR, cigar_off = cigar_len = 0).
 * The caller passes inputs and outputs in device memory, as for
 * fz_extend_batch.  Limits: 1 <= max_len <= 2048, sub entries in [-128, 127];
 * anything beyond returns FZ_ERR_ARG before touching the GPU.
 *
 * Scratch (the work counter and the per-warp strip spill rows, about 10 MB)
 * is one file-scope device array of the library: every GPU that loads the
 * library holds it until the process exits.  This function makes no
 * cudaMalloc, cudaFree or other allocating call.  With CUDA's lazy module
 * loading (the default) the driver loads the library's device code, array
 * included, the first time it is used on a device -- normally at the first
 * call of this function there -- and takes the 10 MB then; make that first
 * call at start-up, before any stream capture.
 *
 * The array's device address is looked up (cudaGetSymbolAddress, current
 * device) at every call made outside stream capture; a call on a capturing
 * stream reuses the address found by the last call outside capture on that
 * device (none yet: FZ_ERR_CUDA).  After cudaDeviceReset, make one call
 * outside capture before capturing again.
 *
 * Every call shares the one array and clears its work counter at the start,
 * so calls that overlap on the GPU (different streams, or host threads, on
 * the same device) race and must be serialised by the caller.  Asynchronous
 * on cuda_stream.  A CUDA error already pending when the call starts (left by
 * earlier work) is returned as FZ_ERR_CUDA and left pending; nothing is
 * launched then.
 */
fz_status fz_local_fill_noalloc(const int32_t sub[16], int32_t gap_open, int32_t gap_extend,
                                int32_t max_len, const uint8_t* d_target2, uint64_t t_len,
                                const uint8_t* d_query2, uint64_t q_len, const fz_seed* d_seeds,
                                uint32_t n_seeds, fz_result* d_out, void* cuda_stream);

/*
 * Two more dynamic programs on the same instructions (the DPX intrinsics
 * article, section 1.3: edit distance and dynamic time warping, like
 * alignment, take a minimum over three sources plus an add; section 4.1 times
 * a batch of 512 edit distances of 1024 x 1024 and 256 DTWs of 800 x 800).
 * Each pair k compares a[a_pos .. a_pos + a_len) with b[b_pos .. b_pos + b_len).
 */
typedef struct {
    uint64_t a_pos, b_pos;
    uint32_t a_len, b_len;      /* at most FZ_DP_MAX_LEN each */
} fz_pair;                      /* 24 bytes */
#define FZ_DP_MAX_LEN 4096

/*
 * Edit distance (Levenshtein: substitution, insertion and deletion cost 1) of
 * n_pairs pairs of 2-bit packed DNA slices (the layout of fz_extend_batch's
 * sequences; a_bases / b_bases bases in d_a2 / d_b2):
 *   D(i,0) = i, D(0,j) = j,
 *   D(i,j) = min(D(i-1,j) + 1, D(i,j-1) + 1, D(i-1,j-1) + [a_i != b_j]).
 * d_dist[k] = D(a_len, b_len), or -2 for a pair longer than FZ_DP_MAX_LEN or
 * outside its sequence.  All pointers are caller-owned device memory (d_pairs:
 * n_pairs records; d_dist: n_pairs int32).  Asynchronous on cuda_stream; no
 * allocation, no host synchronisation.  FZ_ERR_ARG for null pointers with
 * n_pairs > 0; FZ_ERR_CUDA if a CUDA error is pending when called (left
 * pending) or the launch fails.
 */
fz_status fz_edit_distance_batch(const uint8_t* d_a2, uint64_t a_bases, const uint8_t* d_b2, uint64_t b_bases,
                                 const fz_pair* d_pairs, uint32_t n_pairs, int32_t* d_dist, void* cuda_stream);

/*
 * Dynamic time warping of n_pairs pairs of int32 sample slices (d_x: x_len
 * samples, d_y: y_len), cell cost |x_i - y_j|:
 *   D(0,0) = 0, D(i,0) = D(0,j) = infinity for i, j >= 1,
 *   D(i,j) = |x_i - y_j| + min(D(i-1,j), D(i,j-1), D(i-1,j-1)).
 * d_cost[k] = D(a_len, b_len) (below 2^30); 0 when both slices are empty, -1
 * when exactly one is (no warping path), -2 for a pair longer than
 * FZ_DP_MAX_LEN, outside its sequence, or with a sample outside
 * [-32767, 32767].  Memory, streams and errors as fz_edit_distance_batch.
 */
fz_status fz_dtw_batch(const int32_t* d_x, uint64_t x_len, const int32_t* d_y, uint64_t y_len,
                       const fz_pair* d_pairs, uint32_t n_pairs, int32_t* d_cost, void* cuda_stream);

/*
 * Integer-pipe throughput microbenchmark (whole GPU, current device), written
 * to rates[0 .. FZ_INT_RATES-1]:
 *   0  DPX add-max __viaddmax_s32            op/s (one 32-bit lane each)
 *   1  DPX 3-way max __vimax3_s32            op/s
 *   2  32-bit add                            op/s
 *   3  32-bit max                            op/s
 *   4  DPX add-max __viaddmax_s16x2_relu     op/s (two 16-bit halves each)
 *   5  DPX 3-way max __vimax3_s16x2_relu     op/s
 *   6  packed 16-bit add __vadd2             op/s
 *   7  32-bit multiply-add by a runtime 1    op/s
 *   8  cells/s of the costed Gotoh cell in the 16-bit pair form (2 add-max,
 *      1 3-way max, 2 packed adds per two cells), independent cells
 *   9  cells/s of the costed Gotoh cell in 32-bit form (2 add-max, 1 3-way
 *      max, 2 multiply-adds per cell)
 *  10  cells/s of the costed cell of the traced pair sweep: the cell of rate 8
 *      plus its four direction tests (four packed subtractions per two cells)
 * Independent dependency chains per thread, every SM busy; synchronises the
 * device; allocates and frees a small output buffer.  Rates 8, 9 and 10 are
 * the measured integer-pipe rooflines of the extension sweeps.
 */
#define FZ_INT_RATES 11
fz_status fz_bench_int_rates(double rates[FZ_INT_RATES]);

/*
 * Whether a context created by fz_create with these arguments runs the first
 * inspector tier as the 16-bit pair sweep (two cells per 32-bit lane: two
 * window rows kept as 16-bit halves of each register, values relative to the
 * moving prune threshold, so that each DPX s16x2 instruction advances two
 * cells): mode FZ_EXTEND, every sub[k] in [-128, 127],
 * a finite ydrop with ydrop + 2048 + 4 (gap_open + gap_extend + max|sub|) <=
 * 30000, gap_open + gap_extend + max|sub| + 16 < 2048, and the environment
 * variable FZ_NO_PAIR unset or "0" (read at the call).  Returns 1 or 0 (0 for
 * a null sub).  Host only: no device, no allocation.  The roofline of the
 * dominant kernel depends on it (cells per lane and instruction).
 */
int fz_pair_sweep_used(const int32_t sub[16], int32_t gap_open, int32_t gap_extend, int32_t ydrop,
                       fz_mode mode);

#ifdef __cplusplus
}
#endif

#endif /* FZ_H */
