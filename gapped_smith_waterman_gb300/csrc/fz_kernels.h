// Kernel launchers of the fz library (host-side declarations).
#pragma once

#include <cuda_runtime.h>

#include "fz_dev.cuh"

namespace fz {

struct WorkArgs {
  const uint32_t* list;        // extension ids, or nullptr for 0 .. n_work-1
  uint32_t n_work;
  const uint32_t* n_work_dev;  // if set, the work count is read from device memory
  uint32_t* ovf_list;          // register-window inspector: extensions to retry wider
  uint32_t* ovf_count;
  uint32_t* counter;           // dynamic work counter, zeroed before the launch
  ExtRec* rec;
  uint32_t* wide_list;         // inspector: extensions whose band outgrew the register window
  uint32_t* wide_count;
  uint8_t* trace;              // executor: direction-code arena
  const uint64_t* trace_off;   // executor: byte offset per work item
  uint64_t trace_sub;          // executor: subtracted from trace_off (chunked runs)
  unsigned long long* live_total;
  unsigned long long* exec_total;
  unsigned long long* exec_live;   // executor: live cells replayed
  uint32_t* err;               // device error word (0 = fine)
  int32_t* scratch;            // wide path: per-block anti-diagonal buffers (bands wider than the ring)
  uint64_t scratch_stride;     // int32 elements per block
  // window checkpoints (register-window sweeps)
  int32_t* ckpt;               // pool of CK_SLOT_WORDS-word slots, or nullptr (none written)
  uint32_t ckpt_cap;           // slots in the pool
  uint32_t* ckpt_used;         // slot allocator (may run past ckpt_cap: then nothing is written)
  int32_t ckpt_every;          // write one every ckpt_every anti-diagonals (a power of two) ...
  int32_t ckpt_recent;         // ... while the best cell is at most this many anti-diagonals back
  int resume;                  // inspector: continue from the extension's newest checkpoint
  // executor: work items are segments {position in the executor list, start
  // checkpoint + 1 (0 = the origin), last anti-diagonal, first anti-diagonal};
  // list then holds the whole executor list and trace_off is indexed by position
  const uint4* seg;
  // traced pair sweep (inspector of the extensions predicted long): one trace
  // slot of tslot_bytes per resident warp (rows: tslot_rows x 256 B of flags,
  // then tslot_rows int32 window headers, then tslot_rows uint32 walk runs)
  uint8_t* tpool;
  uint64_t tslot_bytes;
  uint32_t tslot_rows;
  uint32_t tslots;             // slots in the pool: warps beyond them take no work
  uint32_t tring;              // ring checkpoints per slot (after the walk runs) ...
  uint32_t tring_every;        // ... one every tring_every anti-diagonals (a power of two)
  uint32_t* truns;             // traced-run arena (runs in forward genomic order)
  uint64_t truns_cap;
  unsigned long long* truns_used;   // runs asked for (may pass truns_cap: those go to the executor)
  const uint32_t* list_base_dev;    // plain pair sweep after the traced one: list offset (device)
  unsigned long long* traced_live;  // traced sweep: its live cells
};

// register-window sweep (extend_fast.cu)
// tier 0: 384-row window, tier 1: 512-row window
int fast_window_rows(int tier);
cudaError_t launch_inspect_fast(int tier, const Params& p, const WorkArgs& wa, int grid, cudaStream_t st);
cudaError_t launch_execute_fast(int tier, const Params& p, const WorkArgs& wa, int grid, cudaStream_t st);
// traced pair sweep (first tier, pair_ok only): list[0 .. *n_work_dev)
cudaError_t launch_inspect_traced(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st);
int traced_blocks_per_sm();
int extend_fast_blocks_per_sm(int tier, bool trace, bool pair);  // pair: the 16-bit first tier

// general band sweep (extend_wide.cu)
uint64_t wide_scratch_elems(int32_t max_len);   // per block
int wide_blocks_per_sm(int32_t max_len);         // 0 on failure (sets the kernels' shared-memory limit)
cudaError_t launch_inspect_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st);
cudaError_t launch_execute_wide(const Params& p, const WorkArgs& wa, int grid, cudaStream_t st);

// local fill (local.cu)
struct LocalArgs {
  uint32_t n_work;
  uint32_t* counter;
  ExtRec* rec;
  unsigned long long* live_total;
  int32_t* spill;              // global spill rows when not in shared memory
  uint64_t spill_stride;       // int32 elements per warp
  int use_smem;
  uint32_t mcol[4];            // byte t of mcol[q] = sub[t][q] + 128
};
int local_warps_per_block();
size_t local_smem_bytes(int32_t max_len);
cudaError_t launch_local(const Params& p, const LocalArgs& la, int grid, cudaStream_t st);
int local_blocks_per_sm(size_t smem);

// binning, scans and CIGAR emission (pipeline.cu)
struct PipeArgs {
  ExtRec* rec;
  uint32_t n_ext;
  uint32_t* ext_bin;           // per extension: 0 none / eager, 1..5 executor bin
  uint32_t* bin_count;         // [8]: 0 eager, 1..5 bins, 6 unused, 7 requested
  uint32_t* bin_cursor;        // [8]
  uint32_t* sub_count;         // [16]: bin 1 by the best cell's anti-diagonal, longest first
  uint32_t* sub_cursor;        // [16]
  uint32_t* exec_list;         // executor order: bins 5, 4, .., 1
  uint32_t* exec_pos;          // per extension: index in exec_list
  uint64_t* trace_sz;          // per exec item
  uint64_t* cig_cap;           // per extension
  uint32_t* err;
  int local;
  int32_t oe;                  // gap open + extend
  int32_t max_sub;             // max(0, largest substitution score)
};
cudaError_t launch_classify(const PipeArgs& a, cudaStream_t st);
// inspector work order: extensions predicted to align far (for the traced
// sweep) first, then by the number of homologous 32-base blocks near the anchor
// (key: per extension; hist, cursor: [34], zeroed; *n_long: the predicted ones,
// list[0 .. *n_long), or 0 when fewer than min_long are predicted)
cudaError_t launch_order(const Params& p, uint32_t n_ext, uint8_t* key, uint32_t* hist, uint32_t* cursor,
                         uint32_t* list, uint32_t* n_long, uint32_t min_long, cudaStream_t st);
cudaError_t launch_scatter(const PipeArgs& a, cudaStream_t st);
// exclusive scan of n uint64 values in place; total written to *total
uint32_t scan_launch_count(uint32_t n);   // kernels one launch_scan_u64 of n elements launches
cudaError_t launch_scan_u64(uint64_t* data, uint32_t n, uint64_t* block_tmp, uint64_t* total, cudaStream_t st);
uint32_t scan_tmp_elems(uint32_t n);

struct EmitArgs {
  const ExtRec* rec;
  const Params* dummy;
  uint32_t n_ext;
  const uint64_t* cig_off;     // per extension
  uint32_t* cigar;             // arena
  fz_result* out;
  const uint32_t* exec_list;
  const uint64_t* trace_off;   // per exec item
  const uint8_t* trace;
  uint64_t trace_sub;
  uint32_t exec_begin, exec_end;
  uint32_t exec_split;         // set by launch_emit_exec: [begin, split) walked by warps
  uint32_t long_blocks;        // set by launch_emit_exec
  uint32_t* err;
  int local;
  int32_t oe;
  int32_t max_sub;
  const uint32_t* truns;       // traced-run arena (k_emit_traced)
};
// executor segments from the checkpoint chains, one list per executor tier
// (0: 384-row window, 1: 512-row window, 2: wide band): nseg holds three
// arrays of n_max counts; item pos < *n_exec counts 1 + its checkpoints
// before the best cell's anti-diagonal in its tier's array.  Then, with
// seg_off the per-tier exclusive scans, the segments themselves (tier t's
// list starts at seg + base_t, base_0 = 0)
cudaError_t launch_seg_count(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                             const int32_t* ckpt, uint64_t* nseg, cudaStream_t st);
cudaError_t launch_seg_fill(const ExtRec* rec, const uint32_t* exec_list, uint32_t n_max, const uint32_t* n_exec,
                            const int32_t* ckpt, const uint64_t* seg_off, uint4* seg, uint64_t base1, uint64_t base2,
                            cudaStream_t st);

cudaError_t launch_emit_direct(const EmitArgs& a, cudaStream_t st);   // eager, empty, local, not requested
cudaError_t launch_emit_traced(const EmitArgs& a, cudaStream_t st);   // walked by the traced sweep
// executor items [exec_begin, exec_end); items before long_end (the bins of
// longer alignments) get a warp each, the rest a thread each
cudaError_t launch_emit_exec(EmitArgs a, uint32_t long_end, int sms, cudaStream_t st);

// CIGAR packing for host copies: lens[x] = out[x].cigar_len; then, with poff
// the exclusive scan of lens, runs copied to dst[poff[x]..] and cigar_off repointed
cudaError_t launch_cig_lens(const fz_result* out, uint32_t n, uint64_t* lens, cudaStream_t st);
cudaError_t launch_cig_pack(fz_result* out, uint32_t n, const uint64_t* poff, const uint32_t* src, uint32_t* dst,
                            cudaStream_t st);

// two-sided alignments: lens[k] = runs of seed k's combined CIGAR; then, with
// off the exclusive scan of lens, the combined records and runs (fz_combine in fz.h)
cudaError_t launch_comb_lens(const fz_result* res, uint32_t n_seeds, const uint32_t* cig, uint64_t* lens,
                             cudaStream_t st);
cudaError_t launch_comb(const fz_seed* seeds, uint32_t n_seeds, const fz_result* res, const uint32_t* cig,
                        const uint64_t* off, uint32_t* out_cig, fz_alignment* aln, cudaStream_t st);

// integer pipe microbenchmark (microbench.cu)
cudaError_t bench_int_rates(double rates[FZ_INT_RATES]);

}  // namespace fz
