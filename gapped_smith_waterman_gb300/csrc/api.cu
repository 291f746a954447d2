// C ABI of the fz library: argument checks, context-owned device memory and
// the launch sequence of one batch (host side).
//
// EXTEND batch:  inspector (register window) -> inspector (wide band, only the
// extensions that outgrew the window) -> classify + bin scatter + scans ->
// [one read-back: bin counts, arena sizes] -> executor (both paths, chunked
// when the direction-code arena would exceed its cap) -> CIGAR emission.
// LOCAL batch:  local fill -> result records.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "fz_dev.cuh"
#include "fz_kernels.h"

using namespace fz;

namespace {

struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
  cudaError_t ensure(size_t need) {
    if (need <= bytes) return cudaSuccess;
    if (p) { cudaFree(p); p = nullptr; bytes = 0; }
    size_t b = need + need / 4 + 256;
    cudaError_t e = cudaMalloc(&p, b);
    if (e != cudaSuccess) { p = nullptr; (void)cudaGetLastError(); return e; }
    bytes = b;
    return cudaSuccess;
  }
  void release() { if (p) cudaFree(p); p = nullptr; bytes = 0; }
  template <class T> T* as() const { return static_cast<T*>(p); }
};

struct Counters {
  unsigned long long live_total;
  unsigned long long exec_total;
  uint64_t trace_total;
  uint64_t cig_total;
  uint64_t cig_packed;         // runs actually written (host-copy packing)
  uint64_t comb_total;         // runs of the combined two-sided CIGARs
  uint32_t work[8];            // dynamic work counters: 0..2 inspectors, 3..5 executors, 6 traced sweep
  uint32_t retry_count;        // extensions retried with the 512-row window
  uint32_t wide_count;
  uint32_t err;
  uint32_t bin_count[8];
  uint32_t bin_cursor[8];
  uint32_t ckpt_used;          // window checkpoint slots taken (may exceed the pool)
  uint32_t pad_;
  uint32_t order_hist[34];     // inspector order: extensions per key (17.. predicted long)
  uint32_t order_cursor[34];
  uint32_t n_long;             // extensions predicted long (the traced sweep's list)
  uint32_t pad2_;
  uint64_t seg_total[3];       // executor segments per tier (384 rows, 512 rows, wide)
  uint32_t sub_count[16];      // bin 1 by walk length (k_classify), longest first
  uint32_t sub_cursor[16];
  unsigned long long exec_live;   // live cells the executors replayed
  unsigned long long truns_used;  // runs the traced sweep asked for in its arena
  unsigned long long traced_live; // live cells of the traced sweep
};

constexpr uint64_t TRACE_CAP_DEFAULT = 1ull << 30;   // smallest executor arena cap before chunking

}  // namespace

struct fz_ctx {
  int device = 0;
  int sms = 0;
  fz_mode mode = FZ_EXTEND;
  Params p{};
  bool fast_ok = false;
  int32_t max_sub = 0;               // max(0, largest substitution score)
  uint32_t mcol[4] = {0, 0, 0, 0};
  std::string err;
  DevBuf rec, ext_bin, exec_list, exec_pos, trace_sz, cig_cap, scan_tmp, wide_list, retry_list, counters;
  DevBuf order_key, order_list;      // inspector work order (likely long extensions first)
  DevBuf cigar, cigar_packed, trace, scratch, spill;
  DevBuf ckpt, seg_cnt, seg;         // window checkpoints, executor segments
  DevBuf comb_off, comb_cig;         // two-sided alignments (fz_combine)
  DevBuf tpool, truns;               // traced sweep: per-warp trace slots, run arena
  bool traced_ok = false;            // the traced sweep may run (pair sweep on)
  uint64_t tpool_cap = 0;            // largest trace pool (30% of the free memory at creation)
  int grid_traced = 0;
  uint32_t tslot_rows = 0;
  uint64_t tslot_bytes = 0;
  uint32_t tring = 0, tring_every = 0;   // traced sweep: ring checkpoints per slot, interval
  uint64_t truns_demand = 0;         // runs the last batch's traced sweep asked for
  DevBuf in_t, in_q, in_seeds, out_res;
  Counters* h_cnt = nullptr;         // pinned
  cudaStream_t last_stream = nullptr;
  fz_stats stats{};
  bool have_batch = false;
  uint64_t trace_cap = TRACE_CAP_DEFAULT;
  uint64_t ckpt_slot_cap = 0;        // most checkpoint slots the pool may hold (0: none written)
  uint64_t ckpt_demand = 0;          // slots the last batch asked for (the pool grows to it)
  int32_t ckpt_every = 256;          // checkpoint interval in anti-diagonals (a power of two)
  int grid_fast[2] = {0, 0}, grid_fast_trace[2] = {0, 0}, grid_wide = 0, grid_local = 0;
  size_t local_smem = 0;
  bool local_use_smem = true;
  uint32_t launches = 0;
  bool profiling = false;
  cudaEvent_t ev[7] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  bool ev_set[7] = {false, false, false, false, false, false, false};
};

namespace {

fz_status fail(fz_ctx* c, fz_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return s;
}

#define CU(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) {                                                              \
      (void)cudaGetLastError();                                                           \
      return fail(ctx, e_ == cudaErrorMemoryAllocation ? FZ_ERR_OOM : FZ_ERR_CUDA,        \
                  "%s: %s", #call, cudaGetErrorString(e_));                               \
    }                                                                                     \
  } while (0)

bool fault_injected(const char* what) {
  const char* f = getenv("FZ_FAULT");
  return f && strcmp(f, what) == 0;
}

fz_status ensure_batch_buffers(fz_ctx* ctx, uint32_t n_ext) {
  const size_t n = std::max<uint32_t>(n_ext, 1);
  if (fault_injected("alloc")) return fail(ctx, FZ_ERR_OOM, "allocation failure injected by FZ_FAULT=alloc");
  CU(ctx->rec.ensure(n * sizeof(ExtRec)));
  CU(ctx->ext_bin.ensure(n * 4));
  CU(ctx->exec_list.ensure(n * 4));
  CU(ctx->exec_pos.ensure(n * 4));
  CU(ctx->trace_sz.ensure(n * 8));
  CU(ctx->cig_cap.ensure(n * 8));
  CU(ctx->scan_tmp.ensure((size_t)scan_tmp_elems((uint32_t)n) * 8));
  CU(ctx->wide_list.ensure(n * 4));
  CU(ctx->retry_list.ensure(n * 4));
  CU(ctx->order_key.ensure(n));
  CU(ctx->order_list.ensure(n * 4));
  CU(ctx->seg_cnt.ensure(3 * n * 8));
  CU(ctx->counters.ensure(sizeof(Counters)));
  if (ctx->mode == FZ_EXTEND) {
    const uint64_t per = wide_scratch_elems(ctx->p.max_len) * 4;
    CU(ctx->scratch.ensure((size_t)ctx->grid_wide * per));
  } else if (!ctx->local_use_smem) {
    const uint64_t per = 2ull * (ctx->p.max_len + 1) * 4;
    CU(ctx->spill.ensure((size_t)ctx->grid_local * local_warps_per_block() * per));
  }
  return FZ_OK;
}

// Phase boundary k (0 = batch start, 1 inspector, 2 wide inspector, 3 bins and
// scans, 4 executor, 5 emission) when profiling is on.
void mark(fz_ctx* ctx, int k, cudaStream_t st) {
  if (!ctx->profiling) return;
  if (cudaEventRecord(ctx->ev[k], st) == cudaSuccess) ctx->ev_set[k] = true;
}

fz_status check_device_error(fz_ctx* ctx) {
  if (ctx->h_cnt->err) return fail(ctx, FZ_ERR_DEVICE, "device check failed (code 0x%x)", ctx->h_cnt->err);
  return FZ_OK;
}

fz_status run_local(fz_ctx* ctx, const fz_seed* d_seeds, uint32_t n_seeds, fz_result* d_out, cudaStream_t st) {
  const uint32_t n_ext = 2 * n_seeds;
  Counters* dc = ctx->counters.as<Counters>();
  LocalArgs la{};
  la.n_work = n_ext;
  la.counter = &dc->work[0];
  la.rec = ctx->rec.as<ExtRec>();
  la.live_total = &dc->live_total;
  la.spill = ctx->spill.as<int32_t>();
  la.spill_stride = 2ull * (ctx->p.max_len + 1);
  la.use_smem = ctx->local_use_smem ? 1 : 0;
  memcpy(la.mcol, ctx->mcol, sizeof(la.mcol));
  mark(ctx, 0, st);
  CU(launch_local(ctx->p, la, ctx->grid_local, st));
  ctx->launches += 1;
  mark(ctx, 1, st);
  EmitArgs ea{};
  ea.rec = ctx->rec.as<ExtRec>();
  ea.n_ext = n_ext;
  ea.out = d_out;
  ea.err = &dc->err;
  ea.local = 1;
  CU(launch_emit_direct(ea, st));
  ctx->launches += 1;
  mark(ctx, 5, st);
  (void)d_seeds;
  return FZ_OK;
}

fz_status run_extend(fz_ctx* ctx, uint32_t n_seeds, fz_result* d_out, cudaStream_t st) {
  const uint32_t n_ext = 2 * n_seeds;
  Counters* dc = ctx->counters.as<Counters>();
  WorkArgs wa{};
  wa.rec = ctx->rec.as<ExtRec>();
  wa.wide_list = ctx->wide_list.as<uint32_t>();
  wa.wide_count = &dc->wide_count;
  wa.live_total = &dc->live_total;
  wa.exec_total = &dc->exec_total;
  wa.exec_live = &dc->exec_live;
  wa.err = &dc->err;
  wa.scratch = ctx->scratch.as<int32_t>();
  wa.scratch_stride = wide_scratch_elems(ctx->p.max_len);
  // window checkpoints: up to 4 per extension, within the pool cap
  if (ctx->ckpt_slot_cap && ctx->fast_ok) {
    const uint64_t slots = std::min<uint64_t>(std::max<uint64_t>(4ull * n_ext + 64, ctx->ckpt_demand),
                                              ctx->ckpt_slot_cap);
    CU(ctx->ckpt.ensure(slots * CK_SLOT_WORDS * sizeof(int32_t)));
    wa.ckpt = ctx->ckpt.as<int32_t>();
    wa.ckpt_cap = (uint32_t)std::min<uint64_t>(ctx->ckpt.bytes / (CK_SLOT_WORDS * sizeof(int32_t)), 0xffffff00ull);
    wa.ckpt_used = &dc->ckpt_used;
    wa.ckpt_every = ctx->ckpt_every;
    wa.ckpt_recent = ctx->ckpt_every / 4;
  }

  // 1. inspector
  mark(ctx, 0, st);
  if (ctx->fast_ok) {
    // 384-row window for every extension; retries with 512 rows; then the wide band
    // the traced sweep runs when at least 4 extensions per resident warp are
    // predicted long (testing: FZ_TRACE_MIN sets that number; FZ_TRACE_ALL
    // makes it 0)
    uint32_t min_long = ctx->traced_ok ? 4u * 4u * (uint32_t)ctx->grid_traced : 0xffffffffu;
    if (ctx->traced_ok && ctx->p.trace_all) min_long = 0;
    const char* tm = getenv("FZ_TRACE_MIN");
    if (ctx->traced_ok && tm) min_long = (uint32_t)strtoul(tm, nullptr, 10);
    CU(launch_order(ctx->p, n_ext, ctx->order_key.as<uint8_t>(), dc->order_hist, dc->order_cursor,
                    ctx->order_list.as<uint32_t>(), &dc->n_long, min_long, st));
    ctx->launches += 2;
    WorkArgs a = wa;
    a.list = ctx->order_list.as<uint32_t>();
    a.n_work = n_ext;
    a.counter = &dc->work[0];
    a.ovf_list = ctx->retry_list.as<uint32_t>();
    a.ovf_count = &dc->retry_count;
    const uint64_t tslots = std::min<uint64_t>((uint64_t)ctx->grid_traced * 4u, n_ext);
    if (ctx->traced_ok && tslots * ctx->tslot_bytes <= ctx->tpool_cap) {
      // the extensions predicted long (the head of the work list) run the traced
      // sweep, the rest the plain one
      CU(ctx->tpool.ensure(ctx->tslot_bytes * tslots));
      uint64_t want = std::max<uint64_t>(ctx->truns_demand + ctx->truns_demand / 4, 256ull * n_ext + 4096);
      // testing: FZ_TRUNS_CAP limits the arena (extensions beyond it go to the executor)
      const char* tc = getenv("FZ_TRUNS_CAP");
      if (tc) want = strtoull(tc, nullptr, 10);
      CU(ctx->truns.ensure(std::max<uint64_t>(want, 1) * 4));
      WorkArgs t = a;
      t.n_work_dev = &dc->n_long;
      t.counter = &dc->work[6];
      t.tpool = ctx->tpool.as<uint8_t>();
      t.tslot_bytes = ctx->tslot_bytes;
      t.tslot_rows = ctx->tslot_rows;
      t.tslots = (uint32_t)tslots;
      t.tring = ctx->tring;
      t.tring_every = ctx->tring_every;
      t.truns = ctx->truns.as<uint32_t>();
      t.truns_cap = tc ? want : ctx->truns.bytes / 4;
      t.truns_used = &dc->truns_used;
      t.traced_live = &dc->traced_live;
      CU(launch_inspect_traced(ctx->p, t, ctx->grid_traced, st));
      mark(ctx, 6, st);
      a.list_base_dev = &dc->n_long;
      ctx->launches += 1;
    }
    CU(launch_inspect_fast(0, ctx->p, a, ctx->grid_fast[0], st));
    WorkArgs b = wa;
    b.list = ctx->retry_list.as<uint32_t>();
    b.n_work = 0;
    b.n_work_dev = &dc->retry_count;
    b.counter = &dc->work[1];
    b.ovf_list = ctx->wide_list.as<uint32_t>();
    b.ovf_count = &dc->wide_count;
    b.resume = 1;                        // continue from the overflow checkpoint
    CU(launch_inspect_fast(1, ctx->p, b, ctx->grid_fast[1], st));
    mark(ctx, 1, st);
    wa.list = ctx->wide_list.as<uint32_t>();
    wa.counter = &dc->work[2];
    CU(launch_inspect_wide(ctx->p, wa, ctx->grid_wide, st));
    ctx->launches += 3;
  } else {
    // every extension takes the general path (scores outside the byte range)
    std::vector<uint32_t> ids(n_ext);
    for (uint32_t k = 0; k < n_ext; ++k) ids[k] = k;
    CU(cudaMemcpyAsync(ctx->wide_list.p, ids.data(), (size_t)n_ext * 4, cudaMemcpyHostToDevice, st));
    CU(cudaMemcpyAsync(&dc->wide_count, &n_ext, 4, cudaMemcpyHostToDevice, st));
    CU(cudaStreamSynchronize(st));
    mark(ctx, 1, st);
    wa.list = ctx->wide_list.as<uint32_t>();
    wa.counter = &dc->work[2];
    CU(launch_inspect_wide(ctx->p, wa, ctx->grid_wide, st));
    ctx->launches += 1;
  }
  mark(ctx, 2, st);

  // 2. bins, executor work list, arena offsets
  PipeArgs pa{};
  pa.rec = ctx->rec.as<ExtRec>();
  pa.n_ext = n_ext;
  pa.ext_bin = ctx->ext_bin.as<uint32_t>();
  pa.bin_count = dc->bin_count;
  pa.bin_cursor = dc->bin_cursor;
  pa.sub_count = dc->sub_count;
  pa.sub_cursor = dc->sub_cursor;
  pa.exec_list = ctx->exec_list.as<uint32_t>();
  pa.exec_pos = ctx->exec_pos.as<uint32_t>();
  pa.trace_sz = ctx->trace_sz.as<uint64_t>();
  pa.cig_cap = ctx->cig_cap.as<uint64_t>();
  pa.err = &dc->err;
  pa.local = 0;
  pa.oe = ctx->p.oe;
  pa.max_sub = ctx->max_sub;
  CU(cudaMemsetAsync(ctx->trace_sz.p, 0, (size_t)n_ext * 8, st));
  CU(launch_classify(pa, st));
  CU(launch_scatter(pa, st));
  CU(launch_scan_u64(pa.cig_cap, n_ext, ctx->scan_tmp.as<uint64_t>(), &dc->cig_total, st));
  CU(launch_scan_u64(pa.trace_sz, n_ext, ctx->scan_tmp.as<uint64_t>(), &dc->trace_total, st));
  // executor segments: count per executor item, then their offsets
  CU(launch_seg_count(pa.rec, pa.exec_list, n_ext, &dc->bin_cursor[0], wa.ckpt, ctx->seg_cnt.as<uint64_t>(), st));
  for (int t = 0; t < 3; ++t)
    CU(launch_scan_u64(ctx->seg_cnt.as<uint64_t>() + (size_t)t * n_ext, n_ext, ctx->scan_tmp.as<uint64_t>(),
                       &dc->seg_total[t], st));
  ctx->launches += 3 + 1 + 5 * scan_launch_count(n_ext);
  mark(ctx, 3, st);
  CU(cudaMemcpyAsync(ctx->h_cnt, dc, sizeof(Counters), cudaMemcpyDeviceToHost, st));
  CU(cudaStreamSynchronize(st));
  fz_status s = check_device_error(ctx);
  if (s != FZ_OK) return s;
  const Counters& hc = *ctx->h_cnt;
  uint32_t n_exec = 0;
  for (int k = 1; k <= 5; ++k) n_exec += hc.bin_count[k];
  // Walks of bins 5..2 come first and are walked by warps, bin 1's by one
  // thread each; a batch with at most 128 walks per SM gives every walk a
  // warp (one thread per walk would leave the SMs with too few warps to hide
  // the walk's dependent loads: 2,000 walks of 256 bp windows 0.22 -> 0.04 ms).
  const uint32_t long_end = n_exec <= (uint32_t)ctx->sms * 128u ? n_exec : n_exec - hc.bin_count[1];
  if (hc.cig_total >= (1ull << 32)) return fail(ctx, FZ_ERR_ARG, "CIGAR arena would exceed 2^32 runs; split the batch");
  CU(ctx->cigar.ensure(std::max<uint64_t>(hc.cig_total, 1) * 4));
  ctx->stats.trace_bytes = hc.trace_total;
  ctx->stats.cigar_runs = hc.cig_total;
  const uint64_t seg_base[4] = {0, hc.seg_total[0], hc.seg_total[0] + hc.seg_total[1],
                                hc.seg_total[0] + hc.seg_total[1] + hc.seg_total[2]};
  const uint64_t n_seg = seg_base[3];
  ctx->truns_demand = std::max<uint64_t>(ctx->truns_demand, hc.truns_used);
  ctx->stats.traced = hc.bin_count[6];
  if (wa.ckpt && hc.ckpt_used > wa.ckpt_cap)   // checkpoints were dropped: a larger pool next batch
    ctx->ckpt_demand = std::max<uint64_t>(ctx->ckpt_demand, (uint64_t)hc.ckpt_used + hc.ckpt_used / 4);
  if (n_exec) {
    CU(ctx->seg.ensure(std::max<uint64_t>(n_seg, 1) * sizeof(uint4)));
    CU(launch_seg_fill(pa.rec, pa.exec_list, n_ext, &dc->bin_cursor[0], wa.ckpt, ctx->seg_cnt.as<uint64_t>(),
                       ctx->seg.as<uint4>(), seg_base[1], seg_base[2], st));
    ctx->launches += 1;
  }

  // 3. executor + traceback, chunked by the arena cap
  std::vector<std::pair<uint32_t, uint32_t>> chunks;
  std::vector<uint64_t> toff, soff;          // per position: trace offset; per tier and position: first segment
  if (n_exec) {
    if (hc.trace_total <= ctx->trace_cap) {
      chunks.push_back({0u, n_exec});
      CU(ctx->trace.ensure(std::max<uint64_t>(hc.trace_total, 16)));
    } else {
      toff.resize(n_exec + 1);
      soff.resize(3 * ((size_t)n_exec + 1));
      CU(cudaMemcpy(toff.data(), ctx->trace_sz.p, (size_t)n_exec * 8, cudaMemcpyDeviceToHost));
      for (int t = 0; t < 3; ++t) {
        CU(cudaMemcpy(soff.data() + (size_t)t * (n_exec + 1), ctx->seg_cnt.as<uint64_t>() + (size_t)t * n_ext,
                      (size_t)n_exec * 8, cudaMemcpyDeviceToHost));
        soff[(size_t)t * (n_exec + 1) + n_exec] = hc.seg_total[t];
      }
      toff[n_exec] = hc.trace_total;
      uint32_t a = 0;
      while (a < n_exec) {
        uint32_t b = a + 1;
        // (a single extension larger than the cap is a chunk of its own; the
        // arena below grows to the largest chunk)
        while (b < n_exec && toff[b + 1] - toff[a] <= ctx->trace_cap) ++b;
        chunks.push_back({a, b});
        a = b;
      }
      uint64_t biggest = 16;
      for (auto& c : chunks) biggest = std::max<uint64_t>(biggest, toff[c.second] - toff[c.first]);
      CU(ctx->trace.ensure(biggest));
    }
  }
  EmitArgs ea{};
  ea.rec = ctx->rec.as<ExtRec>();
  ea.n_ext = n_ext;
  ea.cig_off = ctx->cig_cap.as<uint64_t>();
  ea.cigar = ctx->cigar.as<uint32_t>();
  ea.out = d_out;
  ea.exec_list = ctx->exec_list.as<uint32_t>();
  ea.trace_off = ctx->trace_sz.as<uint64_t>();
  ea.trace = ctx->trace.as<uint8_t>();
  ea.err = &dc->err;
  ea.local = 0;
  ea.oe = ctx->p.oe;
  ea.max_sub = ctx->max_sub;
  ea.truns = ctx->truns.as<uint32_t>();
  bool first_chunk = true;
  for (auto& c : chunks) {
    const uint64_t sub = toff.empty() ? 0 : toff[c.first];
    WorkArgs we = wa;
    we.list = ctx->exec_list.as<uint32_t>();    // segments name executor positions
    we.n_work_dev = nullptr;
    we.trace = ctx->trace.as<uint8_t>();
    we.trace_off = ctx->trace_sz.as<uint64_t>();
    we.trace_sub = sub;
    if (!first_chunk) CU(cudaMemsetAsync(&dc->work[3], 0, 3 * sizeof(uint32_t), st));
    first_chunk = false;
    for (int tier = 0; tier < 3; ++tier) {
      // this tier's segments of the chunk's positions
      const uint64_t* so = soff.empty() ? nullptr : soff.data() + (size_t)tier * (n_exec + 1);
      const uint64_t s0 = so ? so[c.first] : 0, s1 = so ? so[c.second] : hc.seg_total[tier];
      if (s1 == s0) continue;
      we.seg = ctx->seg.as<uint4>() + seg_base[tier] + s0;
      we.n_work = (uint32_t)(s1 - s0);
      we.counter = &dc->work[3 + tier];
      if (tier < 2) CU(launch_execute_fast(tier, ctx->p, we, ctx->grid_fast_trace[tier], st));
      else CU(launch_execute_wide(ctx->p, we, ctx->grid_wide, st));
      ctx->launches += 1;
    }
    if (chunks.size() > 1) {
      EmitArgs ex = ea;
      ex.exec_begin = c.first;
      ex.exec_end = c.second;
      ex.trace_sub = sub;
      CU(launch_emit_exec(ex, long_end, ctx->sms, st));
      ctx->launches += 1;
    }
  }
  mark(ctx, 4, st);
  CU(launch_emit_direct(ea, st));
  ctx->launches += 1;
  if (ctx->traced_ok && hc.bin_count[6]) {
    CU(launch_emit_traced(ea, st));
    ctx->launches += 1;
  }
  if (chunks.size() == 1) {
    EmitArgs ex = ea;
    ex.exec_begin = 0;
    ex.exec_end = n_exec;
    ex.trace_sub = 0;
    CU(launch_emit_exec(ex, long_end, ctx->sms, st));
    ctx->launches += 1;
  }
  mark(ctx, 5, st);
  ctx->stats.eager = hc.bin_count[0];
  for (int k = 0; k < 5; ++k) ctx->stats.bin[k] = hc.bin_count[k + 1];
  ctx->stats.wide = hc.wide_count;
  ctx->stats.retried = hc.retry_count;
  ctx->stats.extensions = hc.bin_count[7];
  return FZ_OK;
}

}  // namespace

namespace {

// The first tier runs as the 16-bit pair sweep when the scores fit in bytes,
// the y-drop is finite, the stored values (relative to the threshold - 2048)
// stay below ydrop + 2048 + 2 max|sub| with room for the rises kept back
// (slack, written to *slack), and a dead cell stays below the threshold after
// adding o + e + max sub; FZ_NO_PAIR=1 turns it off.
bool pair_rule(const int32_t sub[16], int32_t gap_open, int32_t gap_extend, int32_t ydrop, int32_t* slack) {
  int64_t smax = 0;
  bool bytes = true;
  for (int k = 0; k < 16; ++k) {
    smax = std::max<int64_t>(smax, std::llabs((long long)sub[k]));
    if (sub[k] < -128 || sub[k] > 127) bytes = false;
  }
  const int64_t oe = (int64_t)gap_open + gap_extend;
  const char* nop = getenv("FZ_NO_PAIR");
  const bool ok = bytes && ydrop != FZ_YDROP_INF && ydrop >= 0 && (int64_t)ydrop + 2048 + 4 * (oe + smax) <= 30000 &&
                  oe + smax + 16 < 2048 && !(nop && *nop && *nop != '0');
  if (slack) *slack = ok ? (int32_t)std::min<int64_t>(8192, 30000 - ((int64_t)ydrop + 2048 + 4 * (oe + smax))) : 0;
  return ok;
}

}  // namespace

extern "C" {

fz_status fz_create(fz_ctx** out, const int32_t sub[16], int32_t gap_open, int32_t gap_extend, int32_t ydrop,
                    int32_t max_len, fz_mode mode) {
  fz_ctx* ctx = nullptr;
  if (!out) return FZ_ERR_ARG;
  *out = nullptr;
  if (!sub || gap_open < 0 || gap_extend < 1 || (ydrop < 0 && ydrop != FZ_YDROP_INF) || max_len < 1 ||
      max_len > FZ_MAX_LEN_LIMIT || (mode != FZ_EXTEND && mode != FZ_LOCAL))
    return FZ_ERR_ARG;
  int64_t amax = (int64_t)gap_open + gap_extend;
  bool bytes = true;
  for (int k = 0; k < 16; ++k) {
    amax = std::max<int64_t>(amax, std::llabs((long long)sub[k]));
    if (sub[k] < -128 || sub[k] > 127) bytes = false;
  }
  if (amax * (2 * (int64_t)max_len + 1) >= (1ll << 28)) return FZ_ERR_ARG;
  if (mode == FZ_LOCAL && !bytes) return FZ_ERR_ARG;
  ctx = new (std::nothrow) fz_ctx();
  if (!ctx) return FZ_ERR_OOM;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    (void)cudaGetLastError();
    delete ctx;
    return FZ_ERR_CUDA;
  }
  ctx->mode = mode;
  Params& p = ctx->p;
  p.o = gap_open;
  p.e = gap_extend;
  p.oe = gap_open + gap_extend;
  p.ydrop = ydrop;
  p.max_len = max_len;
  p.one = 1;
  for (int k = 0; k < 16; ++k) {
    p.sub[k] = sub[k];
    ctx->max_sub = std::max(ctx->max_sub, sub[k]);
  }
  ctx->fast_ok = bytes;
  p.pair_ok = pair_rule(sub, gap_open, gap_extend, ydrop, &p.pair_slack) ? 1 : 0;
  for (int t = 0; t < 4; ++t) {
    uint32_t row = 0, col = 0;
    for (int q = 0; q < 4; ++q) {
      row |= (uint32_t)((bytes ? sub[t * 4 + q] : 0) + 128) << (8 * q);
      col |= (uint32_t)((bytes ? sub[q * 4 + t] : 0) + 128) << (8 * q);
    }
    p.mrow[t] = row;
    uint32_t row16 = 0;
    for (int q = 0; q < 4; ++q) row16 |= (uint32_t)((bytes ? sub[t * 4 + q] : 0) & 0xff) << (8 * q);
    p.mrow16[t] = row16;
    ctx->mcol[t] = col;
  }
  for (int tier = 0; tier < 2; ++tier) {
    ctx->grid_fast[tier] = ctx->sms * extend_fast_blocks_per_sm(tier, false, p.pair_ok != 0);
    ctx->grid_fast_trace[tier] = ctx->sms * extend_fast_blocks_per_sm(tier, true, false);
  }
  // wide path: one block per extension, as many as fit with the ring
  // (a failure shows as the pending error checked below)
  ctx->grid_wide = ctx->sms * std::max(1, wide_blocks_per_sm(max_len));
  {
    // traced sweep: one trace slot per resident warp (at most one per
    // extension of the batch), enough rows for the longest sweep
    // (anti-diagonals 0 .. 2 max_len); it runs when the pool fits in 30% of
    // the device memory free now (and FZ_TRACED is not "0")
    const char* tv = getenv("FZ_TRACED");
    const bool want = p.pair_ok && mode == FZ_EXTEND && !(tv && *tv == '0');
    ctx->grid_traced = ctx->sms * traced_blocks_per_sm();
    ctx->tslot_rows = (uint32_t)(2 * (int64_t)max_len + 2);
    ctx->tring_every = 1024;        // (set from the checkpoint interval below)
    ctx->tring = 0;
    ctx->tslot_bytes = 0;
    size_t fr = 0, tot = 0;
    if (cudaMemGetInfo(&fr, &tot) != cudaSuccess) fr = 0;
    (void)cudaGetLastError();
    ctx->tpool_cap = (uint64_t)(fr * 0.3);
    ctx->traced_ok = want;
    // every extension goes through the traced sweep when the windows are short
    // (max_len <= 1024: every sweep ends within 2048 anti-diagonals, so storing
    // its codes costs less than a separate executor pass; 256 bp windows:
    // 0.71 -> 0.60 ms per batch of 2,000), or with FZ_TRACE_ALL=1 (testing)
    const char* ta = getenv("FZ_TRACE_ALL");
    p.trace_all = (ctx->traced_ok && ((ta && *ta && *ta != '0') || max_len <= 1024)) ? 1 : 0;
  }
  ctx->local_smem = local_smem_bytes(max_len);
  ctx->local_use_smem = ctx->local_smem <= 200 * 1024;
  ctx->grid_local = ctx->sms * local_blocks_per_sm(ctx->local_use_smem ? ctx->local_smem : 0);
  if (cudaMallocHost(&ctx->h_cnt, sizeof(Counters)) != cudaSuccess) {
    (void)cudaGetLastError();
    delete ctx;
    return FZ_ERR_OOM;
  }
  memset(ctx->h_cnt, 0, sizeof(Counters));
  if (cudaGetLastError() != cudaSuccess) {
    cudaFreeHost(ctx->h_cnt);
    delete ctx;
    return FZ_ERR_CUDA;
  }
  {
    // executor arena cap: 40% of the device memory free now (chunks beyond it)
    size_t fr = 0, tot = 0;
    if (cudaMemGetInfo(&fr, &tot) == cudaSuccess)
      ctx->trace_cap = std::max<uint64_t>(TRACE_CAP_DEFAULT, (uint64_t)(fr * 0.4));
    (void)cudaGetLastError();
  }
  const char* cap = getenv("FZ_TRACE_CAP");
  if (cap) ctx->trace_cap = std::max<uint64_t>(strtoull(cap, nullptr, 10), 4096);
  {
    // checkpoint pool cap: 10% of the device memory free now
    size_t fr = 0, tot = 0;
    if (cudaMemGetInfo(&fr, &tot) == cudaSuccess)
      ctx->ckpt_slot_cap = (uint64_t)(fr * 0.1) / (CK_SLOT_WORDS * sizeof(int32_t));
    (void)cudaGetLastError();
  }
  const char* cks = getenv("FZ_CKPT_SLOTS");
  if (cks) ctx->ckpt_slot_cap = strtoull(cks, nullptr, 10);
  // checkpoint interval: 256 anti-diagonals, longer for long windows so that
  // an extension holds at most ~64 checkpoints
  while (ctx->ckpt_every < (1 << 20) && (int64_t)ctx->ckpt_every * 64 < 2 * (int64_t)max_len) ctx->ckpt_every <<= 1;
  const char* cke = getenv("FZ_CKPT_EVERY");
  if (cke) {
    const long v = strtol(cke, nullptr, 10);
    int32_t e = 32;
    while (e < v && e < (1 << 20)) e <<= 1;   // a power of two, at least 32
    ctx->ckpt_every = e;
  }
  // traced sweep slots: flag rows, window headers, walk runs, then the ring of
  // checkpoints (one every 4 checkpoint intervals) that only an overflow uses
  ctx->tring_every = (uint32_t)ctx->ckpt_every * 4u;
  ctx->tring = (ctx->tslot_rows + ctx->tring_every - 1) / ctx->tring_every;
  ctx->tslot_bytes = ((uint64_t)ctx->tslot_rows * 264u + (uint64_t)ctx->tring * CK_SLOT_WORDS * 4u + 255u) &
                     ~uint64_t(255);
  ctx->traced_ok = ctx->traced_ok && ctx->tslot_bytes <= ctx->tpool_cap;
  if (!ctx->traced_ok) ctx->p.trace_all = 0;
  *out = ctx;
  return FZ_OK;
}

fz_status fz_extend_batch(fz_ctx* ctx, const uint8_t* d_target2, uint64_t t_len, const uint8_t* d_query2,
                          uint64_t q_len, const fz_seed* d_seeds, uint32_t n_seeds, fz_result* d_out,
                          const uint32_t** d_cigar, void* cuda_stream) {
  if (!ctx) return FZ_ERR_ARG;
  ctx->err.clear();
  if (n_seeds && (!d_seeds || !d_out)) return fail(ctx, FZ_ERR_ARG, "null seeds or output with n_seeds > 0");
  if ((t_len && !d_target2) || (q_len && !d_query2)) return fail(ctx, FZ_ERR_ARG, "null sequence with nonzero length");
  if (n_seeds > 0x7fffffffu) return fail(ctx, FZ_ERR_ARG, "n_seeds too large");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  CU(cudaSetDevice(ctx->device));
  ctx->last_stream = st;
  ctx->stats = fz_stats{};
  ctx->have_batch = false;
  ctx->launches = 0;
  for (bool& b : ctx->ev_set) b = false;
  const uint32_t n_ext = 2 * n_seeds;
  fz_status s = ensure_batch_buffers(ctx, n_ext);
  if (s != FZ_OK) return s;
  if (d_cigar) *d_cigar = ctx->cigar.as<uint32_t>();
  CU(cudaMemsetAsync(ctx->counters.p, 0, sizeof(Counters), st));
  Params& p = ctx->p;
  p.t2 = d_target2;
  p.q2 = d_query2;
  p.t_len = t_len;
  p.q_len = q_len;
  p.seeds = d_seeds;
  p.n_seeds = n_seeds;
  if (n_seeds == 0) {
    ctx->have_batch = true;
    return FZ_OK;
  }
  s = ctx->mode == FZ_LOCAL ? run_local(ctx, d_seeds, n_seeds, d_out, st) : run_extend(ctx, n_seeds, d_out, st);
  if (s != FZ_OK) return s;
  if (d_cigar) *d_cigar = ctx->cigar.as<uint32_t>();
  ctx->have_batch = true;
  return FZ_OK;
}

fz_status fz_extend_batch_host(fz_ctx* ctx, const uint8_t* h_target2, uint64_t t_len, const uint8_t* h_query2,
                               uint64_t q_len, const fz_seed* h_seeds, uint32_t n_seeds, fz_result* h_out,
                               uint32_t* h_cigar, uint64_t cigar_cap, uint64_t* cigar_used, void* cuda_stream) {
  if (!ctx) return FZ_ERR_ARG;
  ctx->err.clear();
  if ((n_seeds && (!h_seeds || !h_out)) || (cigar_cap && !h_cigar))
    return fail(ctx, FZ_ERR_ARG, "null host buffer");
  if ((t_len && !h_target2) || (q_len && !h_query2)) return fail(ctx, FZ_ERR_ARG, "null sequence with nonzero length");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  CU(cudaSetDevice(ctx->device));
  const size_t tb = (t_len + 3) / 4, qb = (q_len + 3) / 4;
  CU(ctx->in_t.ensure(std::max<size_t>(tb, 16)));
  CU(ctx->in_q.ensure(std::max<size_t>(qb, 16)));
  CU(ctx->in_seeds.ensure(std::max<size_t>((size_t)n_seeds * sizeof(fz_seed), 16)));
  CU(ctx->out_res.ensure(std::max<size_t>((size_t)n_seeds * 2 * sizeof(fz_result), 16)));
  if (tb) CU(cudaMemcpyAsync(ctx->in_t.p, h_target2, tb, cudaMemcpyHostToDevice, st));
  if (qb) CU(cudaMemcpyAsync(ctx->in_q.p, h_query2, qb, cudaMemcpyHostToDevice, st));
  if (n_seeds) CU(cudaMemcpyAsync(ctx->in_seeds.p, h_seeds, (size_t)n_seeds * sizeof(fz_seed), cudaMemcpyHostToDevice, st));
  const uint32_t* dc = nullptr;
  fz_status s = fz_extend_batch(ctx, ctx->in_t.as<uint8_t>(), t_len, ctx->in_q.as<uint8_t>(), q_len,
                                ctx->in_seeds.as<fz_seed>(), n_seeds, ctx->out_res.as<fz_result>(), &dc, cuda_stream);
  if (s != FZ_OK) return s;
  uint64_t used = 0;
  if (ctx->mode == FZ_EXTEND && n_seeds && ctx->stats.cigar_runs) {
    // pack the runs written (slots are sized for the worst case) so that only
    // they are copied; the records' cigar_off then index h_cigar
    const uint32_t n_ext = 2 * n_seeds;
    Counters* dcn = ctx->counters.as<Counters>();
    fz_result* d_out = ctx->out_res.as<fz_result>();
    CU(launch_cig_lens(d_out, n_ext, ctx->cig_cap.as<uint64_t>(), st));
    CU(launch_scan_u64(ctx->cig_cap.as<uint64_t>(), n_ext, ctx->scan_tmp.as<uint64_t>(), &dcn->cig_packed, st));
    CU(cudaMemcpyAsync(&ctx->h_cnt->cig_packed, &dcn->cig_packed, sizeof(uint64_t), cudaMemcpyDeviceToHost, st));
    CU(cudaStreamSynchronize(st));
    used = ctx->h_cnt->cig_packed;
    CU(ctx->cigar_packed.ensure(std::max<uint64_t>(used, 1) * 4));
    CU(launch_cig_pack(d_out, n_ext, ctx->cig_cap.as<uint64_t>(), dc, ctx->cigar_packed.as<uint32_t>(), st));
    ctx->launches += 2 + scan_launch_count(n_ext);
    dc = ctx->cigar_packed.as<uint32_t>();
  }
  if (n_seeds) CU(cudaMemcpyAsync(h_out, ctx->out_res.p, (size_t)n_seeds * 2 * sizeof(fz_result), cudaMemcpyDeviceToHost, st));
  if (cigar_used) *cigar_used = used;
  if (used && used <= cigar_cap) CU(cudaMemcpyAsync(h_cigar, dc, used * 4, cudaMemcpyDeviceToHost, st));
  CU(cudaStreamSynchronize(st));
  if (used > cigar_cap) return fail(ctx, FZ_ERR_ARG, "CIGAR needs %llu runs, buffer holds %llu",
                                    (unsigned long long)used, (unsigned long long)cigar_cap);
  return FZ_OK;
}

fz_status fz_combine(fz_ctx* ctx, const fz_seed* d_seeds, uint32_t n_seeds, const fz_result* d_res,
                     const uint32_t* d_cigar, fz_alignment* d_aln, const uint32_t** d_aln_cigar,
                     void* cuda_stream) {
  if (!ctx) return FZ_ERR_ARG;
  ctx->err.clear();
  if (n_seeds && (!d_seeds || !d_res || !d_aln || (!d_cigar && ctx->mode == FZ_EXTEND)))
    return fail(ctx, FZ_ERR_ARG, "null seeds, results, CIGAR arena or output");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  CU(cudaSetDevice(ctx->device));
  CU(ctx->counters.ensure(sizeof(Counters)));
  CU(ctx->comb_off.ensure(std::max<size_t>(n_seeds, 1) * 8));
  CU(ctx->scan_tmp.ensure((size_t)scan_tmp_elems(std::max<uint32_t>(n_seeds, 1)) * 8));
  Counters* dc = ctx->counters.as<Counters>();
  CU(launch_comb_lens(d_res, n_seeds, d_cigar, ctx->comb_off.as<uint64_t>(), st));
  CU(launch_scan_u64(ctx->comb_off.as<uint64_t>(), n_seeds, ctx->scan_tmp.as<uint64_t>(), &dc->comb_total, st));
  CU(cudaMemcpyAsync(&ctx->h_cnt->comb_total, &dc->comb_total, sizeof(uint64_t), cudaMemcpyDeviceToHost, st));
  CU(cudaStreamSynchronize(st));
  const uint64_t total = ctx->h_cnt->comb_total;
  CU(ctx->comb_cig.ensure(std::max<uint64_t>(total, 1) * 4));
  CU(launch_comb(d_seeds, n_seeds, d_res, d_cigar, ctx->comb_off.as<uint64_t>(), ctx->comb_cig.as<uint32_t>(),
                 d_aln, st));
  if (d_aln_cigar) *d_aln_cigar = ctx->comb_cig.as<uint32_t>();
  return FZ_OK;
}

fz_status fz_get_stats(fz_ctx* ctx, fz_stats* out) {
  if (!ctx || !out) return FZ_ERR_ARG;
  if (!ctx->have_batch) return fail(ctx, FZ_ERR_ARG, "no completed batch");
  CU(cudaSetDevice(ctx->device));
  CU(cudaStreamSynchronize(ctx->last_stream));
  CU(cudaMemcpy(ctx->h_cnt, ctx->counters.p, sizeof(Counters), cudaMemcpyDeviceToHost));
  fz_status s = check_device_error(ctx);
  ctx->stats.live_cells = ctx->h_cnt->live_total;
  ctx->stats.exec_cells = ctx->h_cnt->exec_total;
  ctx->stats.exec_live_cells = ctx->h_cnt->exec_live;
  ctx->stats.launches = ctx->launches;
  ctx->stats.profiled = 0;
  for (float& f : ctx->stats.phase_ms) f = 0.f;
  ctx->stats.traced_ms = 0.f;
  ctx->stats.traced_live_cells = ctx->h_cnt->traced_live;
  if (ctx->profiling && ctx->ev_set[0]) {
    ctx->stats.profiled = 1;
    int prev = 0;
    if (ctx->ev_set[6]) {          // the traced sweep ran first: phase 0 starts after it
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ctx->ev[0], ctx->ev[6]) == cudaSuccess) ctx->stats.traced_ms = ms;
      prev = 6;
    }
    for (int k = 1; k <= 5; ++k) {
      if (!ctx->ev_set[k]) continue;
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ctx->ev[prev], ctx->ev[k]) == cudaSuccess) ctx->stats.phase_ms[k - 1] = ms;
      prev = k;
    }
    float tot = 0.f;
    if (prev != 6 && cudaEventElapsedTime(&tot, ctx->ev[0], ctx->ev[prev]) == cudaSuccess) ctx->stats.phase_ms[5] = tot;
    (void)cudaGetLastError();
  }
  if (ctx->mode == FZ_LOCAL) {
    ctx->stats.extensions = 0;
  }
  *out = ctx->stats;
  return s;
}

fz_status fz_set_profiling(fz_ctx* ctx, int on) {
  if (!ctx) return FZ_ERR_ARG;
  CU(cudaSetDevice(ctx->device));
  if (on && !ctx->ev[0]) {
    for (int k = 0; k < 7; ++k) CU(cudaEventCreate(&ctx->ev[k]));
  }
  ctx->profiling = on != 0;
  return FZ_OK;
}

const char* fz_last_error(fz_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

void fz_destroy(fz_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  DevBuf* bufs[] = {&ctx->rec, &ctx->ext_bin, &ctx->exec_list, &ctx->exec_pos, &ctx->trace_sz, &ctx->cig_cap,
                    &ctx->scan_tmp, &ctx->wide_list, &ctx->retry_list, &ctx->counters, &ctx->cigar, &ctx->trace, &ctx->scratch,
                    &ctx->spill, &ctx->in_t, &ctx->in_q, &ctx->in_seeds, &ctx->out_res, &ctx->cigar_packed,
                    &ctx->ckpt, &ctx->seg_cnt, &ctx->seg, &ctx->comb_off, &ctx->comb_cig, &ctx->order_key,
                    &ctx->order_list};
  for (DevBuf* b : bufs) b->release();
  if (ctx->h_cnt) cudaFreeHost(ctx->h_cnt);
  for (cudaEvent_t& e : ctx->ev)
    if (e) cudaEventDestroy(e);
  delete ctx;
}

fz_status fz_bench_int_rates(double rates[FZ_INT_RATES]) {
  if (!rates) return FZ_ERR_ARG;
  return bench_int_rates(rates) == cudaSuccess ? FZ_OK : FZ_ERR_CUDA;
}

int fz_pair_sweep_used(const int32_t sub[16], int32_t gap_open, int32_t gap_extend, int32_t ydrop, fz_mode mode) {
  if (!sub || mode != FZ_EXTEND) return 0;
  return pair_rule(sub, gap_open, gap_extend, ydrop, nullptr) ? 1 : 0;
}

}  // extern "C"
