"""Thin ctypes binding of the fz C ABI (``include/fz.h``).

Argument marshalling only: every step of the extension runs in the CUDA
library ``_build/libfz.so``.  There is no CPU fallback; loading fails loudly
when the library has not been built.  Device buffers are passed as raw
pointers (``tensor.data_ptr()``), streams as ``torch.cuda.Stream.cuda_stream``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

FZ_OK, FZ_ERR_ARG, FZ_ERR_OOM, FZ_ERR_CUDA, FZ_ERR_DEVICE = range(5)
FZ_EXTEND, FZ_LOCAL = 0, 1
FZ_YDROP_INF = -1
FZ_FLAG_DONE, FZ_FLAG_EAGER, FZ_FLAG_WIDE = 1, 2, 4
FZ_FLAG_BIN_SHIFT = 4

SYMBOLS = ("fz_create", "fz_extend_batch", "fz_extend_batch_host", "fz_get_stats", "fz_set_profiling",
           "fz_last_error", "fz_destroy", "fz_bench_int_rates", "fz_local_fill_noalloc", "fz_combine",
           "fz_pair_sweep_used", "fz_edit_distance_batch", "fz_dtw_batch")

RESULT_DTYPE = np.dtype([("score", "<i4"), ("t_end", "<i4"), ("q_end", "<i4"), ("cigar_off", "<u4"),
                         ("cigar_len", "<u4"), ("flags", "<u4")])
assert RESULT_DTYPE.itemsize == 24


PAIR_DTYPE = np.dtype([("a_pos", "<u8"), ("b_pos", "<u8"), ("a_len", "<u4"), ("b_len", "<u4")])
assert PAIR_DTYPE.itemsize == 24
FZ_DP_MAX_LEN = 4096

ALIGNMENT_DTYPE = np.dtype([("score", "<i4"), ("cigar_len", "<u4"), ("t_start", "<u8"), ("q_start", "<u8"),
                            ("t_end", "<u8"), ("q_end", "<u8"), ("cigar_off", "<u8")])
assert ALIGNMENT_DTYPE.itemsize == 48


class FzStats(ctypes.Structure):
    _fields_ = [("live_cells", ctypes.c_uint64), ("exec_cells", ctypes.c_uint64), ("eager", ctypes.c_uint32),
                ("bin", ctypes.c_uint32 * 5), ("extensions", ctypes.c_uint32), ("wide", ctypes.c_uint32),
                ("trace_bytes", ctypes.c_uint64), ("cigar_runs", ctypes.c_uint64), ("launches", ctypes.c_uint32),
                ("profiled", ctypes.c_uint32), ("phase_ms", ctypes.c_float * 6),
                ("retried", ctypes.c_uint32), ("exec_live_cells", ctypes.c_uint64), ("traced", ctypes.c_uint32),
                ("traced_ms", ctypes.c_float), ("traced_live_cells", ctypes.c_uint64)]


class FzError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"fz status {status}: {msg}")
        self.status = status


_lib = None


def load(path: str | None = None, build_if_missing: bool = False):
    """Load libfz.so (raises if it is missing; never substitutes another path)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise FileNotFoundError(f"{path} not built; run __graft_entry__.build() or "
                                    f"python -m gapped_smith_waterman_gb300.build")
        _build.build()
    L = ctypes.CDLL(path)
    vp, u8p, u32p, u64p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64
    L.fz_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int]
    L.fz_create.restype = ctypes.c_int
    L.fz_extend_batch.argtypes = [vp, u8p, u64p, u8p, u64p, vp, ctypes.c_uint32, vp,
                                  ctypes.POINTER(ctypes.c_void_p), vp]
    L.fz_extend_batch.restype = ctypes.c_int
    L.fz_extend_batch_host.argtypes = [vp, vp, u64p, vp, u64p, vp, ctypes.c_uint32, vp, vp, u64p,
                                       ctypes.POINTER(ctypes.c_uint64), vp]
    L.fz_extend_batch_host.restype = ctypes.c_int
    L.fz_get_stats.argtypes = [vp, ctypes.POINTER(FzStats)]
    L.fz_get_stats.restype = ctypes.c_int
    L.fz_set_profiling.argtypes = [vp, ctypes.c_int]
    L.fz_set_profiling.restype = ctypes.c_int
    L.fz_last_error.argtypes = [vp]
    L.fz_last_error.restype = ctypes.c_char_p
    L.fz_destroy.argtypes = [vp]
    L.fz_destroy.restype = None
    L.fz_local_fill_noalloc.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, u8p, u64p, u8p, u64p, vp, ctypes.c_uint32, vp, vp]
    L.fz_local_fill_noalloc.restype = ctypes.c_int
    L.fz_combine.argtypes = [vp, vp, ctypes.c_uint32, vp, vp, vp, ctypes.POINTER(ctypes.c_void_p), vp]
    L.fz_combine.restype = ctypes.c_int
    L.fz_edit_distance_batch.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64,
                                         ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    L.fz_edit_distance_batch.restype = ctypes.c_int
    L.fz_dtw_batch.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_uint64,
                               ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    L.fz_dtw_batch.restype = ctypes.c_int
    L.fz_bench_int_rates.argtypes = [ctypes.POINTER(ctypes.c_double)]
    L.fz_bench_int_rates.restype = ctypes.c_int
    L.fz_pair_sweep_used.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int]
    L.fz_pair_sweep_used.restype = ctypes.c_int
    _lib = L
    return L


def _check(ctx, status):
    if status != FZ_OK:
        msg = fz_last_error(ctx) if ctx else ""
        raise FzError(status, msg)


def fz_create(sub, gap_open: int, gap_extend: int, ydrop: int, max_len: int, mode: int = FZ_EXTEND):
    L = load()
    arr = (ctypes.c_int32 * 16)(*[int(x) for x in np.asarray(sub, np.int64).reshape(16)])
    h = ctypes.c_void_p()
    _check(None, L.fz_create(ctypes.byref(h), arr, gap_open, gap_extend, ydrop, max_len, mode))
    return h


def fz_extend_batch(ctx, d_target2: int, t_len: int, d_query2: int, q_len: int, d_seeds: int, n_seeds: int,
                    d_out: int, stream: int = 0) -> int:
    """Returns the device address of the CIGAR arena."""
    cig = ctypes.c_void_p()
    _check(ctx, load().fz_extend_batch(ctx, d_target2, t_len, d_query2, q_len, d_seeds, n_seeds, d_out,
                                       ctypes.byref(cig), stream))
    return cig.value or 0


def fz_extend_batch_host(ctx, h_target2: np.ndarray, t_len: int, h_query2: np.ndarray, q_len: int,
                         h_seeds: np.ndarray, h_out: np.ndarray, h_cigar: np.ndarray, stream: int = 0) -> int:
    """Host-buffer entry; returns the CIGAR runs written (raises if h_cigar is too small)."""
    used = ctypes.c_uint64()
    n_seeds = len(h_seeds)
    assert h_out.dtype == RESULT_DTYPE and h_out.size >= 2 * n_seeds
    st = load().fz_extend_batch_host(ctx, h_target2.ctypes.data, t_len, h_query2.ctypes.data, q_len,
                                     h_seeds.ctypes.data, n_seeds, h_out.ctypes.data,
                                     h_cigar.ctypes.data if h_cigar.size else None, h_cigar.size,
                                     ctypes.byref(used), stream)
    _check(ctx, st)
    return int(used.value)


def fz_get_stats(ctx) -> FzStats:
    s = FzStats()
    _check(ctx, load().fz_get_stats(ctx, ctypes.byref(s)))
    return s


def fz_set_profiling(ctx, on: bool) -> None:
    _check(ctx, load().fz_set_profiling(ctx, 1 if on else 0))


def fz_last_error(ctx) -> str:
    r = load().fz_last_error(ctx)
    return r.decode() if r else ""


def fz_destroy(ctx) -> None:
    if ctx:
        load().fz_destroy(ctx)


def fz_local_fill_noalloc(sub, gap_open: int, gap_extend: int, max_len: int, d_target2: int, t_len: int,
                          d_query2: int, q_len: int, d_seeds: int, n_seeds: int, d_out: int, stream: int = 0) -> None:
    """Allocation-free local fill (results only; see include/fz.h)."""
    arr = (ctypes.c_int32 * 16)(*[int(x) for x in np.asarray(sub, np.int64).reshape(16)])
    _check(None, load().fz_local_fill_noalloc(arr, gap_open, gap_extend, max_len, d_target2, t_len, d_query2,
                                              q_len, d_seeds, n_seeds, d_out, stream))


def fz_combine(ctx, d_seeds: int, n_seeds: int, d_res: int, d_cigar: int, d_aln: int, stream: int = 0) -> int:
    """Two-sided alignments; returns the device address of the combined CIGAR arena."""
    cig = ctypes.c_void_p()
    _check(ctx, load().fz_combine(ctx, d_seeds, n_seeds, d_res, d_cigar or None, d_aln, ctypes.byref(cig), stream))
    return cig.value or 0


def fz_edit_distance_batch(d_a2: int, a_bases: int, d_b2: int, b_bases: int, d_pairs: int, n_pairs: int,
                           d_dist: int, stream: int = 0) -> None:
    """Edit distances of n_pairs pairs (fz.h); device pointers as ints."""
    _check(None, load().fz_edit_distance_batch(d_a2 or None, a_bases, d_b2 or None, b_bases, d_pairs or None,
                                               n_pairs, d_dist or None, stream or None))


def fz_dtw_batch(d_x: int, x_len: int, d_y: int, y_len: int, d_pairs: int, n_pairs: int, d_cost: int,
                 stream: int = 0) -> None:
    """Dynamic time warping costs of n_pairs pairs (fz.h); device pointers as ints."""
    _check(None, load().fz_dtw_batch(d_x or None, x_len, d_y or None, y_len, d_pairs or None, n_pairs,
                                     d_cost or None, stream or None))


def dp_pairs_device(kind: str, a, b, pairs, device="cuda"):
    """Runs fz_edit_distance_batch (kind "edit", a and b base codes) or
    fz_dtw_batch (kind "dtw", a and b int32 samples) on device copies of the
    inputs; returns the int32 results on the host."""
    import torch
    from .workloads import pack2
    dev = torch.device(device)
    if kind == "edit":
        da = torch.from_numpy(pack2(np.asarray(a, np.uint8))).to(dev)
        db = torch.from_numpy(pack2(np.asarray(b, np.uint8))).to(dev)
    else:
        da = torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        db = torch.from_numpy(np.ascontiguousarray(b, np.int32)).to(dev)
    dp = torch.from_numpy(np.ascontiguousarray(pairs, PAIR_DTYPE).view(np.uint8)).to(dev)
    out = torch.full((max(1, len(pairs)),), 0x7fffffff, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    fn = fz_edit_distance_batch if kind == "edit" else fz_dtw_batch
    fn(da.data_ptr(), len(a), db.data_ptr(), len(b), dp.data_ptr(), len(pairs), out.data_ptr(), st)
    torch.cuda.synchronize(dev)
    return out[:len(pairs)].cpu().numpy()


FZ_INT_RATES = 11
INT_RATE_NAMES = ("viaddmax", "vimax3", "iadd", "imax", "viaddmax_s16x2", "vimax3_s16x2", "vadd2", "imad",
                  "cell16_per_s", "cell32_per_s", "cell16_traced_per_s")


def fz_bench_int_rates():
    """Integer-pipe rates (fz.h lists the entries): op/s, and cells/s of the
    costed cell in the 16-bit pair and 32-bit forms."""
    out = (ctypes.c_double * FZ_INT_RATES)()
    _check(None, load().fz_bench_int_rates(out))
    return dict(zip(INT_RATE_NAMES, list(out)))


def fz_pair_sweep_used(sub, gap_open: int, gap_extend: int, ydrop: int, mode: int) -> bool:
    """Whether a context with these arguments runs its first inspector tier as
    the 16-bit pair sweep (host only)."""
    s = np.ascontiguousarray(np.asarray(sub, np.int32).reshape(16))
    return bool(load().fz_pair_sweep_used(s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(gap_open),
                                          int(gap_extend), int(ydrop), int(mode)))


# ---------------------------------------------------------------------------
# Convenience wrapper: torch supplies device memory and streams; the work is
# the library's.  Used by the tests, the benchmark and the smoke check.
# ---------------------------------------------------------------------------
class _DevArray:
    """Raw device pointer exposed through __cuda_array_interface__."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


class Extender:
    """One fz context plus device copies of one workload's inputs."""

    def __init__(self, sub, gap_open, gap_extend, ydrop, max_len, mode=FZ_EXTEND, device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        with torch.cuda.device(self.device):
            self.ctx = fz_create(sub, gap_open, gap_extend, ydrop, max_len, mode)
        self.mode = mode
        self.max_len = max_len

    @classmethod
    def for_workload(cls, w, **kw):
        return cls(w.sub, w.gap_open, w.gap_extend, w.ydrop, w.max_len, w.mode, **kw)

    def close(self):
        if self.ctx:
            fz_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def upload(self, target2: np.ndarray, query2: np.ndarray, seeds: np.ndarray):
        """Device copies (uint8 tensors) of packed sequences and seeds."""
        t = self.torch
        d_t = t.from_numpy(np.ascontiguousarray(target2)).to(self.device)
        d_q = t.from_numpy(np.ascontiguousarray(query2)).to(self.device)
        d_s = t.from_numpy(np.ascontiguousarray(seeds).view(np.uint8)).to(self.device)
        return d_t, d_q, d_s

    def alloc_out(self, n_seeds: int):
        return self.torch.empty(max(1, 2 * n_seeds * RESULT_DTYPE.itemsize), dtype=self.torch.uint8,
                                device=self.device)

    def run(self, d_t, t_len, d_q, q_len, d_s, n_seeds, d_out, stream=None) -> int:
        st = stream.cuda_stream if stream is not None else self.torch.cuda.current_stream(self.device).cuda_stream
        return fz_extend_batch(self.ctx, d_t.data_ptr(), t_len, d_q.data_ptr(), q_len, d_s.data_ptr(), n_seeds,
                               d_out.data_ptr(), st)

    def stats(self) -> FzStats:
        return fz_get_stats(self.ctx)

    def fetch(self, d_out, n_seeds: int, cigar_ptr: int):
        """Copy results and CIGAR arena to the host (synchronises)."""
        t = self.torch
        st = self.stats()
        res = np.frombuffer(d_out[:2 * n_seeds * RESULT_DTYPE.itemsize].cpu().numpy().tobytes(),
                            dtype=RESULT_DTYPE)
        ncig = int(st.cigar_runs) if self.mode == FZ_EXTEND else 0
        if ncig and cigar_ptr:
            cig = t.as_tensor(_DevArray(cigar_ptr, ncig, "<u4"), device=self.device).cpu().numpy().copy()
        else:
            cig = np.zeros(0, np.uint32)
        return res, cig, st

    def extend_workload(self, w, seeds=None):
        """Whole workload through the device entry; returns (results, cigar, stats)."""
        from .workloads import pack2
        seeds = w.seeds if seeds is None else seeds
        d_t, d_q, d_s = self.upload(pack2(w.target), pack2(w.query), seeds)
        d_out = self.alloc_out(len(seeds))
        cp = self.run(d_t, w.target.size, d_q, w.query.size, d_s, len(seeds), d_out)
        return self.fetch(d_out, len(seeds), cp)

    def extend_and_combine(self, w, seeds=None):
        """Whole workload, then fz_combine; returns (alignments, combined cigar)."""
        from .workloads import pack2
        seeds = w.seeds if seeds is None else seeds
        t = self.torch
        d_t, d_q, d_s = self.upload(pack2(w.target), pack2(w.query), seeds)
        d_out = self.alloc_out(len(seeds))
        cp = self.run(d_t, w.target.size, d_q, w.query.size, d_s, len(seeds), d_out)
        d_aln = t.empty(max(1, len(seeds) * ALIGNMENT_DTYPE.itemsize), dtype=t.uint8, device=self.device)
        st = t.cuda.current_stream(self.device).cuda_stream
        acp = fz_combine(self.ctx, d_s.data_ptr(), len(seeds), d_out.data_ptr(), cp, d_aln.data_ptr(), st)
        aln = np.frombuffer(d_aln[:len(seeds) * ALIGNMENT_DTYPE.itemsize].cpu().numpy().tobytes(),
                            dtype=ALIGNMENT_DTYPE)
        n = int(aln["cigar_off"][-1] + aln["cigar_len"][-1]) if len(seeds) else 0
        if n and acp:
            cig = t.as_tensor(_DevArray(acp, n, "<u4"), device=self.device).cpu().numpy().copy()
        else:
            cig = np.zeros(0, np.uint32)
        return aln, cig

    def extend_workload_host(self, w, seeds=None, cigar_cap=None):
        from .workloads import pack2
        seeds = w.seeds if seeds is None else seeds
        out = np.zeros(2 * len(seeds), RESULT_DTYPE)
        cap = cigar_cap if cigar_cap is not None else int(2 * w.max_len * 2 * len(seeds) + 16)
        cig = np.zeros(cap, np.uint32)
        st = self.torch.cuda.current_stream(self.device).cuda_stream
        used = fz_extend_batch_host(self.ctx, pack2(w.target), w.target.size, pack2(w.query), w.query.size,
                                    np.ascontiguousarray(seeds), out, cig, st)
        return out, cig[:used].copy()
