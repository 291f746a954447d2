"""CPU oracle for gapped y-drop seed extension -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never calls it; the
CUDA library and this oracle share no code.

``build()`` compiles ``fz_oracle.c`` (plain C, single-threaded arithmetic, a
pthread pool only to run independent extensions side by side) into
``oracle/_build/liboracle.so`` and ``extend_batch()`` runs it over a batch of
seeds, returning per extension (right, left) the score, end cell, live-cell
count and CIGAR runs.  ``edit_distance()`` and ``dtw()`` are the article's two
other dynamic programs (unit-cost edit distance; dynamic time warping).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fz_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OrcResult(ctypes.Structure):
    _fields_ = [("score", ctypes.c_int32), ("i_end", ctypes.c_int32), ("j_end", ctypes.c_int32),
                ("d_last", ctypes.c_int32), ("live_cells", ctypes.c_int64),
                ("n_cigar", ctypes.c_int32), ("status", ctypes.c_int32), ("max_width", ctypes.c_int32),
                ("narrow_steps", ctypes.c_int32)]


RESULT_DTYPE = np.dtype([("score", "<i4"), ("i_end", "<i4"), ("j_end", "<i4"), ("d_last", "<i4"),
                         ("live_cells", "<i8"), ("n_cigar", "<i4"), ("status", "<i4"), ("max_width", "<i4"),
                         ("narrow_steps", "<i4")])
assert RESULT_DTYPE.itemsize == ctypes.sizeof(OrcResult)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, no SIMD intrinsics)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.POINTER
            u8p, i32p, u32p, i64p, u64p = (P(ctypes.c_uint8), P(ctypes.c_int32), P(ctypes.c_uint32),
                                           P(ctypes.c_int64), P(ctypes.c_uint64))
            L.orc_extend.argtypes = [u8p, ctypes.c_int32, u8p, ctypes.c_int32, i32p, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P(OrcResult),
                                     u32p, ctypes.c_int32]
            L.orc_extend.restype = ctypes.c_int
            L.orc_local.argtypes = [u8p, ctypes.c_int32, u8p, ctypes.c_int32, i32p, ctypes.c_int32,
                                    ctypes.c_int32, P(OrcResult)]
            L.orc_local.restype = ctypes.c_int
            L.orc_batch.argtypes = [u8p, ctypes.c_uint64, u8p, ctypes.c_uint64, u64p, u64p, u32p,
                                    ctypes.c_int64, i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_void_p, u32p, i64p]
            L.orc_batch.restype = ctypes.c_int
            L.orc_edit_distance.argtypes = [u8p, ctypes.c_int32, u8p, ctypes.c_int32]
            L.orc_edit_distance.restype = ctypes.c_int32
            L.orc_dtw.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32]
            L.orc_dtw.restype = ctypes.c_int64
            _lib = L
    return _lib


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def extend_one(t, q, sub, gap_open, gap_extend, ydrop, descending=False):
    """One EXTEND window (bases in extension order).  ydrop < 0: no pruning.

    Returns (score, i_end, j_end, live_cells, d_last, cigar_runs[np.uint32])."""
    t = np.ascontiguousarray(t, np.uint8)
    q = np.ascontiguousarray(q, np.uint8)
    sub = np.ascontiguousarray(np.asarray(sub, np.int32).reshape(16))
    cap = max(1, t.size + q.size)
    cig = np.zeros(cap, np.uint32)
    r = OrcResult()
    rc = lib().orc_extend(_ptr(t, ctypes.c_uint8), t.size, _ptr(q, ctypes.c_uint8), q.size,
                          _ptr(sub, ctypes.c_int32), gap_open, gap_extend, int(ydrop),
                          1 if descending else 0, ctypes.byref(r), _ptr(cig, ctypes.c_uint32), cap)
    if rc != 0:
        raise RuntimeError(f"oracle extend failed: {rc}")
    return r.score, r.i_end, r.j_end, r.live_cells, r.d_last, cig[:r.n_cigar].copy()


def local_one(t, q, sub, gap_open, gap_extend):
    t = np.ascontiguousarray(t, np.uint8)
    q = np.ascontiguousarray(q, np.uint8)
    sub = np.ascontiguousarray(np.asarray(sub, np.int32).reshape(16))
    r = OrcResult()
    rc = lib().orc_local(_ptr(t, ctypes.c_uint8), t.size, _ptr(q, ctypes.c_uint8), q.size,
                         _ptr(sub, ctypes.c_int32), gap_open, gap_extend, ctypes.byref(r))
    if rc != 0:
        raise RuntimeError(f"oracle local failed: {rc}")
    return r.score, r.i_end, r.j_end


def window_lengths(t_len, q_len, seeds, max_len):
    """(m, n) per extension, shape [n_seeds, 2] for [right, left] (0 if not requested)."""
    tp = seeds["t_pos"].astype(np.int64)
    qp = seeds["q_pos"].astype(np.int64)
    side = seeds["side"].astype(np.int64)
    m = np.zeros((len(seeds), 2), np.int64)
    n = np.zeros((len(seeds), 2), np.int64)
    m[:, 0] = np.clip(t_len - tp, 0, max_len)
    n[:, 0] = np.clip(q_len - qp, 0, max_len)
    m[:, 1] = np.clip(np.minimum(tp, t_len), 0, max_len)
    n[:, 1] = np.clip(np.minimum(qp, q_len), 0, max_len)
    m[(side & 1) == 0, 0] = 0
    n[(side & 1) == 0, 0] = 0
    m[(side & 2) == 0, 1] = 0
    n[(side & 2) == 0, 1] = 0
    return m, n


def extend_batch(w, seeds=None, nthreads: int = 1, descending: bool = False, ydrop=None):
    """Run the oracle over a Workload's seeds (or ``seeds``).

    Returns (res[RESULT_DTYPE, 2*n], cigar[uint32], cig_off[int64, 2*n+1]); for
    extension x = 2*k + side (side 0 = right, 1 = left) the CIGAR runs, in
    extension order, are cigar[cig_off[x] : cig_off[x] + res[x]['n_cigar']].
    """
    seeds = w.seeds if seeds is None else seeds
    seeds = np.ascontiguousarray(seeds)
    n = len(seeds)
    tseq = np.ascontiguousarray(w.target, np.uint8)
    qseq = np.ascontiguousarray(w.query, np.uint8)
    m_, n_ = window_lengths(tseq.size, qseq.size, seeds, w.max_len)
    caps = (m_ + n_).reshape(-1) if w.mode == 0 else np.zeros(2 * n, np.int64)
    cig_off = np.zeros(2 * n + 1, np.int64)
    np.cumsum(caps, out=cig_off[1:])
    cigar = np.zeros(max(1, int(cig_off[-1])), np.uint32)
    res = np.zeros(2 * n, RESULT_DTYPE)
    tp = np.ascontiguousarray(seeds["t_pos"], np.uint64)
    qp = np.ascontiguousarray(seeds["q_pos"], np.uint64)
    sd = np.ascontiguousarray(seeds["side"], np.uint32)
    sub = np.ascontiguousarray(np.asarray(w.sub, np.int32).reshape(16))
    yd = w.ydrop if ydrop is None else ydrop
    rc = lib().orc_batch(_ptr(tseq, ctypes.c_uint8), tseq.size, _ptr(qseq, ctypes.c_uint8), qseq.size,
                         _ptr(tp, ctypes.c_uint64), _ptr(qp, ctypes.c_uint64), _ptr(sd, ctypes.c_uint32),
                         n, _ptr(sub, ctypes.c_int32), w.gap_open, w.gap_extend, int(yd), w.max_len,
                         w.mode, 1 if descending else 0, nthreads, res.ctypes.data_as(ctypes.c_void_p),
                         _ptr(cigar, ctypes.c_uint32), _ptr(cig_off, ctypes.c_int64))
    if rc != 0:
        raise RuntimeError(f"oracle batch failed: {rc}")
    return res, cigar, cig_off


def genomic_cigar(runs, left: bool):
    """Runs in forward genomic order: extension order for the right side,
    reversed for the left side (its window is read backwards)."""
    runs = np.asarray(runs, np.uint32)
    return runs[::-1].copy() if left else runs.copy()


def combine(seeds, res, cigar, cig_off):
    """Two-sided alignment per seed from the oracle's one-sided results (FastZ,
    section 3.1.2: LASTZ joins the two extensions of a seed).  Plain definition:
    score = right score + left score; target span [t_pos - left i*, t_pos +
    right i*), query span [q_pos - left j*, q_pos + right j*); CIGAR = the left
    runs then the right runs, both in forward genomic order, the two runs that
    meet at the anchor merged into one when they are the same operation.  A side
    that was not requested contributes nothing.

    Returns a list of (score, t_start, q_start, t_end, q_end, runs[np.uint32])."""
    out = []
    for k in range(len(seeds)):
        side = int(seeds["side"][k])
        tp, qp = int(seeds["t_pos"][k]), int(seeds["q_pos"][k])
        xr, xl = 2 * k, 2 * k + 1
        hr, hl = bool(side & 1), bool(side & 2)
        right = [int(v) for v in cigar[cig_off[xr]:cig_off[xr] + res["n_cigar"][xr]]] if hr else []
        left = [int(v) for v in genomic_cigar(cigar[cig_off[xl]:cig_off[xl] + res["n_cigar"][xl]], True)] if hl else []
        runs = list(left)
        if runs and right and (runs[-1] & 15) == (right[0] & 15):
            runs[-1] += right[0] & ~15
            right = right[1:]
        runs += right
        score = (int(res["score"][xr]) if hr else 0) + (int(res["score"][xl]) if hl else 0)
        out.append((score,
                    tp - (int(res["i_end"][xl]) if hl else 0), qp - (int(res["j_end"][xl]) if hl else 0),
                    tp + (int(res["i_end"][xr]) if hr else 0), qp + (int(res["j_end"][xr]) if hr else 0),
                    np.asarray(runs, np.uint32)))
    return out


def edit_distance(a, b) -> int:
    """Levenshtein distance of two base-code sequences (unit costs; the DPX
    intrinsics article, section 1.3)."""
    a = np.ascontiguousarray(a, np.uint8)
    b = np.ascontiguousarray(b, np.uint8)
    r = lib().orc_edit_distance(_ptr(a, ctypes.c_uint8), a.size, _ptr(b, ctypes.c_uint8), b.size)
    if r < 0:
        raise RuntimeError("oracle edit distance failed")
    return int(r)


def dtw(x, y) -> int:
    """Dynamic time warping cost of two int32 sequences, cell cost |x_i - y_j|
    (the DPX intrinsics article, section 1.3); -1 when exactly one is empty."""
    x = np.ascontiguousarray(x, np.int32)
    y = np.ascontiguousarray(y, np.int32)
    r = lib().orc_dtw(_ptr(x, ctypes.c_int32), x.size, _ptr(y, ctypes.c_int32), y.size)
    if r < -1:
        raise RuntimeError("oracle dtw failed")
    return int(r)


def pairs_batch(fn, a, b, pairs):
    """fn over pairs (fields a_pos, b_pos, a_len, b_len) of the sequences a and b."""
    out = np.zeros(len(pairs), np.int64)
    for k, pr in enumerate(pairs):
        ap, bp, al, bl = int(pr["a_pos"]), int(pr["b_pos"]), int(pr["a_len"]), int(pr["b_len"])
        out[k] = fn(a[ap:ap + al], b[bp:bp + bl])
    return out
