"""Seeded synthetic seed-extension workloads.

This module only makes inputs: random DNA, mutated copies, seed anchors and the
scoring parameters.  It holds none of the alignment arithmetic, so both the CPU
oracle and the CUDA path can be fed from it without sharing any of the method.

Sequences are uint8 arrays of base codes A=0, C=1, G=2, T=3.  ``pack2`` stores
base k at bits 2*(k mod 4) of byte k // 4 (little-endian inside the byte), the
layout the C ABI takes.

Workload shapes follow the five seed-extension batches used throughout this
project: short windows (256 bp), skewed homology lengths in 6 kbp windows (the
FastZ paper, section 1, reports that more than 97% of seeds give alignments no
longer than 128 bp), a chromosome-scale two-sided batch, long high-identity
extensions in 60 kbp windows, and an unpruned local fill of 2048 x 2048 pairs.
The real genomes of the FastZ evaluation (its Table 1) are not available;
these synthetic inputs stand in for them.
"""
from __future__ import annotations

import dataclasses
import numpy as np

# HOXD70 substitution scores (Chiaromonte, Yap & Miller 2002), rows = target
# base, columns = query base, order A, C, G, T.
HOXD70 = np.array(
    [[91, -114, -31, -123],
     [-114, 100, -125, -31],
     [-31, -125, 100, -114],
     [-123, -31, -114, 91]], dtype=np.int32)
GAP_OPEN = 400
GAP_EXTEND = 30
YDROP = 9400
YDROP_INF = -1          # "no pruning" sentinel of the C ABI

MODE_EXTEND = 0
MODE_LOCAL = 1

SIDE_RIGHT = 1
SIDE_LEFT = 2
SIDE_BOTH = 3

SEED_DTYPE = np.dtype([("t_pos", "<u8"), ("q_pos", "<u8"), ("side", "<u4")], align=True)
assert SEED_DTYPE.itemsize == 24

SEED_BASE = 0x4641535400000000  # ASCII "FAST" in the high word


@dataclasses.dataclass
class Workload:
    name: str
    target: np.ndarray          # uint8 base codes
    query: np.ndarray           # uint8 base codes
    seeds: np.ndarray           # SEED_DTYPE records
    sub: np.ndarray             # int32 [4, 4]
    gap_open: int
    gap_extend: int
    ydrop: int                  # >= 0, or YDROP_INF
    max_len: int
    mode: int
    note: str = ""

    @property
    def n_extensions(self) -> int:
        s = self.seeds["side"]
        return int(np.count_nonzero(s & SIDE_RIGHT) + np.count_nonzero(s & SIDE_LEFT))

    def subset(self, idx) -> "Workload":
        return dataclasses.replace(self, seeds=self.seeds[np.asarray(idx)])


def rng_for(config_id: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + config_id + (salt << 8)))


def pack2(bases: np.ndarray) -> np.ndarray:
    """2-bit pack: base k -> bits 2*(k%4) of byte k//4."""
    b = np.asarray(bases, dtype=np.uint8)
    n = b.size
    pad = (-n) % 4
    if pad:
        b = np.concatenate([b, np.zeros(pad, np.uint8)])
    b = b.reshape(-1, 4)
    return (b[:, 0] | (b[:, 1] << 2) | (b[:, 2] << 4) | (b[:, 3] << 6)).astype(np.uint8)


def unpack2(packed: np.ndarray, n: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.size * 4, np.uint8)
    out[0::4] = p & 3
    out[1::4] = (p >> 2) & 3
    out[2::4] = (p >> 4) & 3
    out[3::4] = (p >> 6) & 3
    return out[:n]


def random_bases(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.integers(0, 4, size=n, dtype=np.uint8)


def mutate(rng: np.random.Generator, src: np.ndarray, p_sub: float, p_indel: float,
           mean_len: float, want_map: bool = False):
    """Copy ``src`` with point substitutions and geometric-length indels.

    At every source base: with probability ``p_sub`` it becomes one of the other
    three bases (uniform); with probability ``p_indel`` an indel starts there,
    an insertion or a deletion with equal odds, of length L ~ Geometric with
    mean ``mean_len`` on {1, 2, ...}.  A deletion removes L source bases
    starting at this one; an insertion places L uniform random bases after it.
    Returns the copy, and with ``want_map`` also an int64 array giving, for each
    source position, the output position of the first surviving base at or
    after it.
    """
    src = np.asarray(src, dtype=np.uint8)
    n = src.size
    out_bases = src.copy()
    if n == 0:
        return (out_bases, np.zeros(0, np.int64)) if want_map else out_bases
    subst = rng.random(n) < p_sub
    shift = rng.integers(1, 4, size=n, dtype=np.uint8)
    out_bases = np.where(subst, (src + shift) & 3, src).astype(np.uint8)
    ev = np.flatnonzero(rng.random(n) < p_indel)
    is_ins = rng.random(ev.size) < 0.5
    lens = rng.geometric(1.0 / mean_len, size=ev.size).astype(np.int64)
    keep = np.ones(n, dtype=bool)
    dels = ev[~is_ins]
    dlen = lens[~is_ins]
    if dels.size:
        # mark [p, p+L) deleted via a difference array
        diff = np.zeros(n + 1, np.int64)
        np.add.at(diff, dels, 1)
        np.add.at(diff, np.minimum(dels + dlen, n), -1)
        keep = np.cumsum(diff[:n]) == 0
    ins_len = np.zeros(n, np.int64)
    if np.any(is_ins):
        np.add.at(ins_len, ev[is_ins], lens[is_ins])
    count = keep.astype(np.int64) + ins_len
    start = np.concatenate([[0], np.cumsum(count)[:-1]])
    total = int(count.sum())
    out = random_bases(rng, total)            # inserted bases stay random
    kept = np.flatnonzero(keep)
    out[start[kept]] = out_bases[kept]
    if not want_map:
        return out
    return out, start


def revcomp(x: np.ndarray) -> np.ndarray:
    return (3 - x[::-1]).astype(np.uint8)


def log_uniform_int(rng, lo, hi, size):
    return np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), size=size))).astype(np.int64)


def _pairs_workload(name, rng, n_pairs, win, hom_len, p_sub, p_indel, mean_len, note):
    """n_pairs independent right extensions, each over its own win x win window.

    The target window is random; the query window is a mutated copy of the first
    h target bases followed by unrelated random sequence (cut to ``win``).
    Windows are laid end to end in one target and one query sequence; seed k
    anchors at k*win in both.
    """
    target = random_bases(rng, n_pairs * win)
    query = random_bases(rng, n_pairs * win)
    for k in range(n_pairs):
        h = int(hom_len[k])
        tw = target[k * win:(k + 1) * win]
        hom = mutate(rng, tw[:h], p_sub, p_indel, mean_len)[:win]
        query[k * win:k * win + hom.size] = hom
    seeds = np.zeros(n_pairs, SEED_DTYPE)
    seeds["t_pos"] = np.arange(n_pairs, dtype=np.uint64) * win
    seeds["q_pos"] = np.arange(n_pairs, dtype=np.uint64) * win
    seeds["side"] = SIDE_RIGHT
    return Workload(name, target, query, seeds, HOXD70.copy(), GAP_OPEN, GAP_EXTEND, YDROP,
                    win, MODE_EXTEND, note)


def make_cfg1(n_pairs: int = 2000) -> Workload:
    """2,000 right extensions, 256 bp windows, h ~ U[16, 200], 10% subs, 1% indels (mean 2)."""
    rng = rng_for(1)
    hom = rng.integers(16, 201, size=n_pairs)
    return _pairs_workload("short-256bp", rng, n_pairs, 256, hom, 0.10, 0.01, 2.0,
                           "2000 right extensions, 256 bp windows")


def make_cfg2(n_pairs: int = 100_000) -> Workload:
    """100,000 right extensions, 6,000 bp windows, skewed homology length."""
    rng = rng_for(2)
    short = rng.random(n_pairs) < 0.97
    hom = np.where(short, log_uniform_int(rng, 8, 128, n_pairs), log_uniform_int(rng, 128, 5000, n_pairs))
    return _pairs_workload("skewed-6kbp", rng, n_pairs, 6000, hom, 0.12, 0.02, 3.0,
                           "100000 right extensions, 6000 bp windows, 97% h in [8,128]")


def make_cfg4(n_pairs: int = 2000) -> Workload:
    """2,000 long extensions: h ~ U[20k, 50k], 2% subs, 0.5% indels (mean 4), 60 kbp windows."""
    rng = rng_for(4)
    hom = rng.integers(20_000, 50_001, size=n_pairs)
    return _pairs_workload("long-60kbp", rng, n_pairs, 60_000, hom, 0.02, 0.005, 4.0,
                           "2000 right extensions, 60 kbp windows, h in [20k,50k]")


def make_cfg5(n_pairs: int = 65_536, length: int = 2048) -> Workload:
    """Unpruned local fill: n_pairs independent length x length pairs; half share a
    1 kbp 10%-divergent block at independent uniform offsets."""
    rng = rng_for(5)
    target = random_bases(rng, n_pairs * length)
    query = random_bases(rng, n_pairs * length)
    block = 1000
    has = rng.random(n_pairs) < 0.5
    for k in np.flatnonzero(has):
        b = random_bases(rng, block)
        ot = int(rng.integers(0, length - block + 1))
        oq = int(rng.integers(0, length - block + 1))
        target[k * length + ot:k * length + ot + block] = b
        mb = mutate(rng, b, 0.09, 0.01, 2.0)[:length - oq]
        query[k * length + oq:k * length + oq + mb.size] = mb
    seeds = np.zeros(n_pairs, SEED_DTYPE)
    seeds["t_pos"] = np.arange(n_pairs, dtype=np.uint64) * length
    seeds["q_pos"] = np.arange(n_pairs, dtype=np.uint64) * length
    seeds["side"] = SIDE_RIGHT
    return Workload("local-2048", target, query, seeds, HOXD70.copy(), GAP_OPEN, GAP_EXTEND,
                    YDROP_INF, length, MODE_LOCAL,
                    f"{n_pairs} local pairs of {length} x {length}")


def make_cfg3(n_anchors: int = 1_000_000, t_len: int = 50_000_000, window: int = 6000) -> Workload:
    """Chromosome-scale two-sided batch.

    Target: t_len random bases.  Query: the target with 10 kbp blocks reverse-
    complemented in place or moved elsewhere (50/50) at exponential spacing of
    mean 1 Mbp, then mutated (15% substitutions, 3% indels, mean length 2).
    70% of anchors are homologous (a target position outside any rearranged
    block, mapped into the query); 30% are uniform random pairs.
    """
    rng = rng_for(3)
    target = random_bases(rng, t_len)
    blk = 10_000
    gaps = rng.exponential(1_000_000, size=int(t_len / 1_000_000 * 3) + 10).astype(np.int64)
    starts = np.cumsum(gaps + blk)
    starts = starts[starts + blk < t_len]
    kind_inv = rng.random(starts.size) < 0.5
    rearranged = np.zeros(t_len, dtype=bool)
    # source order of the rearranged query (index into target)
    src = np.arange(t_len, dtype=np.int64)
    comp = np.zeros(t_len, dtype=bool)
    for s, inv in zip(starts, kind_inv):
        rearranged[s:s + blk] = True
        if inv:
            src[s:s + blk] = src[s:s + blk][::-1]
            comp[s:s + blk] = ~comp[s:s + blk]
    moved = starts[~kind_inv]
    if moved.size:
        pieces = []
        cursor = 0
        order = [(int(s), int(rng.integers(0, t_len))) for s in moved]
        cut = np.zeros(t_len, dtype=bool)
        for s, _ in order:
            cut[s:s + blk] = True
        keep_idx = np.flatnonzero(~cut)
        base_src = src[keep_idx]
        base_comp = comp[keep_idx]
        # insert each moved block at a random position of the remaining sequence
        ins_at = np.sort(np.array([rng.integers(0, keep_idx.size) for _ in order], dtype=np.int64))
        pieces_src, pieces_comp = [], []
        for (s, _), at in zip(order, ins_at):
            pieces_src.append(base_src[cursor:at])
            pieces_comp.append(base_comp[cursor:at])
            pieces_src.append(src[s:s + blk])
            pieces_comp.append(comp[s:s + blk])
            cursor = at
        pieces_src.append(base_src[cursor:])
        pieces_comp.append(base_comp[cursor:])
        src = np.concatenate(pieces_src)
        comp = np.concatenate(pieces_comp)
        del pieces
    q0 = target[src]
    q0 = np.where(comp, 3 - q0, q0).astype(np.uint8)
    pos_in_q0 = np.empty(t_len, np.int64)
    pos_in_q0[src] = np.arange(t_len, dtype=np.int64)
    query, qmap = mutate(rng, q0, 0.15, 0.03, 2.0, want_map=True)
    n_hom = int(round(n_anchors * 0.7))
    n_spur = n_anchors - n_hom
    ok = np.flatnonzero(~rearranged)
    t_h = ok[rng.integers(0, ok.size, size=n_hom)]
    q_h = qmap[pos_in_q0[t_h]]
    t_s = rng.integers(0, t_len, size=n_spur)
    q_s = rng.integers(0, query.size, size=n_spur)
    seeds = np.zeros(n_anchors, SEED_DTYPE)
    t_all = np.concatenate([t_h, t_s])
    q_all = np.concatenate([q_h, q_s])
    perm = rng.permutation(n_anchors)
    seeds["t_pos"] = t_all[perm].astype(np.uint64)
    seeds["q_pos"] = np.minimum(q_all[perm], query.size).astype(np.uint64)
    seeds["side"] = SIDE_BOTH
    return Workload("chrom-50Mbp-2sided", target, query, seeds, HOXD70.copy(), GAP_OPEN, GAP_EXTEND,
                    YDROP, window, MODE_EXTEND,
                    f"{n_anchors} two-sided anchors on a {t_len} bp target")


def make_wide(n_pairs: int = 512, win: int = 3000) -> Workload:
    """A batch for the general-band path (not one of the five configurations):
    n_pairs right extensions over win x win windows, the query a mutated copy of
    the whole target window (10% substitutions, 2% indels of mean length 3), and
    a y-drop of 40,000, so that the live bands hold about a thousand rows, more
    than the register windows' 512."""
    rng = rng_for(6)
    hom = np.full(n_pairs, win)
    w = _pairs_workload("wide-band-3kbp", rng, n_pairs, win, hom, 0.10, 0.02, 3.0,
                        f"{n_pairs} right extensions, {win} bp windows, homologous throughout, y-drop 40000")
    return dataclasses.replace(w, ydrop=40000)


MAKERS = {1: make_cfg1, 2: make_cfg2, 3: make_cfg3, 4: make_cfg4, 5: make_cfg5}


def make(config_id: int, **kw) -> Workload:
    return MAKERS[config_id](**kw)


def window_bases(seq: np.ndarray, pos: int, side: int, max_len: int) -> np.ndarray:
    """Bases of a one-sided extension window, in extension order.

    Right side: seq[pos], seq[pos+1], ... (index 1 of the window is seq[pos]).
    Left side: seq[pos-1], seq[pos-2], ... (read backwards from the anchor).
    Length min(max_len, bases available on that side).
    """
    pos = int(pos)
    if side == SIDE_RIGHT:
        n = max(0, min(max_len, seq.size - pos))
        return seq[pos:pos + n]
    n = max(0, min(max_len, pos))
    return seq[pos - n:pos][::-1]


# ---------------------------------------------------------------------------
# The DPX article's other two dynamic programs (section 4.1 times a batch of
# 512 edit distances of 1024 x 1024 and 256 DTWs of 800 x 800 on random
# sequences): pairs laid end to end in two sequences, half of them related.
# ---------------------------------------------------------------------------
DP_PAIR_DTYPE = np.dtype([("a_pos", "<u8"), ("b_pos", "<u8"), ("a_len", "<u4"), ("b_len", "<u4")])


@dataclasses.dataclass
class DPWorkload:
    name: str
    kind: str                   # "edit" (base codes) or "dtw" (int32 samples)
    a: np.ndarray
    b: np.ndarray
    pairs: np.ndarray           # DP_PAIR_DTYPE
    note: str = ""


def dp_pairs(lens_a, lens_b):
    pairs = np.zeros(len(lens_a), DP_PAIR_DTYPE)
    pairs["a_len"] = lens_a
    pairs["b_len"] = lens_b
    pairs["a_pos"][1:] = np.cumsum(np.asarray(lens_a, np.uint64))[:-1]
    pairs["b_pos"][1:] = np.cumsum(np.asarray(lens_b, np.uint64))[:-1]
    return pairs


def make_edit_batch(n_pairs: int = 512, length: int = 1024, seed: int = 6) -> DPWorkload:
    """n_pairs DNA pairs of `length` bases; half the b sequences are the a
    sequence with 10% substitutions and 1% indels (trimmed or padded with
    random bases to `length`), half unrelated."""
    rng = rng_for(seed)
    a_parts, b_parts = [], []
    for k in range(n_pairs):
        a = random_bases(rng, length)
        if k % 2 == 0:
            b = mutate(rng, a, 0.10, 0.01, 2.0)[:length]
            b = np.concatenate([b, random_bases(rng, length - b.size)]) if b.size < length else b
        else:
            b = random_bases(rng, length)
        a_parts.append(a)
        b_parts.append(b.astype(np.uint8))
    return DPWorkload(f"edit-{length}", "edit", np.concatenate(a_parts), np.concatenate(b_parts),
                      dp_pairs([length] * n_pairs, [length] * n_pairs),
                      f"{n_pairs} edit distances of {length} x {length} bases")


def random_walk(rng: np.random.Generator, n: int, step: int = 8) -> np.ndarray:
    return np.clip(np.cumsum(rng.integers(-step, step + 1, n)), -32767, 32767).astype(np.int32)


def make_dtw_batch(n_pairs: int = 256, length: int = 800, seed: int = 7) -> DPWorkload:
    """n_pairs pairs of `length` int32 samples (random walks); half the y
    sequences are x resampled along a random monotone warp plus noise, half
    independent walks."""
    rng = rng_for(seed)
    xs, ys = [], []
    for k in range(n_pairs):
        x = random_walk(rng, length)
        if k % 2 == 0:
            warp = np.sort(rng.integers(0, length, length))
            y = np.clip(x[warp] + rng.integers(-3, 4, length), -32767, 32767).astype(np.int32)
        else:
            y = random_walk(rng, length)
        xs.append(x)
        ys.append(y)
    return DPWorkload(f"dtw-{length}", "dtw", np.concatenate(xs), np.concatenate(ys),
                      dp_pairs([length] * n_pairs, [length] * n_pairs),
                      f"{n_pairs} dynamic time warpings of {length} x {length} samples")
