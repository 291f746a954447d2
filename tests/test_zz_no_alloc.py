"""The allocation-free local fill entry point against the context entry point.

fz_local_fill_noalloc serves callers that cannot allocate device memory at run
time (a locked caching allocator, a host framework that forbids cudaMalloc on
its hot path): its scratch is a fixed device array inside the library.  Its
results must equal those of fz_extend_batch on a FZ_LOCAL context, on two
calls in a row with different inputs (the second call must not see the
first call's scratch contents), and those of the CPU oracle on a
non-symmetric substitution matrix.  Integer results: compared exactly.
"""
import os

import numpy as np
import pytest

from gapped_smith_waterman_gb300 import build as B
from gapped_smith_waterman_gb300 import fz
from gapped_smith_waterman_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    B.build()
    fz.load()


def _context_entry(w, seeds):
    ext = fz.Extender.for_workload(w)
    try:
        res, _, _ = ext.extend_workload(w, seeds)
    finally:
        ext.close()
    return res


def _noalloc_entry(w, seeds):
    import torch
    t2 = torch.from_numpy(W.pack2(w.target)).cuda()
    q2 = torch.from_numpy(W.pack2(w.query)).cuda()
    sd = torch.from_numpy(np.ascontiguousarray(seeds).view(np.uint8)).cuda()
    out = torch.full((2 * len(seeds) * fz.RESULT_DTYPE.itemsize,), 0xAB, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    fz.fz_local_fill_noalloc(w.sub, w.gap_open, w.gap_extend, w.max_len, t2.data_ptr(), w.target.size,
                             q2.data_ptr(), w.query.size, sd.data_ptr(), len(seeds), out.data_ptr(), stream)
    torch.cuda.synchronize()
    return np.frombuffer(out.cpu().numpy().tobytes(), dtype=fz.RESULT_DTYPE)


def _mixed_workload():
    """Uneven pairs (partial strips, empty windows) laid end to end."""
    rng = np.random.default_rng(2024)
    ml = 1500
    n = 120
    T = rng.integers(0, 4, n * ml).astype(np.uint8)
    Q = rng.integers(0, 4, n * ml).astype(np.uint8)
    for k in range(0, n, 2):
        h = int(rng.integers(50, 900))
        blk = T[k * ml:k * ml + h]
        m = W.mutate(rng, blk, 0.1, 0.01, 2.0)[:ml]
        Q[k * ml:k * ml + m.size] = m
    seeds = np.zeros(n, W.SEED_DTYPE)
    seeds["t_pos"] = np.arange(n) * ml + rng.integers(0, 400, n)
    seeds["q_pos"] = np.arange(n) * ml + rng.integers(0, 400, n)
    seeds["side"] = rng.integers(1, 4, n)
    seeds[0]["t_pos"] = T.size          # empty right window
    return W.Workload("mixed", T, Q, seeds, W.HOXD70.copy(), 400, 30, W.YDROP_INF, ml, W.MODE_LOCAL)


def test_noalloc_matches_context_entry_on_two_calls():
    w = W.make_cfg5(n_pairs=160)
    first = w.seeds.copy()
    second = w.seeds[::-1].copy()
    second["side"] = W.SIDE_BOTH
    for seeds in (first, second):
        want = _context_entry(w, seeds)
        got = _noalloc_entry(w, seeds)
        assert np.array_equal(got, want)
    mixed = _mixed_workload()
    for seeds in (mixed.seeds, mixed.seeds[::-1].copy()):
        assert np.array_equal(_noalloc_entry(mixed, seeds), _context_entry(mixed, seeds))


def _oracle_local(w, seeds):
    import oracle
    res, _, _ = oracle.extend_batch(w, seeds=seeds, nthreads=max(1, os.cpu_count() or 1))
    return res


def test_noalloc_non_symmetric_matrix_against_oracle():
    """A substitution matrix with M[t][q] != M[q][t] everywhere off the
    diagonal: a transposed score lookup (target and query roles swapped)
    changes the results.  Compared with the CPU oracle directly and with the
    context entry, on two calls in a row."""
    rng = np.random.default_rng(909)
    sub = rng.integers(-120, 121, size=(4, 4)).astype(np.int32)
    sub[np.arange(4), np.arange(4)] = rng.integers(40, 128, 4)
    for a in range(4):
        for b in range(a + 1, 4):
            if sub[a, b] == sub[b, a]:
                sub[a, b] += 7
    assert not np.array_equal(sub, sub.T)
    base = _mixed_workload()
    w = W.Workload("mixed-asym", base.target, base.query, base.seeds, sub, 350, 20, W.YDROP_INF, base.max_len,
                   W.MODE_LOCAL)
    # the transposed matrix must give different results on this batch, or the check would be blind
    wt = W.Workload("mixed-asym-t", base.target, base.query, base.seeds, np.ascontiguousarray(sub.T), 350, 20,
                    W.YDROP_INF, base.max_len, W.MODE_LOCAL)
    want = _oracle_local(w, w.seeds)
    assert not np.array_equal(want["score"], _oracle_local(wt, w.seeds)["score"])
    for seeds in (w.seeds, w.seeds[::-1].copy()):
        exp = want if seeds is w.seeds else _oracle_local(w, seeds)
        got = _noalloc_entry(w, seeds)
        for f_g, f_o in (("score", "score"), ("t_end", "i_end"), ("q_end", "j_end")):
            assert np.array_equal(got[f_g], exp[f_o]), f_g
        assert np.array_equal(got, _context_entry(w, seeds))


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (which may load the library's device code and with
    it the scratch array), further calls change neither the device's free
    memory nor torch's allocator."""
    import torch
    w = W.make_cfg5(n_pairs=64)
    t2 = torch.from_numpy(W.pack2(w.target)).cuda()
    q2 = torch.from_numpy(W.pack2(w.query)).cuda()
    sd = torch.from_numpy(np.ascontiguousarray(w.seeds).view(np.uint8)).cuda()
    out = torch.zeros(2 * len(w.seeds) * fz.RESULT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        fz.fz_local_fill_noalloc(w.sub, w.gap_open, w.gap_extend, w.max_len, t2.data_ptr(), w.target.size,
                                 q2.data_ptr(), w.query.size, sd.data_ptr(), len(w.seeds), out.data_ptr(), stream)
        torch.cuda.synchronize()

    call()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(2):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_rejects_sizes_beyond_its_limit():
    with pytest.raises(fz.FzError) as ei:
        fz.fz_local_fill_noalloc(W.HOXD70, 400, 30, 2049, 0, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
    with pytest.raises(fz.FzError) as ei:
        fz.fz_local_fill_noalloc(W.HOXD70 * 2, 400, 30, 100, 0, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
