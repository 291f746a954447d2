"""The allocation-free local fill entry point against the context entry point.

fz_local_fill_noalloc serves callers that cannot allocate device memory at run
time (a locked caching allocator, a host framework that forbids cudaMalloc on
its hot path): its scratch is a fixed device array inside the library.  Its
results must equal those of fz_extend_batch on a FZ_LOCAL context, on two
calls in a row with different inputs (the second call must not see the
first call's scratch contents).  Integer results: compared exactly.
"""
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


def test_noalloc_rejects_sizes_beyond_its_limit():
    with pytest.raises(fz.FzError) as ei:
        fz.fz_local_fill_noalloc(W.HOXD70, 400, 30, 2049, 0, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
    with pytest.raises(fz.FzError) as ei:
        fz.fz_local_fill_noalloc(W.HOXD70 * 2, 400, 30, 100, 0, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
