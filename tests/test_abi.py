"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every entry point declared in include/fz.h; argument validation
returns FZ_ERR_ARG before any CUDA call; the binding refuses a missing
library instead of falling back."""
import ctypes
import os
import re

import numpy as np
import pytest

from gapped_smith_waterman_gb300 import build as B
from gapped_smith_waterman_gb300 import fz
from gapped_smith_waterman_gb300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fz.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return fz.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(fz_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"fz_create", "fz_extend_batch", "fz_destroy", "fz_extend_batch_host", "fz_get_stats",
            "fz_last_error", "fz_set_profiling", "fz_bench_int_rates", "fz_local_fill_noalloc",
            "fz_combine", "fz_pair_sweep_used"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB)
    for name in declared_functions():
        assert hasattr(raw, name), name
    for name in fz.SYMBOLS:
        assert hasattr(lib, name), name


def test_struct_layouts_match_header():
    assert W.SEED_DTYPE.itemsize == 24
    assert fz.RESULT_DTYPE.itemsize == 24
    assert fz.ALIGNMENT_DTYPE.itemsize == 48
    # fields of fz_stats in order (4 bytes of padding before exec_live_cells)
    assert ctypes.sizeof(fz.FzStats) == 8 + 8 + 4 + 20 + 4 + 4 + 8 + 8 + 4 + 4 + 24 + 4 + 4 + 8 + 4 + 4 + 8


def test_struct_offsets_match_a_c_compiler(tmp_path):
    """The binding's record layouts against the header as a C compiler lays it out."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fields = [f for f, _ in fz.FzStats._fields_]
    prog = ['#include <stdio.h>', '#include <stddef.h>', '#include "fz.h"', 'int main(void) {',
            'printf("%zu\\n", sizeof(fz_stats));']
    prog += [f'printf("%zu\\n", offsetof(fz_stats, {f}));' for f in fields]
    prog += ['printf("%zu %zu %zu\\n", sizeof(fz_seed), sizeof(fz_result), sizeof(fz_alignment));', 'return 0; }']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(prog) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert int(out[0]) == ctypes.sizeof(fz.FzStats)
    for k, f in enumerate(fields):
        assert int(out[1 + k]) == getattr(fz.FzStats, f).offset, f
    assert out[1 + len(fields)].split() == ["24", "24", "48"]


@pytest.mark.parametrize("args", [
    dict(gap_open=-1, gap_extend=30, ydrop=9400, max_len=100),
    dict(gap_open=400, gap_extend=0, ydrop=9400, max_len=100),
    dict(gap_open=400, gap_extend=30, ydrop=-7, max_len=100),
    dict(gap_open=400, gap_extend=30, ydrop=9400, max_len=0),
    dict(gap_open=400, gap_extend=30, ydrop=9400, max_len=(1 << 20) + 1),
    dict(gap_open=400, gap_extend=30, ydrop=9400, max_len=1 << 20),       # score range would pass 2^28
])
def test_bad_arguments_rejected_without_gpu(lib, args):
    with pytest.raises(fz.FzError) as ei:
        fz.fz_create(W.HOXD70, mode=fz.FZ_EXTEND, **args)
    assert ei.value.status == fz.FZ_ERR_ARG


def test_local_mode_needs_byte_scores(lib):
    with pytest.raises(fz.FzError) as ei:
        fz.fz_create(W.HOXD70 * 2, 400, 30, -1, 100, fz.FZ_LOCAL)
    assert ei.value.status == fz.FZ_ERR_ARG


def test_null_arguments(lib):
    L = fz.load()
    assert L.fz_create(None, None, 400, 30, 9400, 100, 0) == fz.FZ_ERR_ARG
    assert L.fz_extend_batch(None, None, 0, None, 0, None, 0, None, None, None) == fz.FZ_ERR_ARG
    assert L.fz_get_stats(None, None) == fz.FZ_ERR_ARG
    L.fz_destroy(None)


def test_binding_refuses_missing_library(tmp_path, monkeypatch):
    monkeypatch.setattr(fz, "_lib", None)
    with pytest.raises(FileNotFoundError):
        fz.load(str(tmp_path / "nope.so"))
    monkeypatch.setattr(fz, "_lib", None)


def test_no_cpu_fallback_in_product_path():
    """The package never imports the oracle."""
    pkg = os.path.dirname(fz.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_combine_rejects_null_context_without_gpu(lib):
    assert lib.fz_combine(None, None, 0, None, None, None, None, None) == fz.FZ_ERR_ARG


def test_pair_sweep_rule(lib, monkeypatch):
    """The host-only rule that picks the 16-bit first tier (and with it the
    roofline's cells per lane): the benchmark scoring takes it; a y-drop or gap
    costs past the 16-bit range, scores outside bytes, no pruning, the local
    mode and FZ_NO_PAIR=1 do not."""
    monkeypatch.delenv("FZ_NO_PAIR", raising=False)
    hox = W.HOXD70
    assert fz.fz_pair_sweep_used(hox, 400, 30, 9400, W.MODE_EXTEND)
    # ydrop + 2048 + 4 (o + e + max|M|) <= 30000: HOXD70 (max 125), o + e = 430 leaves ydrop <= 25732
    assert fz.fz_pair_sweep_used(hox, 400, 30, 25732, W.MODE_EXTEND)
    assert not fz.fz_pair_sweep_used(hox, 400, 30, 25733, W.MODE_EXTEND)
    assert not fz.fz_pair_sweep_used(hox, 400, 30, W.YDROP_INF, W.MODE_EXTEND)
    assert not fz.fz_pair_sweep_used(hox * 3, 1200, 90, 9400, W.MODE_EXTEND)      # scores beyond a byte
    assert not fz.fz_pair_sweep_used(hox, 1900, 30, 2000, W.MODE_EXTEND)         # o + e + max|M| + 16 >= 2048
    assert not fz.fz_pair_sweep_used(hox, 400, 30, 9400, W.MODE_LOCAL)
    monkeypatch.setenv("FZ_NO_PAIR", "1")
    assert not fz.fz_pair_sweep_used(hox, 400, 30, 9400, W.MODE_EXTEND)
    monkeypatch.setenv("FZ_NO_PAIR", "0")
    assert fz.fz_pair_sweep_used(hox, 400, 30, 9400, W.MODE_EXTEND)
