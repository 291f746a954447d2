"""Host logic of bench.py (no GPU): the reference arm's JSON line, the clock
sampler's parsing of nvidia-smi samples, and the lookup of committed DRAM
traffic (taken only for the same workload and an unchanged kernel source)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gapped_smith_waterman_gb300 import workloads as W  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    p = _run(["--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "0"])
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["unit"] == "GCUPS" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "short-256bp"


def test_wide_band_workload_and_its_reference_line():
    """The general-band batch: 512 right extensions of 3 kbp windows at y-drop
    40,000, each query a mutated copy of its whole target window; the
    reference arm times the oracle on it."""
    w = W.make_wide()
    assert w.ydrop == 40000 and w.max_len == 3000 and len(w.seeds) == 512
    assert np.all(w.seeds["side"] == W.SIDE_RIGHT)
    import oracle
    t0, q0 = w.target[:300], w.query[:300]
    d = oracle.edit_distance(t0, q0)                              # homologous, not identical
    assert 0 < d < 0.35 * 300 < oracle.edit_distance(t0, w.query[3000:3300])
    p = _run(["--impl", "reference", "--wide", "--steps", "1", "--warmup", "0", "--ref-step-seconds", "1"])
    assert p.returncode == 0, p.stderr
    d = json.loads([l for l in p.stdout.splitlines() if l.strip()][0])
    assert d["config"]["workload"] == "wide-band-3kbp" and d["value"] > 0


def test_reference_arm_other_ranks_print_nothing():
    p = _run(["--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "0"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_clock_sampler_parses_samples_and_reasons(tmp_path):
    s = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    path.write_text("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "0, 1950, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "garbage line\n")
    s.path = str(path)

    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = _P()
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert not path.exists()


def test_clock_sampler_without_samples():
    s = bench.ClockSampler(0)
    assert s.stop()["reasons"] == ["clocks not sampled"]


def _kernel(mode):
    return bench.LOCAL_KERNEL if mode == "local" else bench.PHASES[0]


def _fake_tree(tmp_path, mode, config, src_bytes, traffic):
    import hashlib
    _, src, _, _, prof_name = _kernel(mode)
    (tmp_path / "profiles").mkdir(exist_ok=True)
    csrc = tmp_path / "gapped_smith_waterman_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / src).write_bytes(src_bytes)
    (tmp_path / "profiles" / prof_name).write_text(json.dumps({
        "config": config, "source_sha1": hashlib.sha1(src_bytes).hexdigest(),
        "dram_bytes_per_launch_full_batch": traffic}))
    return csrc / src


@pytest.mark.parametrize("mode", ["extend", "local"])
def test_traffic_only_for_the_captured_workload_and_source(mode, monkeypatch, tmp_path):
    src = _fake_tree(tmp_path, mode, 2, b"// kernel source\n", 123456)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    k = _kernel(mode)
    assert bench.traffic_for_kernel(k, 2) == 123456
    assert bench.traffic_for_kernel(k, 3) is None           # another workload
    src.write_bytes(b"// kernel source, changed\n")
    assert bench.traffic_for_kernel(k, 2) is None           # the kernel changed since
    (tmp_path / "profiles" / k[4]).unlink()
    assert bench.traffic_for_kernel(k, 2) is None           # no capture


def test_every_phase_kernel_names_a_source_file():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for k in list(bench.PHASES.values()) + [bench.LOCAL_KERNEL]:
        assert os.path.exists(os.path.join(root, "gapped_smith_waterman_gb300", "csrc", k[1])), k


def test_cpu_model_is_a_nonempty_string():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


@pytest.mark.parametrize("ws", [1, 2, 3, 8])
def test_rank_shards_cover_the_batch_in_order(ws):
    seeds = np.zeros(1001, W.SEED_DTYPE)
    seeds["t_pos"] = np.arange(1001)
    parts = [bench.rank_seeds(seeds, r, ws) for r in range(ws)]
    joined = np.concatenate(parts)
    assert np.array_equal(joined["t_pos"], seeds["t_pos"])
    sizes = [len(p) for p in parts]
    assert max(sizes) - min(sizes) <= 1
