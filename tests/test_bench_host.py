"""Host-side logic of bench.py: the copy/step overlap summary and the
reference arm's JSON line (the CPU oracle timed on the host cores)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_copy_overlap_counts_steps_and_loss():
    steps = [(0.0, 1.0), (1.0, 2.0), (2.0, 3.5), (3.5, 5.0), (5.0, 6.0), (6.0, 7.0)]
    out = bench.copy_overlap(steps, [(1.5, 4.0)])
    assert len(out) == 1
    o = out[0]
    assert o["copy_ms"] == pytest.approx(2.5)
    assert o["steps_overlapped"] == 3  # (1,2), (2,3.5), (3.5,5)
    # overlapped 1 + 1.5 + 1.5 = 4 against 3 x the median 1.0 of the others
    assert o["step_ms_lost"] == pytest.approx(1.0)


def test_copy_overlap_touching_intervals_do_not_overlap():
    steps = [(0.0, 1.0), (1.0, 2.0), (2.0, 3.0)]
    out = bench.copy_overlap(steps, [(1.0, 2.0), (3.0, 4.0)])
    assert out[0]["steps_overlapped"] == 1 and out[0]["step_ms_lost"] == pytest.approx(0.0)
    assert out[1]["steps_overlapped"] == 0 and out[1]["step_ms_lost"] == 0


def test_copy_overlap_without_copies():
    assert bench.copy_overlap([(0.0, 1.0)], []) == []


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
         "--cpu-seconds", "0.25", "--workload", "flat-65536"],
        cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "flat-65536"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched like the multi-GPU bench (torchrun, 2 ranks): rank 0 alone
    times the oracle and prints; the other rank exits 0 without output."""
    r = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
         "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
         "--cpu-seconds", "0.25", "--workload", "flat-65536"],
        cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_kernel_stats_rates_and_fractions():
    # two steps of n = 1e6 parameters: norm 0.001 ms and 0.003 ms (mean 0.002),
    # fused 0.01 ms each; 4 and 28 algorithmic bytes per parameter
    n = 1_000_000
    ks = bench.kernel_stats([(0.001, 0.01), (0.003, 0.01)], n, peak=2000.0)
    assert ks["k_grad_norm"]["avg_ms"] == pytest.approx(0.002)
    assert ks["k_grad_norm"]["min_ms"] == pytest.approx(0.001)
    assert ks["k_grad_norm"]["GB/s"] == pytest.approx(4 * n / 0.002 / 1e6)   # 2000 GB/s
    assert ks["k_grad_norm"]["frac"] == pytest.approx(1.0)
    assert ks["k_clip_adamw"]["GB/s"] == pytest.approx(28 * n / 0.01 / 1e6)  # 2800 GB/s
    assert ks["k_clip_adamw"]["frac"] == pytest.approx(1.4)
    assert ks["k_clip_adamw"]["frac_of_nominal_8tbs"] == pytest.approx(2800 / 8000)


def test_guarded_config_reports_its_error():
    def boom(x):
        raise MemoryError(f"no room for {x}")
    out = bench._guarded(boom, "flat-2^30")
    assert out == {"error": "MemoryError: no room for flat-2^30"}
    assert bench._guarded(lambda a, b: a + b, 2, 3) == 5
