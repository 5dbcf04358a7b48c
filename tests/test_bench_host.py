"""Host-side behaviour of bench.py that needs no GPU: rank spawning, the reference arm's line, shared config."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run(*args, timeout=600):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=timeout, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


def test_gpus_two_starts_two_ranks():
    """--gpus 2 outside a launcher starts two ranks itself (gloo here; NCCL, one rank per GPU, for the bench)."""
    out = _run("--gpus", "2", "--selftest-ranks")
    assert out["ranks"] == 2 and out["rank_sum"] == 1.0 and out["gpus"] == 2


def test_reference_arm_line_matches_gpu_config():
    import bench
    out = _run("--impl", "reference", "--config", "2", "--steps", "1", "--warmup", "0")
    wl = bench.make_workload(2)
    assert out["impl"] == "reference"
    assert out["config"] == bench.config_dict(wl, bench.accounting(wl), 1)
    assert out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
    # ms_per_step is the measured wall time of one sample step, not an extrapolation
    assert out["ms_per_step"] < 60e3
    assert str(bench.sample_size()["fwd_rows"]) in out["cpu_baseline"]["sample"]
