"""Host checks of bench.py's option handling (no GPU): combinations that name no
measurable leg are refused before any device work."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=300)


def test_prefill_needs_a_prefill_stack():
    r = _bench("--prefill")   # the default layer has no prefill stack
    assert r.returncode == 2 and "--prefill needs a workload with a prefill stack" in r.stderr


def test_prefill_refuses_the_paged_cache():
    r = _bench("--workload", "ouro_rho4_b64_16k", "--prefill", "--paged", "256")
    assert r.returncode == 2 and "--prefill" in r.stderr


def test_warmup_floor():
    r = _bench("--warmup", "2")
    assert r.returncode == 2 and "--warmup must be >= 3" in r.stderr


def test_reference_arm_other_ranks_exit_without_work():
    """Under a launcher with N > 1 the reference arm (the oracle on the host cores) runs
    on rank 0 only; every other rank exits 0 at once and prints nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """Rank 0's reference line: the oracle timed on a bounded sample of the headline
    workload, in the GPU arm's metric and unit, with the keys the driver reads."""
    import json
    r = _bench("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "ouro1.4b_rho4_b32_4k"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["steps"] == 3 and d["warmup"] == 3
