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
