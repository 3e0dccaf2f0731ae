"""bench.py's reference arm (the CPU oracle) on CPU: its run time follows
--reference-seconds whatever --steps and --warmup are, because every step runs
one sample sized from a single probe."""
import json
import re
import subprocess
import sys
import time
from pathlib import Path

REPO = Path(__file__).resolve().parent.parent


def _reference_line(*args, timeout=300):
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, str(REPO / "bench.py"), "--impl", "reference", *args],
                         cwd=REPO, capture_output=True, text=True, timeout=timeout)
    wall = time.perf_counter() - t0
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0]), wall


def test_many_steps_stay_within_the_budget():
    """2000 + 3 steps of the Mamba-130M-shaped layer in a 3-second budget: every
    step runs a small sample, and the whole run ends in seconds (the probe,
    the oracle build and interpreter start-up on top)."""
    d, wall = _reference_line("--workload", "1", "--steps", "2000", "--warmup", "3",
                              "--reference-seconds", "3")
    assert d["impl"] == "reference" and d["steps"] == 2000 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "state-updates/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["ms_per_step"] * 2000 / 1e3 < 10.0
    assert wall < 120.0


def _sample_size(line):
    """(batch rows, channels) of the per-step sample the line reports."""
    m = re.match(r"the first (\d+) of \d+ batch rows x the first (\d+) of \d+ channels",
                 line["cpu_baseline"]["sample"])
    assert m, line["cpu_baseline"]["sample"]
    return int(m.group(1)), int(m.group(2))


def test_sample_grows_with_the_budget():
    """A larger budget per step takes a larger sample of the same workload (a
    tiny one: part of the batch rows of one channel)."""
    small, _ = _reference_line("--workload", "1", "--steps", "4", "--warmup", "0",
                               "--reference-seconds", "1e-7")
    large, _ = _reference_line("--workload", "1", "--steps", "4", "--warmup", "0",
                               "--reference-seconds", "4")
    nb_s, ch_s = _sample_size(small)
    nb_l, ch_l = _sample_size(large)
    assert (nb_s, ch_s) == (1, 1)
    assert nb_l * ch_l > nb_s * ch_s
