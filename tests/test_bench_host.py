"""Host logic of the benchmark without a GPU: the clock sampler keeps the
nvidia-smi samples taken inside the timed window."""
import datetime
import os
import tempfile

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _row(t, sm, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), "2070", "900.00", "0x0"] + list(reasons))


def _sampler(rows, window):
    cs = bench.ClockSampler(0)
    fd, cs.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(rows) + "\n")
    cs.proc = _Done()
    cs.window = list(window)
    return cs


def test_samples_inside_the_window_are_kept():
    t0 = 1_800_000_000.0
    rows = [_row(t0 - 0.2, 1200), _row(t0 + 0.05, 2070), _row(t0 + 0.10, 2040),
            _row(t0 + 0.15, 2070, ("Not Active", "Not Active", "Not Active", "Active")),
            _row(t0 + 0.40, 900)]
    r = _sampler(rows, (t0, t0 + 0.2)).stop()
    assert r["samples_in_window"] == 3 and r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_no_sample_in_the_window_falls_back_to_all():
    t0 = 1_800_000_000.0
    rows = [_row(t0 - 1.0, 2000), _row(t0 + 1.0, 2070)]
    r = _sampler(rows, (t0, t0 + 0.1)).stop()
    assert r["samples_in_window"] == 0 and r["samples"] == 2
    assert r["sm_mhz"] == 2035.0


def test_reference_arm_prints_its_line():
    """bench.py --impl reference (the oracle on the host cores): one JSON
    line with the base contract's keys, the oracle's cpu_baseline and an
    e2e object of its own value."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    run = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=root)
    assert run.returncode == 0, run.stderr[-2000:]
    lines = [l for l in run.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    for key in ("metric", "unit", "n_gpus", "ms_per_step", "higher_is_better", "dtype",
                "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
