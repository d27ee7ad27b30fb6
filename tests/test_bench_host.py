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
