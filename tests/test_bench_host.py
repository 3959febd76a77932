"""Host logic of the measurement: the algorithmic bytes behind the roofline's
numerator (hand-computed for the 128K Llama-3.1-8B-shaped step) and the summary
of the clock samples taken during the timed region (median SM clock under load,
throttle reasons), on a fake sample file -- no GPU, no nvidia-smi."""
import os

import pytest

import bench

pytestmark = pytest.mark.cpu


def test_algorithmic_bytes_of_the_128k_step():
    total, crit, rows, l0 = bench.algorithmic_bytes(131072)
    assert l0 == 8 * 131072 * 48                        # 1-bit K/V codes + (scale, zero) pairs
    assert crit == 32 * 8 * 131072 * 2                  # 8 fp16 critical keys per token and q head
    assert rows == 32 * (4 + 128 + 3932) * 512          # selected K and V rows per q head
    assert total == l0 + 31 * (crit + rows) == 4_194_828_288


def test_algorithmic_bytes_scale_with_layers():
    t1 = bench.algorithmic_bytes(4096, n_layers=1)[0]
    t3 = bench.algorithmic_bytes(4096, n_layers=3)[0]
    _, crit, rows, l0 = bench.algorithmic_bytes(4096)
    assert t1 == l0 and t3 == l0 + 2 * (crit + rows)


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _summary(tmp_path, lines):
    path = os.path.join(tmp_path, "clocks.csv")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    c = bench.Clocks.__new__(bench.Clocks)
    c.proc, c.path, c.f = _Done(), path, open(os.devnull, "w")
    return c.stop()


def _row(sm, reasons=()):
    flags = ["Active" if r in reasons else "Not Active"
             for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    return ", ".join(["0", str(sm), "2070", "900.5", "0x0"] + flags)


def test_clock_summary_under_load(tmp_path):
    s = _summary(str(tmp_path), [_row(345), _row(2070), _row(2055), _row(2070), "garbage"])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4}


def test_clock_summary_reports_throttle_reasons(tmp_path):
    s = _summary(str(tmp_path), [_row(1800, ("sw_power_cap",)), _row(1500, ("hw_slowdown", "sw_power_cap")),
                                 _row(1900)])
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["sm_mhz"] == 1800.0 and s["samples"] == 3


def test_clock_summary_without_samples(tmp_path):
    assert _summary(str(tmp_path), []) is None
