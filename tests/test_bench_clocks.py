"""The benchmark's clock record on the CPU, from samples given to it (no GPU, no NVML): the median
SM clock over the sampled region and its mean (the time-averaged clock the tensor duty divides by),
the clock-event reasons named from their NVML bits, and the sample count. Only queries are made by the sampler; these tests make none."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(rows, max_mhz=2070.0):
    c = bench.ClockSampler("GPU-test")
    c.nvml = ("lib", "handle", None)  # as if NVML had opened; summary reads only the rows
    c.max_mhz = max_mhz
    c.rows = rows
    return c


def test_every_sample_counts_and_the_median_is_taken():
    # power readings that trail the load (a moving average) must not drop samples
    rows = [(1700.0, 120.0, 0), (1750.0, 250.0, 0x4), (1800.0, 900.0, 0x4), (1720.0, 1300.0, 0)]
    s = _sampler(rows).summary()
    assert s["samples"] == 4
    assert s["sm_mhz"] == 1735.0
    assert s["sm_mhz_mean"] == 1742.5
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_slowdown_reasons_are_named():
    rows = [(1500.0, 1000.0, 0x8 | 0x40), (1510.0, 1000.0, 0x20)]
    assert _sampler(rows).summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_no_samples_is_reported_as_such():
    s = _sampler([]).summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["no samples"]
