"""Host logic of bench.py that needs no GPU: the percentile helper, the
per-workload table of the bench line's "configs" (every workload of the
configuration list, with its dispatch payloads), and the clock sampler's
selection of samples inside the timed region."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_percentiles():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.pct(xs, 50) == 3.0
    assert bench.pct(xs, 0) == 1.0 and bench.pct(xs, 100) == 5.0
    assert abs(bench.pct(xs, 10) - 1.4) < 1e-12


def test_every_workload_is_in_the_configs_table():
    assert set(bench.CONFIG_RUNS) == set(synth.CONFIGS)
    for name, payloads in bench.CONFIG_RUNS.items():
        assert payloads and set(payloads) <= {"bf16", "fp8"}
        cfg = synth.config(name)
        if "fp8" in payloads:
            assert cfg["H"] % 128 == 0
    # the two workloads quoted with both payloads take both
    assert set(bench.CONFIG_RUNS["skewed"]) == {"bf16", "fp8"}
    assert set(bench.CONFIG_RUNS["decode"]) == {"bf16", "fp8"}


def test_op_bytes_match_the_algorithmic_formulas():
    cfg = synth.config("dsv3")
    T, H, k = cfg["T"], cfg["H"], cfg["k"]
    b = bench.op_bytes(cfg)
    assert b["dispatch_bf16"] == T * (2 * H + 2 * H * k + 4 * k)
    assert b["dispatch_fp8"] == T * (2 * H + k * (H + 4 * (H // 128)) + 4 * k)
    assert b["combine"] == T * (2 * H * k + 8 * k + 2 * H)
    assert b["combine"] == 1057488896


def test_clock_summary_keeps_only_the_timed_region():
    c = bench.ClockSampler(0)
    c.samples = [(0.5, 1000.0, 2070.0, [False] * 4),
                 (1.5, 2070.0, 2070.0, [False, False, False, True]),
                 (2.0, 2000.0, 2070.0, [False] * 4),
                 (3.5, 500.0, 2070.0, [True, False, False, False])]
    c.t0, c.t1 = 1.0, 3.0
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == np.median([2070.0, 2000.0])
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    c.t0, c.t1 = 10.0, 11.0
    assert c.summary()["samples"] == 0
