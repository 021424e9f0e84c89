"""Host logic of bench.py (no GPU): which clock samples count, and how many
kernels a step claims.

The clock record must come from inside the timed regions: samples carry
nvidia-smi's timestamp and only those within a marked region (20 ms slack)
enter the median and the throttle reasons.  The launch counts mirror the
dispatch in the C library for the workloads the bench runs.
"""
import datetime
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _line(t, sm, reasons=("Not Active",) * 4):
    return f"{t.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, {sm}, 2070, 950.00, " + ", ".join(reasons)


def test_only_samples_inside_the_timed_regions_count(bench):
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0)
    ms = lambda x: t0 + datetime.timedelta(milliseconds=x)  # noqa: E731
    c = bench.ClockSampler(0)
    c.lines = [
        _line(ms(0), 900, ("Active", "Not Active", "Not Active", "Not Active")),   # warm-up, throttled: outside
        _line(ms(100), 2070),
        _line(ms(120), 2055),
        _line(ms(140), 2070, ("Not Active", "Not Active", "Not Active", "Active")),  # power cap inside
        _line(ms(400), 1200, ("Not Active", "Active", "Not Active", "Not Active")),  # between regions
        _line(ms(600), 2070),
        "garbage line",
        _line(ms(2000), 800),                                                    # after the last region
    ]
    c.mark(ms(95), ms(150))
    c.mark(ms(590), ms(610))
    s = c.summary()
    assert s["samples"] == 4
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_no_sample_in_a_region_reads_unsampled(bench):
    c = bench.ClockSampler(0)
    t = datetime.datetime(2026, 12, 2, 10, 0, 0)
    c.lines = [_line(t, 2070)]
    c.mark(t + datetime.timedelta(seconds=1), t + datetime.timedelta(seconds=2))
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}


def test_launch_counts_follow_the_dispatch(bench):
    from compressed_sparse_attention_compress_gb300.inputs import WORKLOADS
    wl = WORKLOADS["warmup32k"]
    # both compressors with the offsets, top-k + capacity fill, attention + capacity rows, KL zero + KL + finalize
    assert bench.f_launches(wl) == 1 + 2 + 2 + 3
    # the v4 compressor: offsets and one call per stream
    import dataclasses
    assert bench.f_launches(dataclasses.replace(wl, compressor="v4")) == 1 + 2 + 2 + 2 + 3
    # attention backward: delta, capacity rows, kernel; indexer backward: one kernel
    assert bench.b_launches(wl) == 3 + 1
    assert bench.f_launches(WORKLOADS["hca64k"]) == 1 + 1 + 2


def test_dense_kl_traffic_is_its_operands_read_once(bench):
    """The recorded DRAM bytes of one dense-teacher KL launch at 32K are its operands read
    once (queries, indexer queries and weights, the compressed key and indexer-key rows),
    within a few percent: the key prefix stays in L2 for the blocks that share it."""
    from compressed_sparse_attention_compress_gb300 import inputs as I
    wl = I.WORKLOADS["warmup32k"]
    t = bench._traffic("indexer_kl", "warmup32k")
    if t is None:
        pytest.skip("no capture recorded for the current kernel")
    n_c = wl.T // wl.ratio
    algo = wl.T * (wl.H * wl.d + wl.H_I * wl.d_I + wl.H_I) * 2 + n_c * (wl.d + wl.d_I) * 2
    assert 0.98 * algo <= t <= 1.05 * algo, (t, algo)
