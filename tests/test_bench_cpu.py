"""bench.py without a GPU: every selectable workload is constructed, reports
its configuration and roofline inputs, and names a dominant kernel whose
sources exist (their hash ties the committed ncu summaries to the code)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


BENCH = _bench()


@pytest.mark.parametrize("name", BENCH.WORKLOADS)
def test_workload_describes_itself(name):
    wl = BENCH.make_workload(name)
    cfg = wl.config()
    assert isinstance(cfg.get("workload"), str) and cfg["workload"]
    assert wl.T > 0 and wl.bytes_per_token > 0
    assert wl.launches_per_step > 0
    fma = getattr(wl, "fma_per_token", None)
    assert fma is None or fma > 0
    assert wl.dominant_src in BENCH.KERNEL_SOURCES
    assert len(BENCH.kernel_sources_sha(wl.dominant_src)) == 16


def test_unknown_workload_is_refused():
    with pytest.raises(SystemExit):
        BENCH.make_workload("no_such_workload")


def test_aggregate_is_the_whole_job_rate():
    # all ranks' tokens over the slowest rank's time
    assert BENCH.aggregate(1000, 10, 4, 2000.0) == pytest.approx(1000 * 10 * 4 / 2.0)
