"""Host-side logic of bench.py that needs no GPU: folding the traced launches into per-kind
figures (a K-split fixup belongs to the dW or dH launch just before it) and the traffic
constants' validity."""
import pytest

import bench


class FakeTrace:
    """Stands in for the library's fkl_trace_read with a fixed list of (ms, kind, flops)."""

    def __init__(self, entries):
        self.entries = entries

    def fkl_trace_read(self, ms, kind, flops, cap):
        n = min(len(self.entries), cap)
        for i in range(n):
            ms[i], kind[i], flops[i] = self.entries[i]
        return n


def test_fixup_time_is_folded_into_the_product_it_completes():
    e = [(20.0, 0, 4e13), (1.0, 1, 2e12), (1.2, 2, 2e12), (0.1, 4, 0.0), (1.3, 3, 2e12), (0.05, 4, 0.0),
         (1.0, 1, 2e12), (1.2, 2, 2e12), (1.4, 3, 2e12), (0.05, 4, 0.0)]
    k = bench.trace_summary(FakeTrace(e), 64)
    assert set(k) == {0, 1, 2, 3}
    assert k[2]["launches"] == 2 and k[2]["fixup_launches"] == 1
    assert k[3]["launches"] == 2 and k[3]["fixup_launches"] == 2
    assert k[3]["ms_total"] == pytest.approx(1.3 + 0.05 + 1.4 + 0.05)
    assert k[2]["tflops"] == pytest.approx(4e12 / (2.5e-3) / 1e12)
    assert sum(v["launches"] + v["fixup_launches"] for v in k.values()) == len(e)


def test_a_full_trace_is_an_error():
    e = [(1.0, 1, 2e12)] * 8
    with pytest.raises(RuntimeError):
        bench.trace_summary(FakeTrace(e), 8)
    assert bench.trace_summary(FakeTrace(e), 9)[1]["launches"] == 8


def test_traffic_is_reported_only_for_the_measured_sources_and_shape():
    f = bench.TRAFFIC_FLOPS[3]
    if bench.csrc_sha() == bench.TRAFFIC_SOURCES_SHA:
        assert bench.traffic_per_launch(3, f, 2880) == pytest.approx(bench.TRAFFIC_BYTES[3])
        assert bench.traffic_per_launch(3, f / 2, 2880) == pytest.approx(bench.TRAFFIC_BYTES[3] / 2)
    assert bench.traffic_per_launch(3, f, 4096) is None
    assert bench.traffic_per_launch(9, f, 2880) is None

