"""The issue-rate probe the benchmark reports beside the head's ALU roofline."""
import pytest

pytestmark = pytest.mark.gpu

NOMINAL_LANE_OPS = 148 * 128 * 2032e6  # one instruction per lane per clock at the max clock


def test_probe_rates_are_physical(dust):
    rates = {}
    for kind, iters in ((0, 4000), (1, 2000), (2, 20000)):
        dust.issue_probe(kind, 16)
        rates[kind], ms = dust.issue_probe(kind, iters)
        assert ms > 0.1
    # fp32 fma issues at about one instruction per lane and clock, never above
    assert 0.5 * NOMINAL_LANE_OPS < rates[2] < 1.05 * NOMINAL_LANE_OPS, rates
    # the XU pipe and the 64-bit multiply are slower than plain fma
    assert rates[1] < rates[2] and rates[0] < 1.05 * NOMINAL_LANE_OPS, rates


def test_probe_rejects_bad_kind(dust):
    with pytest.raises(dust.DustError):
        dust.issue_probe(5, 10)
