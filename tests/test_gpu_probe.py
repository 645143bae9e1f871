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


def test_packed_fma_probe_counts_two_operations_per_instruction(dust):
    dust.issue_probe(5, 16)
    packed, ms = dust.issue_probe(5, 20000)
    assert ms > 0.1
    # at most two fp32 operations per lane and clock
    assert 0.25 * NOMINAL_LANE_OPS < packed < 2.1 * NOMINAL_LANE_OPS, packed


def test_probe_rejects_bad_kind(dust):
    with pytest.raises(dust.DustError):
        dust.issue_probe(6, 10)
