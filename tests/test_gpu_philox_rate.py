"""The ALU roof the benchmark reports: dspark_selftest_philox_rate measures
the blocks per second of the draft's own Philox4x32-10 code on this device.
"""
import pytest

from speculative_decoding_draft_head_gb300 import binding

pytestmark = pytest.mark.gpu


def test_philox_rate_probe_reports_a_plausible_rate():
    # between 10^10 and 10^13 blocks per second on any GPU this library targets
    rate = binding.selftest_philox_rate(64)
    assert 1e10 < rate < 1e13
    # a longer run measures the same rate within a factor of two
    rate2 = binding.selftest_philox_rate(512)
    assert 0.5 < rate2 / rate < 2.0
