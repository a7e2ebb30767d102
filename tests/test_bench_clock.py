"""bench.py's device clock summary (CPU): from two sets of per-SM stamps
(SM id, cycle counter, global timer ns) it reports each SM's average clock
over the window, matched by SM, with repeated SM ids and SMs missing from
one set handled."""

import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_device_clock_matches_by_sm():
    # SM 0 at 2000 MHz, SM 1 at 1000 MHz, SM 2 only in the first set, SM 0 twice
    a = torch.tensor([[0, 1_000, 10_000], [1, 5_000, 10_000], [2, 0, 10_000], [0, 1_100, 10_050]],
                     dtype=torch.int64)
    b = torch.tensor([[1, 5_000 + 1_000_000, 1_010_000], [0, 1_000 + 2_000_000, 1_010_000]], dtype=torch.int64)
    d = bench.device_clock(a, b)
    assert d["device_sms"] == 2
    assert d["sm_mhz_device_min"] == 1000.0
    assert d["sm_mhz_device"] in (1000.0, 2000.0, 1500.0)
    assert d["device_window_us"] == 1000.0


def test_device_clock_without_matches():
    a = torch.tensor([[3, 0, 0]], dtype=torch.int64)
    b = torch.tensor([[4, 10, 10]], dtype=torch.int64)
    assert bench.device_clock(a, b) == {"sm_mhz_device": None}
