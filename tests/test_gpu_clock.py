"""The clock-stamp measurement aid on the GPU: two stamps around a stretch of
work give every SM an average clock no faster than its maximum, and the SM
ids, cycle counters and timer behave as the header states."""

import pytest
import torch

import paged_kv_cache_46_gb300 as ts

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()


def test_two_stamps_give_each_sm_a_plausible_clock():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    a = torch.zeros(2 * sms, 3, dtype=torch.int64, device=DEV)
    b = torch.zeros_like(a)
    x = torch.randn(4096, 4096, device=DEV)
    ts.ts_clock_stamp(a)
    for _ in range(20):
        x = torch.tanh(x @ x * 1e-3)  # a few ms of work between the stamps
    ts.ts_clock_stamp(b)
    torch.cuda.synchronize()
    a, b = a.cpu(), b.cpu()
    assert int(a[:, 0].max()) < sms and int(b[:, 0].max()) < sms and int(a[:, 0].min()) >= 0
    first = {}
    for sm, clk, ns in a.tolist():
        first.setdefault(sm, (clk, ns))
    mhz = []
    for sm, clk, ns in b.tolist():
        if sm in first:
            dc, dt = clk - first[sm][0], ns - first[sm][1]
            assert dc > 0 and dt > 0
            mhz.append(dc / dt * 1e3)
    assert len(mhz) >= sms // 2
    mhz.sort()
    med = mhz[len(mhz) // 2]
    # the maximum SM clock of the part is 2070 MHz; allow timer granularity
    assert 200.0 < med < 2300.0, med


def test_bad_stamp_tensor_is_rejected():
    with pytest.raises(ts.TSError):
        ts.ts_clock_stamp(torch.zeros(4, 2, dtype=torch.int64, device=DEV))
