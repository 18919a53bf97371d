"""Failure detection on the GPU without a fault: every wait in the library's kernels is bounded,
and a wait that runs out reports PCF_ERR_DEVICE_TIMEOUT through the device error word while the
device stays usable.  The check kernel waits, with a short limit, on a barrier that nothing arrives
on; the production kernels are not altered."""
from __future__ import annotations

import pytest
import torch

import position_independent_kv_critical_gb300 as pcf
from workload import make_batch

from gpu_util import GpuBatch, assert_close_imp

pytestmark = pytest.mark.gpu

PCF_ERR_DEVICE_TIMEOUT = -4


@pytest.mark.parametrize("limit", [100_000, 2_000_000])
def test_a_wait_that_runs_out_reports_a_timeout_and_the_device_stays_usable(limit):
    pcf.check_device_error()                      # start from a clean error word
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pcf.wait_limit_check(limit, flag)
    with pytest.raises(pcf.PcfError) as e:
        pcf.check_device_error()
    assert e.value.status == PCF_ERR_DEVICE_TIMEOUT
    assert int(flag.item()) == 1                  # the wait returned false: it gave up
    pcf.check_device_error()                      # the word was cleared
    # the same stream runs the hot path correctly right after
    gb = GpuBatch(make_batch("tiny"))
    imp = gb.score()
    n = gb.b.requests[0].n_cached
    assert_close_imp(imp[:n], gb.oracle_score(0), "scoring after a timed-out wait")


def test_timeout_on_a_side_stream_is_seen_by_its_check():
    pcf.check_device_error()
    s = torch.cuda.Stream()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pcf.wait_limit_check(50_000, flag)
    with pytest.raises(pcf.PcfError) as e:
        pcf.check_device_error(s)
    assert e.value.status == PCF_ERR_DEVICE_TIMEOUT
    pcf.check_device_error(s)
