"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes must give up, record its bit in the device status word and return,
leaving the context usable."""
import time

import numpy as np
import pytest

import attention_residual_fusion_gb300 as ar
import oracle
from attention_residual_fusion_gb300 import _build
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    ar.lib()


def test_wait_timeout_is_reported_and_recoverable():
    ar.device_status(clear=True)
    t0 = time.perf_counter()
    bits = ar.selftest_wait_timeout(20000)  # 20 ms
    dt = time.perf_counter() - t0
    assert bits & 1, "the wait did not report its time-out"
    assert dt >= 0.015, "the wait returned before its limit"
    assert ar.device_status(clear=True) & 1
    assert ar.device_status() == 0
    # the context still works: a normal call right after is correct
    wl = W.make_workload(3, 4, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=5, seed=21, mixing=True)
    ref = oracle.run_workload(wl)
    gpu = G.run_gpu(wl)
    G.check_against_oracle(wl, gpu, ref, tag="after-timeout")
    assert ar.device_status() == 0


def test_selftest_rejects_bad_limits():
    for bad in (0, 2_000_000):
        with pytest.raises(ar.AttnResError):
            ar.selftest_wait_timeout(bad)
