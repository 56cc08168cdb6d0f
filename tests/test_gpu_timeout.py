"""Failure detection on the device, without a fault: a kernel whose barrier wait
can never complete gives up after the library's wait limit, the host reads the
timeout and its wait site from the device status word, and the GPU keeps
working (a GEMM after it still matches the oracle)."""

import time

import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, B, DeviceWeight, assert_device_status_ok, run_gemm

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    b = B()
    assert_device_status_ok()                       # nothing pending from earlier tests
    t0 = time.perf_counter()
    b.selftest_wait_timeout()
    code, site = b.device_status()                  # synchronises, reads, clears
    waited = time.perf_counter() - t0
    assert (code, site) == (b.ERR_DEVICE_TIMEOUT, b.SELFTEST_SITE), (code, site, b.last_error())
    assert "timed out" in b.last_error()
    assert 0.9 < waited < 30, waited                # the one-second limit, not an early return
    assert b.device_status() == (b.OK, 0)           # read-and-clear

    # the context is intact: a GEMM through the C ABI still matches the oracle
    p = synth.Problem(4, 512, 1024, 128, "uint4b8", "bf16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    got = run_gemm(w, x.A)
    ref = orc.linear(x.A, x.q, x.scales, x.zeros, p.group_size, p.dtype)
    assert orc.rel_error(orc.values(got, p.dtype), ref) <= TOL[p.dtype]
    assert torch.cuda.is_available()
    assert_device_status_ok()
