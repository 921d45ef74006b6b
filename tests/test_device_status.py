"""Failure detection on the GPU without a fault: every pipeline wait in the kernels is bounded.
A diagnostic kernel waits on a barrier phase nothing completes; the wait must give up after its
short limit, record FA_ERR_DEVICE_TIMEOUT in the device status word and exit, leaving the CUDA
context usable for the next call."""
import math
import time

import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import normal_bf16
from tests.helpers import bf16_to_f64, compare, to_dev

pytestmark = pytest.mark.gpu

FA_ERR_DEVICE_TIMEOUT = 7
SELFTEST_SITE = 99


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch

    import io_aware_exact_flash_gb300 as fa

    t0 = time.perf_counter()
    code, site = fa.fa_selftest_wait_timeout(50)
    elapsed = time.perf_counter() - t0
    assert code == FA_ERR_DEVICE_TIMEOUT and site == SELFTEST_SITE
    assert elapsed < 1.5, f"the 50 ms wait took {elapsed:.2f} s"
    assert fa.fa_get_device_status() == (0, 0)  # reading cleared it
    # the context is still usable: a normal forward runs and is correct
    q, k, v = (normal_bf16(8, (1, 300, 2, 64), stream=s) for s in range(3))
    o, lse = fa.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=1 / math.sqrt(64))
    torch.cuda.synchronize()
    o_ref, lse_ref, va_ref = oracle.get().dense(q, k, v, True, 1 / math.sqrt(64), vabs=True)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref, "after timeout", vabs=va_ref)
    assert fa.fa_get_device_status() == (0, 0)


def test_selftest_argument_checks():
    import io_aware_exact_flash_gb300 as fa

    for bad in (0, -5, 2001):
        with pytest.raises(fa.FaError):
            fa.fa_selftest_wait_timeout(bad)
