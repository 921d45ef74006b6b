"""The fp64 oracle against facts the definition of exact attention fixes (CPU only)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.get())


def test_thread_count_does_not_change_results():
    import numpy as np

    from io_aware_exact_flash_gb300.workloads import normal_bf16

    q = normal_bf16(5, (1, 64, 2, 16))
    k = normal_bf16(6, (1, 64, 2, 16))
    v = normal_bf16(7, (1, 64, 2, 16))
    o1, l1 = oracle.get().dense(q, k, v, True, 0.25, threads=1)
    o7, l7 = oracle.get().dense(q, k, v, True, 0.25, threads=7)
    assert np.array_equal(o1, o7) and np.array_equal(l1, l7)
