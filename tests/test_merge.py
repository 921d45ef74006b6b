"""The LSE-weighted merge of partial attention states against the oracle: attention over a key
set equals the merge of attention over the parts of any partition of it."""
import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import normal_bf16
from tests.helpers import bf16_to_f64, compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cuts,d", [([0, 100, 200, 333], 128), ([0, 1, 2, 333], 64), ([0, 333], 128),
                                    ([0, 50, 50, 333], 128)])
def test_merge_equals_full_attention(cuts, d):
    import torch

    import io_aware_exact_flash_gb300 as fa

    n, H, S = 6, 4, 333
    q = normal_bf16(3, (1, n, H, d), stream=0)
    k = normal_bf16(3, (1, S, H, d), stream=1)
    v = normal_bf16(3, (1, S, H, d), stream=2)
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:  # an empty part: no keys; its O carries NaN that must never be read
            parts_o.append(np.full((n, H, d), np.nan))
            parts_l.append(np.full((n, H), -np.inf))
            continue
        o_p, l_p = oracle.get().dense(q, np.ascontiguousarray(k[:, a:b]), np.ascontiguousarray(v[:, a:b]), False, 0.1)
        parts_o.append(o_p[0])
        parts_l.append(l_p[0])
    o_parts = torch.tensor(np.stack(parts_o), dtype=torch.float32, device="cuda")
    l_parts = torch.tensor(np.stack(parts_l), dtype=torch.float32, device="cuda")
    o, lse = fa.fa_merge_states(o_parts, l_parts)
    torch.cuda.synchronize()
    o_ref, lse_ref, va_ref = oracle.get().dense(q, k, v, False, 0.1, vabs=True)
    compare(bf16_to_f64(o), o_ref[0], lse.cpu().numpy(), lse_ref[0], f"merge {cuts}", vabs=va_ref[0])


def test_merge_all_parts_empty():
    import torch

    import io_aware_exact_flash_gb300 as fa

    o_parts = torch.full((3, 2, 2, 64), float("nan"), device="cuda")
    l_parts = torch.full((3, 2, 2), float("-inf"), device="cuda")
    o, lse = fa.fa_merge_states(o_parts, l_parts)
    assert bool((o == 0).all()) and bool(torch.isneginf(lse).all())
