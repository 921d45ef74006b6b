"""Seeded random shapes against the fp64 oracle: dense batches (lengths, head counts, GQA groups,
head dims, masking, scales) and paged batches (ragged prefill, chunked prefill and decode rows,
page sizes, groups that do and do not pack, forced and planned key splits, unused pool pages).
Each case is drawn from its own seed, so a failure names a reproducible shape. Q, K and V are
N(0,1), as in the workloads, so rows with a handful of keys (early causal rows, short sequences)
reach |O| of 2 to 4, where the bf16 output rounding alone is 7.8e-3."""
import math

import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import normal_bf16
from tests.helpers import bf16_to_f64, compare, to_dev
from tests.test_parity_paged import build_case, oracle_paged, run_paged

pytestmark = pytest.mark.gpu


def dense_case(i):
    rng = np.random.default_rng(5000 + i)
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, 1101))
    Hkv = int(rng.choice([1, 2, 3, 4]))
    group = int(rng.choice([1, 2, 3, 4, 8]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.uniform(0.03, 0.2))
    return B, S, Hkv * group, Hkv, d, causal, scale


@pytest.mark.parametrize("i", range(48))
def test_fuzz_dense(i):
    import torch

    import io_aware_exact_flash_gb300 as fa

    B, S, Hq, Hkv, d, causal, scale = dense_case(i)
    q = normal_bf16(6000 + i, (B, S, Hq, d), stream=0)
    k = normal_bf16(6000 + i, (B, S, Hkv, d), stream=1)
    v = normal_bf16(6000 + i, (B, S, Hkv, d), stream=2)
    o, lse = fa.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    o_ref, lse_ref, va_ref = oracle.get().dense(q, k, v, causal, scale, vabs=True)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref,
            f"dense case {i}: B={B} S={S} Hq={Hq} Hkv={Hkv} d={d} causal={causal} scale={scale:.3f}", vabs=va_ref)


def paged_case(i):
    rng = np.random.default_rng(7000 + i)
    kind = ("prefill", "chunk", "decode")[i % 3]
    n = int(rng.integers(1, 25))
    lengths = rng.integers(0, 5001 if kind == "decode" else 901, size=n).tolist()
    if kind == "chunk":
        q_lens = [int(rng.integers(1, L + 1)) if L > 0 else 0 for L in lengths]
    elif kind == "decode":
        q_lens = [1] * n
    else:
        q_lens = None
    Hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([g for g in (1, 2, 3, 4, 8) if Hkv * g <= 32]))
    d = int(rng.choice([64, 128]))
    page_size = int(rng.choice([16, 32, 64, 128]))
    causal = bool(rng.integers(0, 2)) if kind != "decode" else True
    splits = int(rng.choice([0, 0, 1, 2, 5]))
    extra = int(rng.integers(0, 3))
    return kind, lengths, q_lens, Hkv * group, Hkv, d, page_size, causal, splits, extra


@pytest.mark.parametrize("i", range(48))
def test_fuzz_paged(i):
    kind, lengths, q_lens, Hq, Hkv, d, page_size, causal, splits, extra = paged_case(i)
    if kind == "decode":
        t = build_case(lengths, Hq, Hkv, d, page_size, True, 8000 + i, extra_pages=extra)
    else:
        t = build_case(lengths, Hq, Hkv, d, page_size, False, 8000 + i, q_lens=q_lens, extra_pages=extra)
    if int(t["q_lens"].sum()) == 0:
        pytest.skip("no query rows drawn")
    scale = 1 / math.sqrt(d)
    o, lse = run_paged(t, causal, scale, num_splits=splits)
    o_ref, lse_ref, va_ref = oracle_paged(t, causal, scale)
    compare(o, o_ref, lse, lse_ref,
            f"paged case {i}: {kind} lengths={lengths} q_lens={q_lens} Hq={Hq} Hkv={Hkv} d={d} "
            f"page={page_size} causal={causal} splits={splits}", vabs=va_ref)
