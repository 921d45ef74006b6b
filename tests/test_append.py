"""Paged KV append on the GPU against the append oracle: whole page pools compared bit for bit
(data movement is exact), including pool slots that must stay untouched, plus an append followed
by decode over the grown cache."""
import math

import numpy as np
import pytest

import oracle
from oracle.kv_append import paged_append as oracle_append
from io_aware_exact_flash_gb300.workloads import normal_bf16
from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev

pytestmark = pytest.mark.gpu

NAN_BITS = np.uint16(0x7FC0)


def bits(t):
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_case(before, new, Hkv, d, page_size, seed, spare_pages=2):
    """A pool whose cached rows are random, every other slot NaN, with room for the new rows."""
    rng = np.random.default_rng(seed)
    total = [b + n for b, n in zip(before, new)]
    npages = [max(1, (L + page_size - 1) // page_size) for L in total]
    P = sum(npages) + spare_pages
    perm = rng.permutation(P).astype(np.int32)
    table = np.full((len(total), max(npages) + 1), -1, np.int32)
    off = 0
    for s, n in enumerate(npages):
        table[s, :n] = perm[off:off + n]
        off += n
    kp = np.full((P, page_size, Hkv, d), NAN_BITS, np.uint16)
    vp = kp.copy()
    ck = normal_bf16(seed, (P, page_size, Hkv, d), stream=1)
    cv = normal_bf16(seed, (P, page_size, Hkv, d), stream=2)
    for s, b in enumerate(before):
        for pos in range(b):
            pg, sl = table[s, pos // page_size], pos % page_size
            kp[pg, sl], vp[pg, sl] = ck[pg, sl], cv[pg, sl]
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    k_new = normal_bf16(seed, (int(cu[-1]), Hkv, d), stream=3)
    v_new = normal_bf16(seed, (int(cu[-1]), Hkv, d), stream=4)
    return dict(kp=kp, vp=vp, table=table, before=np.asarray(before, np.int32), cu=cu, k_new=k_new, v_new=v_new)


def run_append(c):
    import torch

    import io_aware_exact_flash_gb300 as fa

    kp, vp = to_dev(c["kp"]), to_dev(c["vp"])
    fa.fa_paged_append(to_dev(c["k_new"]), to_dev(c["v_new"]), i32_dev(c["cu"]), i32_dev(c["before"]),
                       i32_dev(c["table"]), kp, vp)
    torch.cuda.synchronize()
    return kp, vp


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("Hkv,d", [(8, 128), (1, 64), (2, 128), (3, 64)])
def test_append_matches_oracle(page_size, Hkv, d):
    import io_aware_exact_flash_gb300 as fa

    before = [0, 5, 16, 100, 0, 127, 300]
    new = [1, 12, 1, 60, 0, 129, 17]
    c = make_case(before, new, Hkv, d, page_size, seed=page_size + Hkv + d)
    kp, vp = run_append(c)
    assert fa.fa_get_device_status() == (0, 0)
    ek, ev = oracle_append(c["kp"], c["vp"], c["table"], c["before"], c["cu"], c["k_new"], c["v_new"])
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev)


def test_append_nothing_new_is_a_no_op():
    import io_aware_exact_flash_gb300 as fa

    c = make_case([3, 40], [0, 0], 2, 128, 16, seed=3)
    kp, vp = run_append(c)
    assert np.array_equal(bits(kp), c["kp"]) and np.array_equal(bits(vp), c["vp"])
    assert fa.fa_get_device_status() == (0, 0)


def test_append_unmapped_page_is_reported_and_skipped():
    """Sequence 1's table has no page for its new rows: those rows are skipped and the status
    word says so; the other sequences' rows still land where the oracle puts them."""
    import io_aware_exact_flash_gb300 as fa

    c = make_case([4, 16, 9], [5, 3, 20], 2, 64, 16, seed=8)
    c["table"][1, 1:] = -1  # positions 16..18 of sequence 1 have no page
    kp, vp = run_append(c)
    code, site = fa.fa_get_device_status()
    assert code == 8  # FA_ERR_DEVICE_BAD_PAGE
    keep = np.ones(len(c["k_new"]), bool)
    keep[c["cu"][1]:c["cu"][2]] = False
    cu = np.concatenate([[0], np.cumsum([5, 0, 20])]).astype(np.int32)
    ek, ev = oracle_append(c["kp"], c["vp"], c["table"], c["before"], cu, c["k_new"][keep], c["v_new"][keep])
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev)


def test_append_then_decode():
    """One serving step: append each sequence's newest token, then decode over the grown cache."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    Hq, Hkv, d, ps = 32, 8, 128, 16
    before = [0, 1, 15, 16, 200, 1023, 4095]
    c = make_case(before, [1] * len(before), Hkv, d, ps, seed=21)
    kp, vp = run_append(c)
    ek, ev = oracle_append(c["kp"], c["vp"], c["table"], c["before"], c["cu"], c["k_new"], c["v_new"])
    q = normal_bf16(22, (len(before), Hq, d))
    kv_lens = c["before"] + 1
    cu_q = np.arange(len(before) + 1, dtype=np.int32)
    o, lse = fa.fa_paged_fwd(to_dev(q), kp, vp, i32_dev(c["table"]), i32_dev(cu_q), i32_dev(kv_lens),
                             max_q_len=1, causal=True, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    o_ref, lse_ref, va_ref = oracle.get().paged(q, ek, ev, c["table"], cu_q, kv_lens, True, 1 / math.sqrt(d), vabs=True)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref, "append then decode", vabs=va_ref)


def test_append_full_size_prefill_batch():
    """All K/V rows of the 64-sequence paged batch (lengths 512..8192, Hkv=8, d=128, page 16)
    appended into an empty pool in one call, as the benchmark times it."""
    import torch

    import io_aware_exact_flash_gb300 as fa
    from io_aware_exact_flash_gb300.workloads import WORKLOADS, make_append

    w = WORKLOADS["paged_append_64seq_512_8192_hkv8_d128_p16"]
    t = make_append(w)
    empty = np.full((t["num_pages"], w.page_size, w.Hkv, w.d), NAN_BITS, np.uint16)
    kp, vp = to_dev(empty), to_dev(empty)
    fa.fa_paged_append(to_dev(t["k_new"]), to_dev(t["v_new"]), i32_dev(t["cu_seqlens_new"]),
                       i32_dev(t["kv_lens_before"]), i32_dev(t["page_table"]), kp, vp)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    ek, ev = oracle_append(empty, empty, t["page_table"], t["kv_lens_before"], t["cu_seqlens_new"], t["k_new"],
                           t["v_new"])
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev)
