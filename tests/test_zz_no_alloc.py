"""The no-allocation decode entry point, called through the C ABI, against the fp64 oracle and
against fa_paged_fwd.

fa_paged_decode_noalloc exists for callers that may not call cudaMalloc and so cannot hand
fa_paged_fwd a workspace; it keeps its split-KV partials in a fixed scratch array inside the
library instead. Two calls in a row (different batches, so stale scratch contents from the first
must not leak into the second) must each match the oracle within the parity tolerance, and the
workspace entry point's output as a second check. A batch whose automatic split count would not
fit the scratch must run with a lowered count and still match the oracle. The file sorts last so
that a failure here stops a -x run only after every other test.
"""
import ctypes

import numpy as np
import pytest

from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev
from tests.test_parity_paged import build_case, oracle_paged

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


def _noalloc_call(lib, q, kp, vp, pt, cu, kl, out, lse, scale, splits):
    import torch

    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = kp.shape
    num_seqs, max_pages = pt.shape
    vpt = ctypes.c_void_p
    return lib.fa_paged_decode_noalloc(
        vpt(q.data_ptr()), vpt(kp.data_ptr()), vpt(vp.data_ptr()), vpt(pt.data_ptr()), vpt(cu.data_ptr()),
        vpt(kl.data_ptr()), num_seqs, total_q, page_size, max_pages, num_pages, Hq, Hkv, d, scale,
        vpt(out.data_ptr()), vpt(lse.data_ptr()), splits, vpt(torch.cuda.current_stream().cuda_stream))


def _scratch_bytes(splits, num_seqs, Hq, Hkv, d):
    """The scratch a split count needs, as include/fa.h states it: partial O and LSE floats and one
    counter per sequence and block of up to 8 kv heads, each part rounded up to 256 bytes."""
    if splits <= 1:
        return 0
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    hpc = next(h for h in range(min(8, Hkv), 0, -1) if Hkv % h == 0)
    return (a(splits * num_seqs * Hq * d * 4) + a(splits * num_seqs * Hq * 4) + a(num_seqs * (Hkv // hpc) * 4))


def _run_and_check(lib, fa, t, splits, what):
    import torch

    q, kp, vp = to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"])
    pt, cu, kl = i32_dev(t["page_table"]), i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"])
    d = q.shape[2]
    scale = 1.0 / np.sqrt(d)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    code = _noalloc_call(lib, q, kp, vp, pt, cu, kl, out, lse, scale, splits)
    assert code == 0, f"{what}: {fa.status_string(code)}"
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    o_gpu, l_gpu = bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)
    o_ref, l_ref, va_ref = oracle_paged(t, True, scale)
    compare(o_gpu, o_ref, l_gpu, l_ref, f"{what} vs oracle", vabs=va_ref)
    o_ws, l_ws = fa.fa_paged_fwd(q, kp, vp, pt, cu, kl, max_q_len=1, causal=True, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    compare(o_gpu, bf16_to_f64(o_ws), l_gpu, l_ws.cpu().numpy().astype(np.float64), f"{what} vs fa_paged_fwd", vabs=va_ref)


def test_noalloc_decode_two_calls_in_a_row():
    import io_aware_exact_flash_gb300 as fa

    lib = fa.load_library()
    calls = [
        ([1000, 17, 4096, 3333, 250, 1, 64, 2048], 32, 8, 128, 4),    # explicit split count
        ([5, 0, 700, 12000, 16, 129, 9000], 16, 4, 128, 0),            # automatic, an empty sequence
    ]
    for n, (lengths, Hq, Hkv, d, splits) in enumerate(calls):
        t = build_case(lengths, Hq, Hkv, d, 16, True, 300 + n, extra_pages=2)
        _run_and_check(lib, fa, t, splits, f"no-alloc call {n}")


def test_noalloc_lowers_an_automatic_split_count_that_does_not_fit():
    """128 decode sequences of 200 to 300 keys with 32 query heads: the automatic split count of
    the decode kernel needs more partials than the scratch holds (one split is 2 MiB here), so the
    call lowers it to the largest count that fits and must still match the oracle."""
    import io_aware_exact_flash_gb300 as fa

    lib = fa.load_library()
    rng = np.random.default_rng(310)
    lengths = rng.integers(200, 301, size=128).tolist()
    Hq, Hkv, d, ps = 32, 8, 128, 16
    t = build_case(lengths, Hq, Hkv, d, ps, True, 311, extra_pages=1)
    num_seqs, max_pages = t["page_table"].shape
    auto = fa.fa_decode_num_splits(num_seqs, ps, max_pages, t["num_pages"], Hkv)
    assert _scratch_bytes(auto, num_seqs, Hq, Hkv, d) > SCRATCH_BYTES, f"automatic count {auto} fits the scratch"
    chosen = auto
    while chosen > 1 and _scratch_bytes(chosen, num_seqs, Hq, Hkv, d) > SCRATCH_BYTES:
        chosen -= 1
    assert chosen > 1 and _scratch_bytes(chosen, num_seqs, Hq, Hkv, d) <= SCRATCH_BYTES
    _run_and_check(lib, fa, t, 0, f"no-alloc, automatic {auto} splits lowered to {chosen}")


def test_noalloc_caps_then_rejects_explicit_split_counts():
    """An explicit split count is first capped at the pages of the longest sequence: 64 splits of
    4-page sequences run as 4 splits, which fit the scratch, and match the oracle. 64 splits of
    64-page sequences (64 x 128 sequences x 32 heads x 129 floats) do not fit: the call returns
    FA_ERR_WORKSPACE and enqueues nothing."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    lib = fa.load_library()
    assert _scratch_bytes(4, 128, 32, 8, 128) <= SCRATCH_BYTES < _scratch_bytes(64, 128, 32, 8, 128)
    t = build_case([64] * 128, 32, 8, 128, 16, True, 400)
    _run_and_check(lib, fa, t, 64, "no-alloc, 64 splits capped at 4 pages")
    t = build_case([1024] * 128, 32, 8, 128, 16, True, 401, poison=False)
    q, kp, vp = to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"])
    pt, cu, kl = i32_dev(t["page_table"]), i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"])
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda")
    code = _noalloc_call(lib, q, kp, vp, pt, cu, kl, out, lse, 0.1, 64)
    assert code == 4, fa.status_string(code)  # FA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((out == 0).all())
