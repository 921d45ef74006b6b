"""The no-allocation decode entry point, called through the C ABI, against fa_paged_fwd.

fa_paged_decode_noalloc exists for callers that may not call cudaMalloc and so cannot hand
fa_paged_fwd a workspace; it keeps its split-KV partials in a fixed scratch array inside the
library instead. Two calls in a row (different batches, so stale scratch contents from the first
must not leak into the second) must each match the workspace entry point within the parity
tolerance. The file sorts last so that a failure here stops a -x run only after every other test.
"""
import ctypes

import numpy as np
import pytest

from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev
from tests.test_parity_paged import build_case

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, t, q, kp, vp, pt, cu, kl, out, lse, scale, splits):
    import torch

    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = kp.shape
    num_seqs, max_pages = pt.shape
    vpt = ctypes.c_void_p
    return lib.fa_paged_decode_noalloc(
        vpt(q.data_ptr()), vpt(kp.data_ptr()), vpt(vp.data_ptr()), vpt(pt.data_ptr()), vpt(cu.data_ptr()),
        vpt(kl.data_ptr()), num_seqs, total_q, page_size, max_pages, num_pages, Hq, Hkv, d, scale,
        vpt(out.data_ptr()), vpt(lse.data_ptr()), splits, vpt(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_entry_point():
    import torch

    import io_aware_exact_flash_gb300 as fa

    lib = fa.load_library()
    calls = [
        ([1000, 17, 4096, 3333, 250, 1, 64, 2048], 32, 8, 128, 4),    # explicit split count
        ([5, 0, 700, 12000, 16, 129, 9000], 16, 4, 128, 0),            # automatic, an empty sequence
    ]
    for n, (lengths, Hq, Hkv, d, splits) in enumerate(calls):
        t = build_case(lengths, Hq, Hkv, d, 16, True, 300 + n, extra_pages=2)
        q, kp, vp = to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"])
        pt, cu, kl = i32_dev(t["page_table"]), i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"])
        scale = 1.0 / np.sqrt(d)
        o_ref, l_ref = fa.fa_paged_fwd(q, kp, vp, pt, cu, kl, max_q_len=1, causal=True, scale=scale,
                                       num_splits=splits)
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        code = _noalloc_call(lib, t, q, kp, vp, pt, cu, kl, out, lse, scale, splits)
        assert code == 0, f"call {n}: {fa.status_string(code)}"
        torch.cuda.synchronize()
        compare(bf16_to_f64(out), bf16_to_f64(o_ref), lse.cpu().numpy(), l_ref.cpu().numpy(), f"no-alloc call {n}")
        assert fa.fa_get_device_status() == (0, 0)


def test_noalloc_rejects_split_counts_beyond_the_scratch():
    import torch

    import io_aware_exact_flash_gb300 as fa

    lib = fa.load_library()
    t = build_case([64] * 128, 32, 8, 128, 16, True, 400, poison=False)
    q, kp, vp = to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"])
    pt, cu, kl = i32_dev(t["page_table"]), i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"])
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda")
    # 64 splits x 128 sequences x 32 heads x 129 floats is far above the 16 MiB scratch
    code = _noalloc_call(lib, t, q, kp, vp, pt, cu, kl, out, lse, 0.1, 64)
    assert code == 4, fa.status_string(code)  # FA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((out == 0).all())
