"""Calls captured into a CUDA graph from the caller's stream and replayed: the cascade (whose suffix
pass forks onto the library's side stream and joins back) and a paged decode batch on the key-row
kernel (planning, attention and the key-split merge). Replays must reproduce the direct calls bit
for bit (the kernels are deterministic) and leave the device status word clear; the direct call
is checked against the oracle too."""
import math

import numpy as np
import pytest

from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev
from tests.test_cascade import build, oracle_flat
from tests.test_parity_paged import build_case, oracle_paged

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch

    return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _capture_and_replay(call, outs):
    """Runs call() once directly (warm-up and reference), captures it into a graph, clears the
    outputs, replays twice and returns (direct results, replayed results)."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    call()
    torch.cuda.synchronize()
    direct = [_bits(t).copy() for t in outs]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for t in outs:
        t.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    return direct, [_bits(t) for t in outs]


def test_cascade_in_a_cuda_graph():
    import torch

    import io_aware_exact_flash_gb300 as fa

    c = build([40, 24, 64], [3000, 500, 1200], [1] * 128, list(np.random.default_rng(5).integers(1, 900, 128)),
              32, 8, 128, 16, seed=77)
    scale = 1 / math.sqrt(128)
    q, kp, vp = to_dev(c["q"]), to_dev(c["kp"]), to_dev(c["vp"])
    idx = [i32_dev(c[k]) for k in ("cu_groups", "pre_table", "prefix_lens", "cu", "table", "kv_lens")]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    need = fa.fa_cascade_workspace_bytes(len(c["groups"]), len(c["q_lens"]), q.shape[0], c["max_group_q"], 1,
                                         16, c["pre_table"].shape[1], c["table"].shape[1], c["kp"].shape[0], 32, 8,
                                         128)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)

    def call():
        fa.fa_cascade_fwd(q, kp, vp, idx[0], idx[1], idx[2], c["max_group_q"], idx[3], idx[4], idx[5], 1,
                          causal=True, scale=scale, out=o, lse=lse, workspace=ws,
                          stream=torch.cuda.current_stream())

    direct, replayed = _capture_and_replay(call, [o, lse])
    for a, b in zip(direct, replayed):
        assert np.array_equal(a, b), "a replayed cascade differs from the direct call"
    o_ref, lse_ref, va_ref = oracle_flat(c, True, scale)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref, "cascade graph", vabs=va_ref)


def test_key_row_decode_with_splits_in_a_cuda_graph():
    import torch

    import io_aware_exact_flash_gb300 as fa

    t = build_case([1, 15, 16, 130, 300, 1000, 5000, 2049], 32, 8, 128, 16, True, 78, extra_pages=2)
    scale = 1 / math.sqrt(128)
    q, kp, vp = to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"])
    pt, cu, kl = i32_dev(t["page_table"]), i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"])
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    need = fa.fa_paged_workspace_bytes(len(t["kv_lens"]), q.shape[0], 1, 16, t["page_table"].shape[1],
                                       t["num_pages"], 32, 8, 128, num_splits=3)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)

    def call():
        fa.fa_paged_fwd(q, kp, vp, pt, cu, kl, 1, causal=True, scale=scale, out=o, lse=lse, workspace=ws,
                        num_splits=3, stream=torch.cuda.current_stream())

    direct, replayed = _capture_and_replay(call, [o, lse])
    for a, b in zip(direct, replayed):
        assert np.array_equal(a, b), "a replayed decode differs from the direct call"
    o_ref, lse_ref, va_ref = oracle_paged(t, True, scale)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref, "decode graph", vabs=va_ref)
