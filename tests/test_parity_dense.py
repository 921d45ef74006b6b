"""Dense attention forward on the GPU against the fp64 oracle, element by element (small and
ragged shapes) and on sampled rows of the full-size long-context workloads."""
import math

import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import WORKLOADS, make_dense, normal_bf16
from tests.helpers import bf16_to_f64, compare, to_dev

pytestmark = pytest.mark.gpu


def run_fa(q, k, v, causal, scale):
    import torch

    import io_aware_exact_flash_gb300 as fa

    o, lse = fa.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


CASES = [
    # (B, S, Hq, Hkv, d, causal)
    (1, 256, 2, 2, 64, False),    # the small non-causal workload
    (1, 256, 2, 2, 64, True),
    (1, 128, 1, 1, 128, False),   # one query tile: the CTA's second tile is empty
    (1, 128, 1, 1, 128, True),
    (2, 384, 4, 4, 128, True),    # a CTA with two tiles and one with one
    (1, 1, 1, 1, 64, True),       # S = 1
    (1, 1, 1, 1, 128, False),
    (1, 200, 2, 1, 128, True),    # ragged tail, GQA 2
    (2, 517, 8, 2, 128, True),    # several tiles + ragged tail, GQA 4
    (1, 1000, 2, 2, 64, False),
    (1, 777, 4, 1, 64, True),
    (3, 640, 2, 2, 128, False),
    (1, 2048, 2, 2, 128, True),
    (2, 2048, 16, 16, 128, True),  # head chunks of the persistent schedule, the last one partial
    (1, 1024, 24, 8, 64, False),   # several rounds of the persistent schedule, GQA 3
    # more work items than SMs: CTAs that finish take over the items of CTAs not yet started
    (1, 512, 320, 64, 64, True),   # 320 mirrored-pair items, GQA 5
    (1, 300, 160, 32, 128, True),  # 160 items with a ragged tail
    (1, 256, 304, 304, 64, False), # 304 one-unit items
]


@pytest.mark.parametrize("B,S,Hq,Hkv,d,causal", CASES)
def test_dense_matches_oracle(B, S, Hq, Hkv, d, causal):
    seed = 7 + S + 31 * Hq + d
    q = normal_bf16(seed, (B, S, Hq, d), stream=0)
    k = normal_bf16(seed, (B, S, Hkv, d), stream=1)
    v = normal_bf16(seed, (B, S, Hkv, d), stream=2)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fa(q, k, v, causal, scale)
    o_ref, lse_ref, va_ref = oracle.get().dense(q, k, v, causal, scale, vabs=True)
    compare(o, o_ref, lse, lse_ref, f"dense {B, S, Hq, Hkv, d, causal}", vabs=va_ref)


@pytest.mark.parametrize("gain", [4.0, 16.0])
def test_dense_large_scores_force_rescales(gain):
    """Scores far beyond the deferred-rescale threshold, growing along the sequence, so the
    running maximum keeps rising and O is rescaled many times."""
    B, S, H, d = 1, 1024, 2, 128
    rng = np.random.default_rng(3)
    from io_aware_exact_flash_gb300.workloads import bf16_bits

    q = bf16_bits(rng.standard_normal((B, S, H, d)).astype(np.float32) * gain)
    ramp = np.linspace(0.2, 2.0, S, dtype=np.float32)[None, :, None, None]
    k = bf16_bits(rng.standard_normal((B, S, H, d)).astype(np.float32) * ramp * gain)
    v = bf16_bits(rng.standard_normal((B, S, H, d)).astype(np.float32))
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal, 1.0 / math.sqrt(d))
        o_ref, lse_ref, va_ref = oracle.get().dense(q, k, v, causal, 1.0 / math.sqrt(d), vabs=True)
        compare(o, o_ref, lse, lse_ref, f"large scores gain={gain} causal={causal}", vabs=va_ref)


def test_dense_outlier_keys_small():
    """The long-context recipe (activations x0.5, 1% of key rows x8) at a size the full oracle runs."""
    from io_aware_exact_flash_gb300.workloads import DenseWorkload

    w = DenseWorkload("outliers_small", B=1, S=1536, Hq=8, Hkv=2, d=128, causal=True, seed=55, act_scale=0.5,
                      outlier_frac=0.01, outlier_gain=8.0)
    t = make_dense(w)
    o, lse = run_fa(t["q"], t["k"], t["v"], True, w.scale)
    o_ref, lse_ref, va_ref = oracle.get().dense(t["q"], t["k"], t["v"], True, w.scale, vabs=True)
    compare(o, o_ref, lse, lse_ref, "outliers", vabs=va_ref)


def test_dense_deterministic():
    q, k, v = (normal_bf16(99, (2, 700, 4, 128), stream=s) for s in range(3))
    o1, l1 = run_fa(q, k, v, True, 0.09)
    o2, l2 = run_fa(q, k, v, True, 0.09)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_dense_reads_and_writes_stay_in_bounds():
    """Inputs sit between NaN guard regions and the output between sentinel regions: a read
    outside q/k/v would surface as NaN, a write outside o would change a sentinel."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    B, S, H, d = 2, 300, 2, 128
    n = B * S * H * d
    guard = 4096
    tensors = []
    for s in range(3):
        bits = normal_bf16(5, (n,), stream=s)
        buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
        buf[guard:guard + n] = to_dev(bits)
        tensors.append((bits.reshape(B, S, H, d), buf[guard:guard + n].view(B, S, H, d)))
    obuf = torch.full((n + 2 * guard,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = obuf[guard:guard + n].view(B, S, H, d)
    lbuf = torch.full((B * S * H + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
    lse = lbuf[guard:guard + B * S * H].view(B, S, H)
    fa.fa_fwd(tensors[0][1], tensors[1][1], tensors[2][1], causal=True, scale=0.1, out=out, lse=lse)
    torch.cuda.synchronize()
    assert bool((obuf[:guard] == 3.0).all()) and bool((obuf[guard + n:] == 3.0).all())
    assert bool((lbuf[:guard] == 7.0).all()) and bool((lbuf[guard + B * S * H:] == 7.0).all())
    o_ref, lse_ref, va_ref = oracle.get().dense(tensors[0][0], tensors[1][0], tensors[2][0], True, 0.1, vabs=True)
    compare(bf16_to_f64(out), o_ref, lse.cpu().numpy(), lse_ref, "guarded", vabs=va_ref)


def _sample_rows(B, S, H, rng, n_random):
    rows = []
    fixed = [0, 1, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 2, S - 1]
    for b in range(B):
        for i in fixed:
            rows.append((b, i, int(rng.integers(H))))
    for _ in range(n_random):
        rows.append((int(rng.integers(B)), int(rng.integers(S)), int(rng.integers(H))))
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("name,n_random", [
    ("causal_prefill_b4_h32_s4096_d128", 400),
    ("gqa_causal_prefill_b1_hq32_hkv8_s32768_d128", 150),
])
def test_full_size_sampled_rows(name, n_random):
    """The full-size workloads in the launch configuration the benchmark times, checked on
    sampled rows (tile edges, the first and last rows, and random rows) that the oracle computes
    one by one."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    w = WORKLOADS[name]
    t = make_dense(w)
    o, lse = fa.fa_fwd(to_dev(t["q"]), to_dev(t["k"]), to_dev(t["v"]), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rows = _sample_rows(w.B, w.S, w.Hq, np.random.default_rng(0), n_random)
    o_ref, lse_ref, va_ref = oracle.get().dense_rows(t["q"], t["k"], t["v"], w.causal, w.scale, rows, vabs=True)
    ridx = torch.from_numpy(rows).cuda()
    o_s = o[ridx[:, 0], ridx[:, 1], ridx[:, 2]]
    l_s = lse[ridx[:, 0], ridx[:, 1], ridx[:, 2]]
    compare(bf16_to_f64(o_s), o_ref, l_s.cpu().numpy(), lse_ref, name, vabs=va_ref)
    # properties that hold at any size: every row finite, LSE finite
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())


def test_dense_long_sequence_sampled():
    """B=1, S=131072, GQA 2 (causal): query rows and key positions far from zero on the dense
    path, checked on sampled rows (tile edges, the last rows, random rows)."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    B, S, Hq, Hkv, d = 1, 131072, 2, 1, 128
    q = normal_bf16(111, (B, S, Hq, d), stream=0)
    k = normal_bf16(111, (B, S, Hkv, d), stream=1)
    v = normal_bf16(111, (B, S, Hkv, d), stream=2)
    o, lse = fa.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    idx = np.concatenate([[0, 127, 128, 255, 256, S - 129, S - 128, S - 1], rng.integers(0, S, 24)])
    rows = np.stack([np.zeros_like(idx), idx, rng.integers(0, Hq, len(idx))], axis=1).astype(np.int64)
    o_ref, lse_ref, va_ref = oracle.get().dense_rows(q, k, v, True, 1 / math.sqrt(d), rows, vabs=True)
    ridx = torch.from_numpy(rows).cuda()
    compare(bf16_to_f64(o[ridx[:, 0], ridx[:, 1], ridx[:, 2]]), o_ref,
            lse[ridx[:, 0], ridx[:, 1], ridx[:, 2]].cpu().numpy(), lse_ref, "dense S=131072", vabs=va_ref)



@pytest.mark.parametrize("B,S,Hq,Hkv,causal", [
    (4, 4096, 32, 32, True),    # the causal prefill workload's shape: many more work items than SMs
    (4, 4096, 32, 32, False),
    (1, 32768, 32, 8, True),    # the long-context GQA workload's shape
])
def test_full_size_every_row_closed_form(B, S, Hq, Hkv, causal):
    """Every output row of a full-size launch, against a closed form. All keys of a (batch, kv
    head) are one row k and all its values one constant c, so every allowed score of row i is
    equal: O = c exactly and LSE = scale * q_i . k + ln(n_i), n_i the number of allowed keys.
    O and LSE start as NaN, so a work item that no CTA ran, or a row written with another head's
    data, fails here whichever rows a sampled check would have picked."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    d = 128
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d)
    q = normal_bf16(321, (B, S, Hq, d), stream=0)
    krow = normal_bf16(321, (B, 1, Hkv, d), stream=1)
    k = np.ascontiguousarray(np.broadcast_to(krow, (B, S, Hkv, d)))
    c = (1 + np.arange(B * Hkv) % 64).reshape(B, Hkv) / 16.0   # exact in bf16
    c_bits = c.astype(np.float32).view(np.uint32) >> np.uint32(16)
    v = np.ascontiguousarray(np.broadcast_to(c_bits.astype(np.uint16)[:, None, :, None], (B, S, Hkv, d)))
    out = torch.full((B, S, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    c_dev = torch.from_numpy(np.repeat(c, G, axis=1)).cuda()  # (B, Hq)
    o_err = (out.double() - c_dev[:, None, :, None]).abs().amax().item()
    assert o_err <= 1e-2, f"max |O - c| = {o_err}"
    qf = (q.astype(np.uint32) << np.uint32(16)).view(np.float32)
    kf = (krow.astype(np.uint32) << np.uint32(16)).view(np.float32)[:, 0]  # (B, Hkv, d)
    n = np.arange(1, S + 1, dtype=np.float64) if causal else np.full(S, float(S))
    lse_gpu = lse.cpu().numpy().astype(np.float64)
    worst = 0.0
    for b in range(B):
        for h in range(Hq):
            s = qf[b, :, h, :].astype(np.float64) @ kf[b, h // G].astype(np.float64)
            worst = max(worst, float(np.abs(lse_gpu[b, :, h] - (scale * s + np.log(n))).max()))
    assert worst <= 1e-3, f"max |dLSE| = {worst}"
