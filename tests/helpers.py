"""Shared test helpers: moving seeded bf16 bit patterns to the GPU and comparing results with the
fp64 oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

# Tolerances on O (bf16 output of bf16 inputs with fp32 accumulation) and on LSE (fp32).
O_MAX_ABS = 1e-2
O_REL_FRO = 5e-3
LSE_MAX_ABS = 1e-3
# Unit roundoff of bf16 (8 significant bits, 7 of them stored): rounding a softmax weight to bf16
# moves it by at most this relative amount.
BF16_U = 2.0 ** -8


def bf16_floor(o_ref, vabs):
    """Per element of O, the error that bf16 softmax weights and a bf16 output can cause by
    themselves. The kernel multiplies V by the weights rounded to bf16, p_j (1 + d_j) with
    |d_j| <= u = 2^-8, and divides by the fp32 sum of the unrounded weights, so O_c moves by
    sum_j p_j d_j v_jc, at most u * sum_j p_j |v_jc| = u * vabs_c. Rounding the result to bf16 adds
    half an ulp of it, and fp32 arithmetic elsewhere (scores, exponentials, sums) far less than
    2^-12 relative. Where this floor exceeds the 1e-2 bound, it replaces that bound."""
    e_p = BF16_U * vabs
    mag = np.abs(o_ref) + e_p
    ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 2.0 ** -126))) - 7)
    return 0.5 * ulp + e_p + 2.0 ** -12 * (np.abs(o_ref) + vabs)


def to_dev(bits, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def i32_dev(a, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_to_f64(t):
    """bf16 CUDA tensor -> fp64 numpy array (exact)."""
    import torch

    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def compare(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what="", vabs=None):
    """Assert the GPU result matches the oracle; returns (max_abs, rel_fro, max_dlse).

    vabs: the oracle's sum_j p_j |v_jc| for each element of o_ref. With it, an element whose bf16
    floor (bf16_floor) exceeds the 1e-2 bound is held to that floor instead; max_abs is then
    reported over the other elements. Without it, only elements with |O| >= 4 (where half a bf16
    ulp alone exceeds 1e-2) are held to faithful rounding instead."""
    o_ref = np.asarray(o_ref, dtype=np.float64)
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, f"{what}: shape {o_gpu.shape} vs {o_ref.shape}"
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite values in O"
    diff = o_gpu - o_ref
    if vabs is not None:
        vabs = np.asarray(vabs, dtype=np.float64)
        assert vabs.shape == o_ref.shape, f"{what}: vabs shape {vabs.shape} vs {o_ref.shape}"
        floor = bf16_floor(o_ref, vabs)
        over_floor = floor > O_MAX_ABS
        if over_floor.any():
            bad = np.abs(diff[over_floor]) > floor[over_floor]
            assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the bf16 floor, worst "
                                   f"{float(np.abs(diff[over_floor])[bad].max())}")
            diff = np.where(over_floor, 0.0, diff)
    else:
        # A bf16 output cannot be closer to the exact value than half a bf16 ulp, which exceeds the
        # max-abs bound once |O| >= 4. Only there the bound becomes faithful rounding: the GPU value
        # must be one of the two bf16 numbers around the exact one (within one ulp of it).
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 2.0 ** -126))) - 7)
        over_floor = 0.5 * ulp > O_MAX_ABS
        if over_floor.any():
            assert np.all(np.abs(diff[over_floor]) <= ulp[over_floor]), f"{what}: not faithfully rounded where |O| >= 4"
            diff = np.where(over_floor, 0.0, diff)
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    full = o_gpu - o_ref
    denom = float(np.sqrt((o_ref ** 2).sum()))
    rel_fro = float(np.sqrt((full ** 2).sum()) / denom) if denom > 0 else float(np.sqrt((full ** 2).sum()))
    dl = 0.0
    if lse_gpu is not None:
        lg = np.asarray(lse_gpu, dtype=np.float64)
        lr = np.asarray(lse_ref, dtype=np.float64)
        both_ninf = np.isneginf(lg) & np.isneginf(lr)
        assert np.array_equal(np.isneginf(lg), np.isneginf(lr)), f"{what}: -inf LSE pattern differs"
        with np.errstate(invalid="ignore"):
            d = np.where(both_ninf, 0.0, np.abs(lg - lr))
        assert np.isfinite(d).all(), f"{what}: non-finite LSE"
        dl = float(d.max()) if d.size else 0.0
    assert max_abs <= O_MAX_ABS, f"{what}: max |dO| {max_abs} > {O_MAX_ABS}"
    assert rel_fro <= O_REL_FRO, f"{what}: rel Frobenius {rel_fro} > {O_REL_FRO}"
    assert dl <= LSE_MAX_ABS, f"{what}: max |dLSE| {dl} > {LSE_MAX_ABS}"
    return max_abs, rel_fro, dl
