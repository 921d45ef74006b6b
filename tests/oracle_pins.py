"""Pins for the fp64 oracle: facts that the definition of exact attention fixes independently of
the oracle's own code (closed forms, invariants, a library routine, high-precision brute force).

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the oracle disagrees.
``test_oracle_pins.py`` runs them against the real oracle; ``test_oracle_mutants.py`` runs them
against copies of the oracle with a planted mistake and requires each mistake to be caught.

The method and its exactness claim come from "I/O-Aware Kernels" (datasystem.school, Module 5),
sections "Naive attention: materializing the k x k score matrix" and "FlashAttention: tiling +
online softmax"; grouped-query heads and the paged layout from its section "FlashInfer: I/O-aware
attention for serving".
"""
from __future__ import annotations

import math

import numpy as np

from io_aware_exact_flash_gb300.workloads import bf16_bits, bits_to_f32


def _bf(x):
    return bf16_bits(np.asarray(x, dtype=np.float32))


def _f64(bits):
    return bits_to_f32(bits).astype(np.float64)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    assert not np.isnan(err).any(), f"{what}: NaN where a finite value or a matching infinity was expected"
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max error {worst} > {tol}"


# ------------------------------------------------------------------------- closed forms


def pin_identical_keys(orc):
    """All keys equal: every allowed score is the same, so O_i is the mean of the allowed V rows
    and LSE_i = s_i + ln(n_i). Exercised with GQA heads and both mask modes."""
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, d = 2, 37, 4, 2, 16
    scale = 1.0 / math.sqrt(d)
    q = _bf(rng.standard_normal((B, S, Hq, d)))
    k0 = _bf(rng.standard_normal((B, 1, Hkv, d)))
    k = np.ascontiguousarray(np.broadcast_to(k0, (B, S, Hkv, d)))
    v = _bf(rng.standard_normal((B, S, Hkv, d)))
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for causal in (False, True):
        o, lse = orc.dense(q, k, v, causal, scale, threads=2)
        for b in range(B):
            for i in range(S):
                for h in range(Hq):
                    hk = h // (Hq // Hkv)
                    n = i + 1 if causal else S
                    _close(o[b, i, h], vf[b, :n, hk].mean(axis=0), 1e-13, "identical keys O")
                    s = scale * float(qf[b, i, h] @ kf[b, 0, hk])
                    _close(lse[b, i, h], s + math.log(n), 1e-12, "identical keys LSE")


def pin_dominant_key(orc):
    """Each query row has exactly one key whose score exceeds every other by >= 60, so O_i is
    that key's V row (to 1e-12) and LSE_i is that score (to 1e-12)."""
    rng = np.random.default_rng(12)
    S, d, Hq, Hkv = 16, 16, 2, 1
    scale = 0.25
    for causal in (False, True):
        key_axis = rng.permutation(d) if not causal else np.arange(d)
        k = np.zeros((1, S, Hkv, d), np.float32)
        for j in range(S):
            k[0, j, 0, key_axis[j]] = 32.0
        q = np.zeros((1, S, Hq, d), np.float32)
        target = np.zeros((S, Hq), np.int64)
        for i in range(S):
            for h in range(Hq):
                j = ((i * 5 + 3 * h) % (i + 1)) if causal else int((i + 7 * h) % S)
                target[i, h] = j
                q[0, i, h, key_axis[j]] = 32.0
        v = _bf(rng.standard_normal((1, S, Hkv, d)))
        o, lse = orc.dense(_bf(q), _bf(k), v, causal, scale, threads=1)
        vf = _f64(v)
        for i in range(S):
            for h in range(Hq):
                _close(o[0, i, h], vf[0, target[i, h], 0], 1e-12, "dominant key O")
                _close(lse[0, i, h], 32.0 * 32.0 * scale, 1e-12, "dominant key LSE")


def pin_large_scores_stay_exact(orc):
    """Scores in the thousands: one key per row scores 4096 while the rest score 0 or less, so
    exp() of an unshifted score would overflow. The softmax is invariant to subtracting the row
    maximum; the result must still be that key's V row and LSE must be 4096."""
    rng = np.random.default_rng(26)
    S, d = 12, 16
    k = np.zeros((1, S, 1, d), np.float32)
    q = np.zeros((1, S, 1, d), np.float32)
    for j in range(S):
        k[0, j, 0, j] = 128.0
    target = [(3 * i + 1) % S for i in range(S)]
    for i in range(S):
        q[0, i, 0, target[i]] = 128.0
        q[0, i, 0, (target[i] + 1) % S] = -64.0
    v = _bf(rng.standard_normal((1, S, 1, d)))
    o, lse = orc.dense(_bf(q), _bf(k), v, False, 0.25, threads=1)
    vf = _f64(v)
    for i in range(S):
        _close(o[0, i, 0], vf[0, target[i], 0], 0.0, "large scores O")
        _close(lse[0, i, 0], 4096.0, 1e-12, "large scores LSE")


def pin_causal_first_row(orc):
    """Causal row 0 sees only key 0: O = V[0] exactly and LSE = scale * q_0 . k_0."""
    rng = np.random.default_rng(13)
    B, S, Hq, Hkv, d = 3, 9, 4, 4, 8
    scale = 0.3
    q, k, v = (_bf(rng.standard_normal((B, S, H, d))) for H in (Hq, Hkv, Hkv))
    o, lse = orc.dense(q, k, v, True, scale, threads=1)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for b in range(B):
        for h in range(Hq):
            _close(o[b, 0, h], vf[b, 0, h], 0.0, "causal row 0 O")
            _close(lse[b, 0, h], scale * float(qf[b, 0, h] @ kf[b, 0, h]), 1e-13, "causal row 0 LSE")


def pin_rows_of_p_sum_to_one(orc):
    """With every V entry equal to c, O = c * sum_j P_ij = c exactly up to rounding."""
    rng = np.random.default_rng(14)
    B, S, H, d = 1, 50, 2, 8
    q = _bf(rng.standard_normal((B, S, H, d)) * 3)
    k = _bf(rng.standard_normal((B, S, H, d)) * 3)
    v = _bf(np.full((B, S, H, d), 1.5))
    for causal in (False, True):
        o, _ = orc.dense(q, k, v, causal, 0.5, threads=1)
        _close(o, np.full(o.shape, 1.5), 1e-13, "P row sum")


def pin_scale_zero(orc):
    """scale = 0 makes every score 0: O_i = mean of the allowed V rows, LSE_i = ln(n_i)."""
    rng = np.random.default_rng(15)
    B, S, H, d = 1, 21, 1, 4
    q, k, v = (_bf(rng.standard_normal((B, S, H, d))) for _ in range(3))
    vf = _f64(v)
    for causal in (False, True):
        o, lse = orc.dense(q, k, v, causal, 0.0, threads=1)
        for i in range(S):
            n = i + 1 if causal else S
            _close(o[0, i, 0], vf[0, :n, 0].mean(axis=0), 1e-14, "scale 0 O")
            _close(lse[0, i, 0], math.log(n), 1e-14, "scale 0 LSE")


# ------------------------------------------------------------------------- invariants


def pin_linear_in_v(orc):
    """O is linear in V: O(V1 + V2) = O(V1) + O(V2) (small integers keep V1 + V2 exact in bf16)."""
    rng = np.random.default_rng(16)
    B, S, H, d = 1, 33, 2, 8
    q = _bf(rng.standard_normal((B, S, H, d)))
    k = _bf(rng.standard_normal((B, S, H, d)))
    v1 = rng.integers(-8, 9, (B, S, H, d)).astype(np.float32)
    v2 = rng.integers(-8, 9, (B, S, H, d)).astype(np.float32)
    for causal in (False, True):
        o1, l1 = orc.dense(q, k, _bf(v1), causal, 0.4, threads=1)
        o2, l2 = orc.dense(q, k, _bf(v2), causal, 0.4, threads=1)
        o12, l12 = orc.dense(q, k, _bf(v1 + v2), causal, 0.4, threads=1)
        _close(o12, o1 + o2, 1e-12, "linearity O")
        _close(l12, l1, 0.0, "LSE independent of V")


def pin_shift_invariance(orc):
    """Adding the same vector u to every key adds scale * q_i . u to every score of row i: O is
    unchanged and LSE_i moves by exactly that amount."""
    rng = np.random.default_rng(17)
    B, S, H, d = 1, 24, 2, 8
    scale = 0.125
    q = rng.integers(-3, 4, (B, S, H, d)).astype(np.float32)
    k = rng.integers(-3, 4, (B, S, H, d)).astype(np.float32)
    u = rng.integers(-3, 4, (1, 1, H, d)).astype(np.float32)
    v = _bf(rng.standard_normal((B, S, H, d)))
    for causal in (False, True):
        o0, l0 = orc.dense(_bf(q), _bf(k), v, causal, scale, threads=1)
        o1, l1 = orc.dense(_bf(q), _bf(k + u), v, causal, scale, threads=1)
        _close(o1, o0, 1e-12, "shift O")
        shift = scale * np.einsum("bshd,hd->bsh", q.astype(np.float64), u[0, 0].astype(np.float64))
        _close(l1, l0 + shift, 1e-11, "shift LSE")


def pin_permutation_equivariance(orc):
    """Non-causal: permuting keys and values together leaves O and LSE unchanged; permuting query
    rows permutes the outputs the same way."""
    rng = np.random.default_rng(18)
    B, S, H, d = 2, 29, 2, 8
    q, k, v = (_bf(rng.standard_normal((B, S, H, d))) for _ in range(3))
    o, lse = orc.dense(q, k, v, False, 0.35, threads=2)
    pk = rng.permutation(S)
    o2, l2 = orc.dense(q, k[:, pk], v[:, pk], False, 0.35, threads=2)
    _close(o2, o, 1e-13, "key permutation O")
    _close(l2, lse, 1e-13, "key permutation LSE")
    pq = rng.permutation(S)
    o3, l3 = orc.dense(q[:, pq], k, v, False, 0.35, threads=2)
    _close(o3, o[:, pq], 0.0, "query permutation O")
    _close(l3, lse[:, pq], 0.0, "query permutation LSE")


def pin_gqa_equals_repeated_mha(orc):
    """Grouped-query heads (contiguous groups) equal multi-head attention with each K/V head
    repeated Hq/Hkv times in place."""
    rng = np.random.default_rng(19)
    B, S, Hq, Hkv, d = 2, 19, 8, 2, 8
    q = _bf(rng.standard_normal((B, S, Hq, d)))
    k = _bf(rng.standard_normal((B, S, Hkv, d)))
    v = _bf(rng.standard_normal((B, S, Hkv, d)))
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    for causal in (False, True):
        o, lse = orc.dense(q, k, v, causal, 0.3, threads=2)
        o2, l2 = orc.dense(q, kr, vr, causal, 0.3, threads=2)
        _close(o, o2, 0.0, "GQA vs repeated MHA O")
        _close(lse, l2, 0.0, "GQA vs repeated MHA LSE")


# ------------------------------------------------------------------------- special cases


def pin_bottom_right_causal(orc):
    """With q_len < kv_len, causal row i attends to the first i + (kv_len - q_len) + 1 keys; a
    single query row (decode) attends to all keys, as without a mask."""
    rng = np.random.default_rng(20)
    Sq, Skv, H, d = 3, 10, 2, 8
    q = _bf(rng.standard_normal((1, Sq, H, d)))
    k = np.ascontiguousarray(np.broadcast_to(_bf(rng.standard_normal((1, 1, H, d))), (1, Skv, H, d)))
    v = _bf(rng.standard_normal((1, Skv, H, d)))
    o, lse = orc.dense(q, k, v, True, 0.5, threads=1)
    vf = _f64(v)
    for i in range(Sq):
        n = i + (Skv - Sq) + 1
        for h in range(H):
            _close(o[0, i, h], vf[0, :n, h].mean(axis=0), 1e-13, "bottom-right O")
    q1 = q[:, :1]
    k2 = _bf(rng.standard_normal((1, Skv, H, d)))
    oc, lc = orc.dense(q1, k2, v, True, 0.5, threads=1)
    on, ln = orc.dense(q1, k2, v, False, 0.5, threads=1)
    _close(oc, on, 0.0, "decode causal == non-causal O")
    _close(lc, ln, 0.0, "decode causal == non-causal LSE")


def pin_rows_without_keys(orc):
    """Causal with q_len > kv_len: the top q_len - kv_len rows see no key (O = 0, LSE = -inf);
    an empty key set (kv_len = 0) does the same for every row."""
    rng = np.random.default_rng(21)
    Sq, Skv, H, d = 5, 2, 1, 4
    q = _bf(rng.standard_normal((1, Sq, H, d)))
    k, v = (_bf(rng.standard_normal((1, Skv, H, d))) for _ in range(2))
    o, lse = orc.dense(q, k, v, True, 1.0, threads=1)
    vf = _f64(v)
    for i in range(3):
        _close(o[0, i, 0], np.zeros(d), 0.0, "empty row O")
        assert lse[0, i, 0] == -math.inf, "empty row LSE"
    _close(o[0, 3, 0], vf[0, 0, 0], 0.0, "one key O")
    o0, l0 = orc.dense(q, k[:, :0], v[:, :0], False, 1.0, threads=1)
    _close(o0, np.zeros_like(o0), 0.0, "kv_len 0 O")
    assert np.all(l0 == -math.inf), "kv_len 0 LSE"


def pin_sdpa_fp64(orc):
    """A library routine: torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU
    (run, not read) agrees to 1e-12, without and with the causal mask (equal lengths), with GQA
    expanded by repetition, and for a shorter query block with a bottom-right boolean mask."""
    import torch

    rng = np.random.default_rng(22)
    cases = [(2, 40, 40, 4, 4, 16, False), (2, 40, 40, 4, 4, 16, True), (1, 33, 33, 8, 2, 32, True),
             (1, 7, 31, 2, 1, 8, True), (1, 65, 65, 2, 2, 64, False)]
    for B, Sq, Skv, Hq, Hkv, d, causal in cases:
        scale = 1.0 / math.sqrt(d)
        q = _bf(rng.standard_normal((B, Sq, Hq, d)))
        k = _bf(rng.standard_normal((B, Skv, Hkv, d)))
        v = _bf(rng.standard_normal((B, Skv, Hkv, d)))
        o, lse = orc.dense(q, k, v, causal, scale, threads=2)
        tq = torch.from_numpy(_f64(q)).permute(0, 2, 1, 3)
        tk = torch.from_numpy(np.repeat(_f64(k), Hq // Hkv, axis=2)).permute(0, 2, 1, 3)
        tv = torch.from_numpy(np.repeat(_f64(v), Hq // Hkv, axis=2)).permute(0, 2, 1, 3)
        mask = None
        if causal:
            mask = torch.ones(Sq, Skv, dtype=torch.bool).tril(diagonal=Skv - Sq)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
        _close(o, ref.permute(0, 2, 1, 3).numpy(), 1e-12, f"SDPA O {B, Sq, Skv, Hq, Hkv, d, causal}")
        scores = torch.matmul(tq, tk.transpose(-1, -2)) * scale
        if mask is not None:
            scores = scores.masked_fill(~mask, -math.inf)
        ref_lse = torch.logsumexp(scores, dim=-1).permute(0, 2, 1).numpy()
        _close(lse, ref_lse, 1e-12, "logsumexp LSE")


def pin_bruteforce_high_precision(orc):
    """Tiny inputs: the softmax written directly as exp(s_j) / sum_k exp(s_k) without the max
    shift, in 50-digit arithmetic (mpmath), with exact rational dot products."""
    from fractions import Fraction

    import mpmath

    mpmath.mp.dps = 50
    rng = np.random.default_rng(23)
    for S, d, causal in [(1, 1, False), (3, 2, False), (5, 4, True), (6, 3, False), (6, 4, True)]:
        q = _bf(rng.standard_normal((1, S, 1, d)) * 2)
        k = _bf(rng.standard_normal((1, S, 1, d)) * 2)
        v = _bf(rng.standard_normal((1, S, 1, d)))
        scale = 0.7
        o, lse = orc.dense(q, k, v, causal, scale, threads=1)
        qf, kf, vf = _f64(q), _f64(k), _f64(v)
        for i in range(S):
            n = i + 1 if causal else S
            e = []
            for j in range(n):
                dot = sum(Fraction(float(qf[0, i, 0, c])) * Fraction(float(kf[0, j, 0, c])) for c in range(d))
                e.append(mpmath.exp(mpmath.mpf(scale) * mpmath.mpf(dot.numerator) / dot.denominator))
            tot = mpmath.fsum(e)
            for c in range(d):
                want = mpmath.fsum(e[j] * mpmath.mpf(float(vf[0, j, 0, c])) for j in range(n)) / tot
                _close(o[0, i, 0, c], float(want), 1e-14, "brute-force O")
            _close(lse[0, i, 0], float(mpmath.log(tot)), 1e-14, "brute-force LSE")


# ------------------------------------------------------------------------- paged layout


def _small_paged(seed, lengths, Hq, Hkv, d, page_size, decode):
    rng = np.random.default_rng(seed)
    kv_lens = np.asarray(lengths, np.int32)
    q_lens = np.ones_like(kv_lens) if decode else kv_lens.copy()
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    npages = (kv_lens + page_size - 1) // page_size
    P = int(npages.sum())
    perm = rng.permutation(P).astype(np.int32)
    table = np.full((len(kv_lens), int(npages.max())), -1, np.int32)
    off = 0
    for s, n in enumerate(npages):
        table[s, :n] = perm[off:off + n]
        off += n
    q = _bf(rng.standard_normal((int(cu[-1]), Hq, d)))
    kp = _bf(rng.standard_normal((P, page_size, Hkv, d)))
    vp = _bf(rng.standard_normal((P, page_size, Hkv, d)))
    return q, kp, vp, table, cu, kv_lens


def pin_paged_equals_dense(orc):
    """The paged layout read through its page table equals the dense layout of the same keys and
    values (gathered here with numpy indexing), sequence by sequence, bit for bit."""
    for decode in (False, True):
        lengths = [1, 16, 17, 40, 5]
        Hq, Hkv, d, ps = 4, 2, 8, 16
        q, kp, vp, table, cu, kv_lens = _small_paged(24, lengths, Hq, Hkv, d, ps, decode)
        o, lse = orc.paged(q, kp, vp, table, cu, kv_lens, True, 0.3, threads=2)
        for s, L in enumerate(lengths):
            pos = np.arange(L)
            phys = table[s, pos // ps]
            kd = kp[phys, pos % ps][None]
            vd = vp[phys, pos % ps][None]
            qd = q[cu[s]:cu[s + 1]][None]
            od, ld = orc.dense(qd, kd, vd, True, 0.3, threads=1)
            _close(o[cu[s]:cu[s + 1]], od[0], 0.0, "paged vs dense O")
            _close(lse[cu[s]:cu[s + 1]], ld[0], 0.0, "paged vs dense LSE")


def pin_paged_rows_subset(orc):
    """Selected rows equal the same rows of the full computation (rows are independent)."""
    q, kp, vp, table, cu, kv_lens = _small_paged(25, [33, 7, 64], 4, 1, 8, 16, False)
    o, lse = orc.paged(q, kp, vp, table, cu, kv_lens, True, 0.3, threads=1)
    rows = np.array([[0, 0], [40, 3], [103, 2], [35, 1]], np.int64)
    o2, l2 = orc.paged_rows(q, kp, vp, table, cu, kv_lens, True, 0.3, rows, threads=2)
    _close(o2, o[rows[:, 0], rows[:, 1]], 0.0, "row subset O")
    _close(l2, lse[rows[:, 0], rows[:, 1]], 0.0, "row subset LSE")


def pin_vabs_closed_forms(orc):
    """The softmax-weighted mean magnitude of V, sum_j p_j |v_jc|, in cases where the weights are
    known in closed form. Identical keys: uniform weights over the n allowed keys, so it is the
    mean of |v_jc| over those rows. Two keys whose scores differ by g: weights w = 1 / (1 + e^-g)
    and 1 - w, so it is w |v_0c| + (1 - w) |v_1c|. Constant V = c: |c|. Dense and paged layouts;
    a row with no key gives zero."""
    rng = np.random.default_rng(31)
    B, S, Hq, Hkv, d = 1, 12, 2, 1, 8
    q = _bf(rng.standard_normal((B, S, Hq, d)))
    k0 = _bf(rng.standard_normal((B, 1, Hkv, d)))
    k = np.ascontiguousarray(np.broadcast_to(k0, (B, S, Hkv, d)))
    v = _bf(rng.standard_normal((B, S, Hkv, d)) * 2.0)
    vf = _f64(v)
    _, _, va = orc.dense(q, k, v, True, 0.3, threads=2, vabs=True)
    for i in range(S):
        for h in range(Hq):
            _close(va[0, i, h], np.abs(vf[0, :i + 1, 0]).mean(axis=0), 1e-13, "weighted |V| of identical keys")
    # two keys with a known score gap: q = 2 e_0, k_0 = 1.5 e_0, k_1 = -0.25 e_0
    d2 = 4
    qq = np.zeros((1, 1, 1, d2), np.float32)
    qq[0, 0, 0, 0] = 2.0
    kk = np.zeros((1, 2, 1, d2), np.float32)
    kk[0, 0, 0, 0], kk[0, 1, 0, 0] = 1.5, -0.25
    vv = _bf(rng.standard_normal((1, 2, 1, d2)))
    scale = 0.75
    g = scale * 2.0 * (1.5 - (-0.25))
    w = 1.0 / (1.0 + math.exp(-g))
    vvf = _f64(vv)
    _, _, va2 = orc.dense(_bf(qq), _bf(kk), vv, False, scale, threads=1, vabs=True)
    _close(va2[0, 0, 0], w * np.abs(vvf[0, 0, 0]) + (1 - w) * np.abs(vvf[0, 1, 0]), 1e-13, "weighted |V| of two keys")
    # constant V rows (negative, so the magnitude is taken)
    vc = np.ascontiguousarray(np.broadcast_to(_bf(np.full((1, 1, Hkv, d), -1.75)), (B, S, Hkv, d)))
    _, _, va3 = orc.dense(q, _bf(rng.standard_normal((B, S, Hkv, d))), vc, False, 0.3, threads=1, vabs=True)
    _close(va3, np.full_like(va3, 1.75), 1e-13, "weighted |V| of constant V")
    # paged: the identical-key case laid out in pages
    pq, pk, pv, tab, cu, kv = _small_paged(32, [S], Hq, Hkv, d, 4, False)
    pk = np.ascontiguousarray(np.broadcast_to(k0[0, 0][None, None], pk.shape))
    _, _, vap = orc.paged(pq, pk, pv, tab, cu, kv, True, 0.3, threads=2, vabs=True)
    vpf = _f64(pv)
    seq_rows = np.stack([vpf[tab[0, j // 4], j % 4, 0] for j in range(S)])
    for i in range(S):
        _close(vap[i, 0], np.abs(seq_rows[:i + 1]).mean(axis=0), 1e-13, "paged weighted |V| of identical keys")
    # a decode row of a sequence with no key has no weights: zero
    pq, pk, pv, tab, cu, kv = _small_paged(33, [5, 0], Hq, Hkv, d, 4, True)
    tab = np.where(tab < 0, 0, tab)  # the empty sequence's entry is never read
    _, _, vae = orc.paged(pq, pk, pv, tab, cu, kv, True, 0.3, threads=1, vabs=True)
    _close(vae[1], np.zeros_like(vae[1]), 0.0, "weighted |V| of a row with no key")


ALL_PINS = [
    pin_identical_keys,
    pin_dominant_key,
    pin_large_scores_stay_exact,
    pin_causal_first_row,
    pin_rows_of_p_sum_to_one,
    pin_scale_zero,
    pin_linear_in_v,
    pin_shift_invariance,
    pin_permutation_equivariance,
    pin_gqa_equals_repeated_mha,
    pin_bottom_right_causal,
    pin_rows_without_keys,
    pin_sdpa_fp64,
    pin_bruteforce_high_precision,
    pin_paged_equals_dense,
    pin_paged_rows_subset,
    pin_vabs_closed_forms,
]
