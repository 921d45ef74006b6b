"""Shared-prefix (cascade) attention on the GPU against the fp64 oracle. The oracle attends each
sequence over its prefix keys followed by its suffix keys, laid out contiguously (gathered here
through the page tables); the cascade path attends the prefix once per group and merges."""
import math

import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import WORKLOADS, make_cascade, normal_bf16
from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev

pytestmark = pytest.mark.gpu

NAN_BITS = np.uint16(0x7FC0)


def build(groups, prefix_lens, q_lens, suffix_lens, Hq, Hkv, d, ps, seed):
    """groups: number of consecutive sequences in each group. Pages of prefixes and suffixes are
    interleaved in one pool by a seeded permutation; unused slots of last pages hold NaN."""
    rng = np.random.default_rng(seed)
    n_pre = [(P + ps - 1) // ps for P in prefix_lens]
    n_suf = [(L + ps - 1) // ps for L in suffix_lens]
    total_pages = sum(n_pre) + sum(n_suf) + 2
    perm = rng.permutation(total_pages).astype(np.int32)
    kp = normal_bf16(seed, (total_pages, ps, Hkv, d), stream=1)
    vp = normal_bf16(seed, (total_pages, ps, Hkv, d), stream=2)
    off = 0
    pre_table = np.full((len(groups), max(1, max(n_pre))), -1, np.int32)
    for g, n in enumerate(n_pre):
        pre_table[g, :n] = perm[off:off + n]
        off += n
    table = np.full((len(q_lens), max(1, max(n_suf))), -1, np.int32)
    for s, n in enumerate(n_suf):
        table[s, :n] = perm[off:off + n]
        off += n
    for tbl, lens in ((pre_table, prefix_lens), (table, suffix_lens)):
        for r, L in enumerate(lens):
            if L % ps:
                last = tbl[r, (L - 1) // ps]
                kp[last, L % ps:] = NAN_BITS
                vp[last, L % ps:] = NAN_BITS
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    first = np.concatenate([[0], np.cumsum(groups)]).astype(np.int32)
    cu_groups = cu[first]
    q = normal_bf16(seed, (int(cu[-1]), Hq, d), stream=3)
    return dict(q=q, kp=kp, vp=vp, pre_table=pre_table, prefix_lens=np.asarray(prefix_lens, np.int32),
                cu_groups=cu_groups, table=table, kv_lens=np.asarray(suffix_lens, np.int32), cu=cu,
                q_lens=np.asarray(q_lens, np.int32), groups=groups, max_group_q=int(np.diff(cu_groups).max()))


def oracle_flat(c, causal, scale):
    """Each sequence's prefix ++ suffix keys written contiguously into fresh pages, then the
    paged oracle (bottom-right causal over the full length)."""
    ps = c["kp"].shape[1]
    group_of = np.repeat(np.arange(len(c["groups"])), c["groups"])
    rows_k, rows_v, lens = [], [], []
    for s in range(len(c["q_lens"])):
        g = group_of[s]
        idx = [(c["pre_table"][g, p // ps], p % ps) for p in range(int(c["prefix_lens"][g]))]
        idx += [(c["table"][s, p // ps], p % ps) for p in range(int(c["kv_lens"][s]))]
        pg = np.array([i[0] for i in idx], np.int64)
        sl = np.array([i[1] for i in idx], np.int64)
        rows_k.append(c["kp"][pg, sl])
        rows_v.append(c["vp"][pg, sl])
        lens.append(len(idx))
    n_pages = [(L + ps - 1) // ps for L in lens]
    shape = (sum(n_pages),) + c["kp"].shape[1:]
    k2, v2 = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    table2 = np.full((len(lens), max(1, max(n_pages))), -1, np.int32)
    off = 0
    for s, (L, n) in enumerate(zip(lens, n_pages)):
        table2[s, :n] = np.arange(off, off + n)
        k2[off:off + n].reshape(-1, *shape[2:])[:L] = rows_k[s]
        v2[off:off + n].reshape(-1, *shape[2:])[:L] = rows_v[s]
        off += n
    return oracle.get().paged(c["q"], k2, v2, table2, c["cu"], np.asarray(lens, np.int32), causal, scale,
                              vabs=True)


def run_cascade(c, causal, scale):
    import torch

    import io_aware_exact_flash_gb300 as fa

    o, lse = fa.fa_cascade_fwd(to_dev(c["q"]), to_dev(c["kp"]), to_dev(c["vp"]), i32_dev(c["cu_groups"]),
                               i32_dev(c["pre_table"]), i32_dev(c["prefix_lens"]), c["max_group_q"],
                               i32_dev(c["cu"]), i32_dev(c["table"]), i32_dev(c["kv_lens"]), int(c["q_lens"].max()),
                               causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("ps", [16, 64])
def test_cascade_decode_one_group(ps):
    """Decode rows (one per sequence) behind a shared prefix that does not end on a page edge."""
    suffix = [1, 5, 16, 17, 100, 300, 2, 64, 129]
    c = build([len(suffix)], [300], [1] * len(suffix), suffix, 32, 8, 128, ps, seed=40 + ps)
    scale = 1 / math.sqrt(128)
    o, lse = run_cascade(c, True, scale)
    o_ref, lse_ref, va_ref = oracle_flat(c, True, scale)
    compare(o, o_ref, lse, lse_ref, f"cascade decode ps={ps}", vabs=va_ref)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (64, 4, 4)])
def test_cascade_groups_and_chunks(causal, d, Hq, Hkv):
    """Several groups (one without a shared prefix), query chunks of several rows per sequence
    (chunked prefill / multi-token verify behind a shared prefix)."""
    groups = [3, 2, 1]
    prefix = [64, 0, 129]
    q_lens = [5, 1, 17, 3, 40, 2]
    suffix = [5, 30, 17, 200, 40, 9]
    c = build(groups, prefix, q_lens, suffix, Hq, Hkv, d, 16, seed=50 + d)
    scale = 1 / math.sqrt(d)
    o, lse = run_cascade(c, causal, scale)
    o_ref, lse_ref, va_ref = oracle_flat(c, causal, scale)
    compare(o, o_ref, lse, lse_ref, f"cascade groups causal={causal} d={d}", vabs=va_ref)


def test_cascade_prefix_pass_on_the_key_row_kernel():
    """Groups of one to four decode rows at group size 4 (at most 16 query rows per kv head), so
    the prefix pass runs on the key-row decode kernel too, with the cascade's fork event recorded
    between that pass's planning kernel and its attention kernel."""
    groups = [4, 3, 1, 2]
    prefix = [700, 2049, 16, 300]
    suffix = [1, 5, 16, 17, 100, 300, 2, 64, 129, 1000]
    c = build(groups, prefix, [1] * len(suffix), suffix, 32, 8, 128, 16, seed=61)
    scale = 1 / math.sqrt(128)
    o, lse = run_cascade(c, True, scale)
    o_ref, lse_ref, va_ref = oracle_flat(c, True, scale)
    compare(o, o_ref, lse, lse_ref, "cascade, key-row prefix pass", vabs=va_ref)


def test_cascade_full_size_decode():
    """128 decode sequences behind one 16384-token prefix (suffixes of 256..2048 tokens): every
    output row against the oracle over the flat layout (the prefix is page aligned, so each
    sequence's flat table lists the shared prefix pages, then its own)."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    w = WORKLOADS["cascade_decode_128seq_prefix16384_suffix256_2048_hq32_hkv8_d128_p16"]
    t = make_cascade(w)
    kp, vp = to_dev(t["k_pages"]), to_dev(t["v_pages"])
    o, lse = fa.fa_cascade_fwd(to_dev(t["q"]), kp, vp, i32_dev(t["cu_q_groups"]), i32_dev(t["prefix_page_table"]),
                               i32_dev(t["prefix_lens"]), t["total_q"], i32_dev(t["cu_seqlens_q"]),
                               i32_dev(t["page_table"]), i32_dev(t["kv_lens"]), w.q_len, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    o_ref, lse_ref, va_ref = oracle.get().paged(t["q"], t["k_pages"], t["v_pages"], t["flat_page_table"], t["cu_seqlens_q"],
                                        t["flat_kv_lens"], True, w.scale, vabs=True)
    compare(bf16_to_f64(o), o_ref, lse.cpu().numpy().astype(np.float64), lse_ref, "cascade full size", vabs=va_ref)
