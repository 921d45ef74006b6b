"""Paged, ragged attention (prefill through the tensor-core kernel, decode through split-KV)
on the GPU against the fp64 oracle."""
import math

import numpy as np
import pytest

import oracle
from io_aware_exact_flash_gb300.workloads import WORKLOADS, PagedWorkload, make_paged
from tests.helpers import bf16_to_f64, compare, i32_dev, to_dev

pytestmark = pytest.mark.gpu

NAN_BF16 = np.uint16(0x7FC0)


def build_case(lengths, Hq, Hkv, d, page_size, decode, seed, q_lens=None, extra_pages=0, poison=True):
    """Paged inputs for the given kv lengths (q_len = kv_len for prefill, 1 for decode, or
    explicit q_lens). Unused slots of last pages and `extra_pages` unreferenced pool pages hold
    NaN when poison is set, so any read of them would show in the output."""
    w = PagedWorkload("case", num_seqs=len(lengths), len_lo=0, len_hi=0, Hq=Hq, Hkv=Hkv, d=d,
                      page_size=page_size, causal=True, decode=decode, seed=seed, lengths=list(lengths))
    t = make_paged(w)
    if q_lens is not None:
        from io_aware_exact_flash_gb300.workloads import normal_bf16

        q_lens = np.asarray(q_lens, np.int32)
        cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        t["cu_seqlens_q"] = cu
        t["q_lens"] = q_lens
        t["q"] = normal_bf16(seed + 1, (int(cu[-1]), Hq, d), stream=20)
        t["total_q"] = int(cu[-1])
    kp, vp = t["k_pages"], t["v_pages"]
    if extra_pages:
        shape = (extra_pages,) + kp.shape[1:]
        kp = np.concatenate([kp, np.full(shape, NAN_BF16)])
        vp = np.concatenate([vp, np.full(shape, NAN_BF16)])
    if poison:
        kp, vp = kp.copy(), vp.copy()
        for s, L in enumerate(t["kv_lens"].tolist()):
            if L % page_size:
                last = t["page_table"][s, (L - 1) // page_size]
                kp[last, L % page_size:] = NAN_BF16
                vp[last, L % page_size:] = NAN_BF16
    t["k_pages"], t["v_pages"] = kp, vp
    t["num_pages"] = kp.shape[0]
    return t


def run_paged(t, causal, scale, num_splits=0):
    import torch

    import io_aware_exact_flash_gb300 as fa

    max_q = int(t["q_lens"].max()) if len(t["q_lens"]) else 1
    o, lse = fa.fa_paged_fwd(to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"]), i32_dev(t["page_table"]),
                             i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"]), max_q_len=max(1, max_q),
                             causal=causal, scale=scale, num_splits=num_splits)
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, f"device status {code} at site {site}"
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def oracle_paged(t, causal, scale):
    return oracle.get().paged(t["q"], t["k_pages"], t["v_pages"], t["page_table"], t["cu_seqlens_q"], t["kv_lens"],
                              causal, scale, vabs=True)


PREFILL_LENGTHS = [1, 15, 16, 17, 100, 128, 129, 255, 256, 257, 300, 513]


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
def test_paged_prefill_page_sizes(page_size):
    t = build_case(PREFILL_LENGTHS, 8, 2, 128, page_size, False, 11 + page_size, extra_pages=3)
    scale = 1 / math.sqrt(128)
    o, lse = run_paged(t, True, scale)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, scale)
    compare(o, o_ref, lse, lse_ref, f"paged prefill ps={page_size}", vabs=va_ref)


@pytest.mark.parametrize("d,Hq,Hkv,causal", [(64, 4, 4, True), (128, 4, 1, False), (64, 8, 1, False),
                                             (128, 6, 3, True), (128, 32, 1, True), (64, 16, 1, False),
                                             (128, 12, 4, True)])
def test_paged_prefill_heads_and_dims(d, Hq, Hkv, causal):
    t = build_case([40, 700, 129, 1, 384], Hq, Hkv, d, 16, False, 5 + d + Hq)
    o, lse = run_paged(t, causal, 1 / math.sqrt(d))
    o_ref, lse_ref, va_ref = oracle_paged(t, causal, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, f"paged prefill d={d} Hq={Hq} Hkv={Hkv} causal={causal}", vabs=va_ref)


def test_paged_prefill_query_shorter_than_keys():
    """Chunked prefill: the last q_len tokens of each sequence attend to a longer cached prefix
    (bottom-right causal alignment)."""
    lengths = [300, 1000, 77, 512]
    t = build_case(lengths, 8, 2, 128, 16, False, 21, q_lens=[45, 257, 77, 2])
    o, lse = run_paged(t, True, 0.08)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 0.08)
    compare(o, o_ref, lse, lse_ref, "chunked prefill", vabs=va_ref)


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (64, 8, 8), (128, 16, 2), (128, 8, 4), (128, 32, 1),
                                     (64, 12, 4), (128, 6, 1)])
def test_paged_decode_splits(splits, d, Hq, Hkv):
    lengths = [1, 16, 17, 1000, 4096, 3333, 64, 250]
    t = build_case(lengths, Hq, Hkv, d, 16, True, 31 + d + Hq, extra_pages=2)
    o, lse = run_paged(t, True, 1 / math.sqrt(d), num_splits=splits)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, f"decode splits={splits} d={d} Hq={Hq} Hkv={Hkv}", vabs=va_ref)


@pytest.mark.parametrize("page_size", [32, 128])
def test_paged_decode_page_sizes(page_size):
    t = build_case([5, 130, 999, 2048], 8, 2, 128, page_size, True, 41)
    o, lse = run_paged(t, True, 0.1, num_splits=3)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 0.1)
    compare(o, o_ref, lse, lse_ref, f"decode ps={page_size}", vabs=va_ref)


def test_paged_decode_empty_sequence():
    """A sequence with no keys gets O = 0 and LSE = -inf; the others are unaffected."""
    t = build_case([100, 0, 37], 4, 2, 128, 16, True, 51)
    for splits in (1, 2):
        o, lse = run_paged(t, True, 0.1, num_splits=splits)
        o_ref, lse_ref, va_ref = oracle_paged(t, True, 0.1)
        compare(o, o_ref, lse, lse_ref, f"decode with empty sequence, splits={splits}", vabs=va_ref)
        assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))


def test_key_row_many_key_splits():
    """The key-row kernel with 16 key splits over sequences of 0 to 5000 keys, so most splits of
    the short sequences hold no key tile, and verify rows besides decode ones; a second call gives
    the same bits (the planning state is rebuilt on every call)."""
    t = build_case([1, 0, 130, 5000, 16, 2049, 700, 3], 32, 8, 128, 16, False, 97, q_lens=[1, 1, 2, 1, 4, 1, 3, 1],
                   extra_pages=2)
    o1, lse1 = run_paged(t, True, 1 / math.sqrt(128), num_splits=16)
    o2, lse2 = run_paged(t, True, 1 / math.sqrt(128), num_splits=16)
    assert np.array_equal(o1, o2) and np.array_equal(lse1, lse2)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(128))
    compare(o1, o_ref, lse1, lse_ref, "key rows, 16 key splits", vabs=va_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [0, 2])
def test_partly_filled_query_tiles_over_many_key_tiles(d, splits):
    """Chunks of 1 to 40 tokens at the end of 640 to 2560 keys, one query head per kv head, so a
    query tile has one or two warps with query rows and two or three without, over 5 to 20 key
    tiles. At d = 64 a tile's next scores can be ready before its P is released; the warps without
    rows must still arrive on the P barrier in their own tile's phase, which a wrong order breaks
    (non-finite or wrong O)."""
    lengths = [700, 2049, 1500, 640, 2560, 999]
    q_lens = [1, 17, 33, 40, 9, 31]
    t = build_case(lengths, 8, 8, d, 64, False, 131 + d + splits, q_lens=q_lens, extra_pages=2)
    o, lse = run_paged(t, True, 1 / math.sqrt(d), num_splits=splits)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, f"partly filled tiles d={d} splits={splits}", vabs=va_ref)


def test_paged_prefill_full_size_sampled():
    """The ragged paged prefill workload (64 sequences, lengths 512..8192) at full size, in the
    benchmark's launch configuration, checked on sampled (token, head) rows."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    w = WORKLOADS["paged_prefill_64seq_512_8192_hq32_hkv8_d128_p16"]
    t = make_paged(w)
    o, lse = fa.fa_paged_fwd(to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"]), i32_dev(t["page_table"]),
                             i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"]), max_q_len=int(t["q_lens"].max()),
                             causal=True, scale=w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    cu = t["cu_seqlens_q"]
    rows = []
    for s in range(w.num_seqs):
        for i in (0, int(t["q_lens"][s]) - 1, int(rng.integers(t["q_lens"][s]))):
            rows.append((int(cu[s]) + i, int(rng.integers(w.Hq))))
    rows = np.array(rows, np.int64)
    o_ref, lse_ref, va_ref = oracle.get().paged_rows(t["q"], t["k_pages"], t["v_pages"], t["page_table"], cu, t["kv_lens"],
                                             True, w.scale, rows, vabs=True)
    ridx = torch.from_numpy(rows).cuda()
    compare(bf16_to_f64(o[ridx[:, 0], ridx[:, 1]]), o_ref, lse[ridx[:, 0], ridx[:, 1]].cpu().numpy(), lse_ref,
            "paged prefill full size", vabs=va_ref)
    assert bool(torch.isfinite(o.float()).all())


def test_paged_decode_full_size():
    """The GQA decode workload (128 sequences, kv lengths 1024..16384) at full size, with the
    automatic split count the benchmark uses, against the oracle on every row."""
    w = WORKLOADS["paged_decode_128seq_1024_16384_hq32_hkv8_d128_p16"]
    t = make_paged(w)
    o, lse = run_paged(t, True, w.scale, num_splits=0)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, w.scale)
    compare(o, o_ref, lse, lse_ref, "decode full size", vabs=va_ref)


def test_mixed_batch_prefill_chunks_and_decode():
    """One launch over a batch mixing full prefill (q_len = kv_len), chunked prefill (a few new
    tokens behind cached keys) and decode rows (q_len = 1), bottom-right causal."""
    lengths = [300, 1, 77, 1000, 129, 16, 2048, 5, 513, 64]
    q_lens = [300, 1, 1, 129, 1, 16, 1, 3, 257, 1]
    t = build_case(lengths, 8, 2, 128, 16, False, 61, q_lens=q_lens, extra_pages=2)
    for causal in (True, False):
        o, lse = run_paged(t, causal, 0.09)
        o_ref, lse_ref, va_ref = oracle_paged(t, causal, 0.09)
        compare(o, o_ref, lse, lse_ref, f"mixed batch causal={causal}", vabs=va_ref)


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (64, 8, 2), (128, 32, 1), (128, 12, 4)])
def test_multi_token_verify(d, Hq, Hkv):
    """Speculative-decoding verification: 2..8 query tokens at the end of every sequence, each
    seeing the cached keys and the draft tokens before it."""
    lengths = [2, 8, 9, 100, 1024, 3000, 777, 16]
    q_lens = [2, 8, 3, 5, 8, 7, 2, 6]
    t = build_case(lengths, Hq, Hkv, d, 16, False, 71 + d, q_lens=q_lens)
    o, lse = run_paged(t, True, 1 / math.sqrt(d))
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, f"verify d={d} Hq={Hq} Hkv={Hkv}", vabs=va_ref)


@pytest.mark.parametrize("Hq,Hkv,q_lens,page_size,splits", [
    (32, 8, [1, 4, 2, 3, 1, 4, 2, 1], 16, 0),    # verify of <= 4 tokens, group 4: 16 query columns
    (32, 8, [2, 1, 2, 2, 1, 1, 2, 2], 64, 3),    # 8 columns, key splits, 64-row pages
    (32, 2, [1] * 8, 16, 0),                     # decode, group 16: 16 columns
    (12, 4, [1, 4, 5, 2, 3, 1, 5, 4], 32, 2),    # group 3 (not a power of two), up to 15 rows
    (8, 8, [1, 2, 4, 3, 1, 4, 2, 1], 128, 0),    # MHA verify, 128-row pages
])
def test_key_row_kernel_shapes(Hq, Hkv, q_lens, page_size, splits):
    """Batches of at most 16 query rows per kv head, which run on the key-row kernel: every
    column count it compiles (4, 8, 16), groups that do and do not divide 16, causal verify rows,
    key splits and page sizes, against the oracle."""
    lengths = [5, 16, 130, 300, 1000, 2049, 777, 4100]
    t = build_case(lengths, Hq, Hkv, 128, page_size, False, 91 + Hq + page_size, q_lens=q_lens, extra_pages=2)
    o, lse = run_paged(t, True, 1 / math.sqrt(128), num_splits=splits)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(128))
    compare(o, o_ref, lse, lse_ref, f"key rows Hq={Hq} Hkv={Hkv} ps={page_size}", vabs=va_ref)


@pytest.mark.parametrize("name", ["mixed_paged_64seq_512_8192_hq32_hkv8_d128_p16",
                                  "verify_paged_128seq_q2_8_kv1024_16384_hq32_hkv8_d128_p16"])
def test_mixed_and_verify_workloads_full_size(name):
    """The mixed and verify workloads at full size in the benchmark's launch configuration:
    every query token of the verify batch (four random heads each), and sampled rows (first,
    last, random of each sequence) of the mixed batch, against the oracle."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    w = WORKLOADS[name]
    t = make_paged(w)
    o, lse = fa.fa_paged_fwd(to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"]), i32_dev(t["page_table"]),
                             i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"]), max_q_len=int(t["q_lens"].max()),
                             causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    cu = t["cu_seqlens_q"]
    rng = np.random.default_rng(2)
    if w.q_hi > 0:
        # every query token, four of its heads
        tok = np.repeat(np.arange(t["total_q"]), 4)
        rows = np.stack([tok, rng.integers(0, w.Hq, len(tok))], axis=1).astype(np.int64)
    else:
        rows = []
        for s in range(w.num_seqs):
            for i in (0, int(t["q_lens"][s]) - 1, int(rng.integers(t["q_lens"][s]))):
                rows.append((int(cu[s]) + i, int(rng.integers(w.Hq))))
        rows = np.array(rows, np.int64)
    o_ref, lse_ref, va_ref = oracle.get().paged_rows(t["q"], t["k_pages"], t["v_pages"], t["page_table"], cu, t["kv_lens"],
                                             True, w.scale, rows, vabs=True)
    ridx = torch.from_numpy(rows).cuda()
    compare(bf16_to_f64(o[ridx[:, 0], ridx[:, 1]]), o_ref, lse[ridx[:, 0], ridx[:, 1]].cpu().numpy(), lse_ref,
            f"{name} full size", vabs=va_ref)
    assert bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("decode", [False, True])
def test_many_tiny_sequences(decode):
    """1500 sequences of 0 to 40 keys: many work items, many packed tiles with a few rows, empty
    sequences among them, and (decode) an automatic split plan over very short key ranges. Rows
    with a handful of keys reach |O| of 2 to 4 with N(0,1) values, the edge of the 1e-2 bound:
    there the output rounding alone is 7.8e-3, so any bias of P's weights shows."""
    rng = np.random.default_rng(81 + decode)
    lengths = rng.integers(0, 41, size=1500).tolist()
    t = build_case(lengths, 32, 8, 128, 16, decode, 83 + decode, extra_pages=2)
    o, lse = run_paged(t, True, 1 / math.sqrt(128))
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(128))
    compare(o, o_ref, lse, lse_ref, f"1500 tiny sequences decode={decode}", vabs=va_ref)


@pytest.mark.parametrize("n_seqs,max_len", [(5000, 300), (20000, 64)])
def test_more_sequences_than_planner_threads(n_seqs, max_len):
    """Thousands of sequences (prefill chunks of 1 to 6 rows over short, often equal lengths): more
    than one per thread of the work-list planner, whose sort then runs over chunks of the batch
    (a stable placement per chunk); every row must be planned exactly once."""
    rng = np.random.default_rng(85 + n_seqs)
    lengths = rng.integers(0, max_len + 1, size=n_seqs).tolist()
    q_lens = [min(L, int(rng.integers(1, 7))) for L in lengths]
    t = build_case(lengths, 8, 2, 64, 16, False, 87, q_lens=q_lens)
    o, lse = run_paged(t, True, 0.125)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 0.125)
    compare(o, o_ref, lse, lse_ref, f"{n_seqs} sequences", vabs=va_ref)


def test_decode_more_splits_than_key_tiles():
    """An explicit split count far above the key tiles of most sequences: most splits are empty
    (LSE = -inf) and must drop out of the merge."""
    lengths = [1, 17, 130, 700, 2000]
    t = build_case(lengths, 32, 8, 128, 16, True, 91)
    o, lse = run_paged(t, True, 1 / math.sqrt(128), num_splits=64)
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(128))
    compare(o, o_ref, lse, lse_ref, "decode with 64 splits", vabs=va_ref)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4)])
def test_more_query_rows_than_keys(Hq, Hkv):
    """Sequences with more query rows than keys: under bottom-right causal masking their top
    q_len - kv_len rows see no key (O = 0, LSE = -inf); without masking every row sees them all."""
    kv = [20, 10, 100, 0, 64]
    q = [50, 10, 300, 7, 65]
    t = build_case(kv, Hq, Hkv, 128, 16, False, 97 + Hq, q_lens=q)
    for causal in (True, False):
        o, lse = run_paged(t, causal, 0.1)
        o_ref, lse_ref, va_ref = oracle_paged(t, causal, 0.1)
        compare(o, o_ref, lse, lse_ref, f"q_len > kv_len causal={causal}", vabs=va_ref)
        if causal:
            top = np.isneginf(lse_ref)
            assert top.any() and np.all(o[top] == 0)


def test_decode_one_million_keys():
    """Decode at a million cached keys (MQA: 8 query heads on one kv head, so the pool stays
    ~0.5 GB): page ids and key positions far from zero, hundreds of key splits, one large merge.
    Every output row against the oracle."""
    lengths = [1_000_000, 3]
    t = build_case(lengths, 8, 1, 128, 16, True, 101, poison=False)
    o, lse = run_paged(t, True, 1 / math.sqrt(128))
    o_ref, lse_ref, va_ref = oracle_paged(t, True, 1 / math.sqrt(128))
    compare(o, o_ref, lse, lse_ref, "decode at 1M keys", vabs=va_ref)


def test_chunk_deep_in_a_long_context():
    """Chunked prefill of 300 new tokens behind 200,000 cached keys (bottom-right causal), next
    to a short sequence: large key-tile indices on the tensor-core path."""
    lengths = [200_300, 50]
    t = build_case(lengths, 8, 2, 128, 16, False, 103, q_lens=[300, 50], poison=False)
    o, lse = run_paged(t, True, 1 / math.sqrt(128))
    rows = np.array([[0, 0], [1, 3], [150, 5], [299, 7], [300, 1], [349, 6]], np.int64)
    o_ref, lse_ref, va_ref = oracle.get().paged_rows(t["q"], t["k_pages"], t["v_pages"], t["page_table"], t["cu_seqlens_q"],
                                             t["kv_lens"], True, 1 / math.sqrt(128), rows, vabs=True)
    compare(o[rows[:, 0], rows[:, 1]], o_ref, lse[rows[:, 0], rows[:, 1]], lse_ref, "chunk at 200K keys", vabs=va_ref)
