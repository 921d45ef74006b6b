"""Seeded synthetic inputs shaped like the workloads of "I/O-Aware Kernels" (datasystem.school,
Module 5): long-context prefill, paged variable-length serving batches and grouped-query decode.

This module draws random numbers and lays them out; it holds none of the attention arithmetic.
Both the CUDA path and the fp64 oracle consume exactly the arrays made here:

* activations are drawn in fp32 from ``numpy.random.PCG64`` streams and rounded to bf16 with
  round-to-nearest-even; they are returned as uint16 bit patterns;
* integers "uniform in [a, b]" include both ends;
* a paged pool holds exactly sum(ceil(kv_len / page_size)) pages whose physical ids are a seeded
  permutation, assigned in logical page order; unused page-table entries are -1.

Large arrays are filled in fixed 4 Mi-element chunks, each from its own child seed of
``SeedSequence(seed)``, so results do not depend on the number of worker threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return 4


def normal_bf16(seed: int, shape, scale: float = 1.0, stream: int = 0) -> np.ndarray:
    """iid N(0,1) * scale in fp32, rounded to bf16; returns uint16 bits of the given shape."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    n_chunks = max(1, (n + CHUNK - 1) // CHUNK)
    children = np.random.SeedSequence([seed, stream]).spawn(n_chunks)

    def fill(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[lo:hi] = bf16_bits(x)

    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


# ----------------------------------------------------------------------------- dense


@dataclass
class DenseWorkload:
    """Dense [B, S, H, d] attention; q/o use Hq heads, k/v use Hkv heads."""

    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    d: int
    causal: bool
    seed: int
    act_scale: float = 1.0          # every activation is multiplied by this before rounding
    outlier_frac: float = 0.0       # fraction of key positions whose K rows are multiplied ...
    outlier_gain: float = 1.0       # ... by this factor (all kv heads), before rounding

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def allowed_scores(self) -> int:
        """Number of (query, key) pairs that are attended (the algorithmic work unit)."""
        per_head = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return self.B * self.Hq * per_head

    def flops(self) -> float:
        """Algorithmic flops: 2d for the score dot product and 2d for P.V per attended pair."""
        return 4.0 * self.d * self.allowed_scores()


def make_dense(w: DenseWorkload):
    """Returns dict(q, k, v) of uint16 bf16 bits."""
    q = normal_bf16(w.seed, (w.B, w.S, w.Hq, w.d), w.act_scale, stream=0)
    v = normal_bf16(w.seed, (w.B, w.S, w.Hkv, w.d), w.act_scale, stream=2)
    if w.outlier_frac > 0.0:
        n = int(round(w.outlier_frac * w.S))
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 99])))
        pos = np.sort(g.permutation(w.S)[:n])
        # K is drawn in fp32 per batch so the outlier gain is applied before bf16 rounding
        kf = np.empty((w.B, w.S, w.Hkv, w.d), dtype=np.uint16)
        for b in range(w.B):
            g2 = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 1, b])))
            x = g2.standard_normal((w.S, w.Hkv, w.d), dtype=np.float32) * np.float32(w.act_scale)
            x[pos] *= np.float32(w.outlier_gain)
            kf[b] = bf16_bits(x)
        return dict(q=q, k=kf, v=v, outlier_positions=pos)
    k = normal_bf16(w.seed, (w.B, w.S, w.Hkv, w.d), w.act_scale, stream=1)
    return dict(q=q, k=k, v=v)


# ----------------------------------------------------------------------------- paged


@dataclass
class PagedWorkload:
    """Paged, ragged batch. q is packed [total_q, Hq, d]; pages are [P, page_size, Hkv, d]."""

    name: str
    num_seqs: int
    len_lo: int
    len_hi: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    causal: bool
    decode: bool          # True: one query token per sequence; False: q_len = kv_len
    seed: int
    lengths: list = field(default=None)  # explicit kv lengths override the random draw
    # query lengths other than "all of kv_len" (prefill) or 1 (decode); each sequence's queries
    # are its last q_len tokens:
    q_lo: int = 0         # q_hi > 0: q_len ~ U[q_lo, q_hi], at most kv_len (multi-token verify)
    q_hi: int = 0
    mix: tuple = None     # (n_full, n_chunk, chunk_lo, chunk_hi): n_full sequences with
    #                       q_len = kv_len, n_chunk with q_len ~ U[chunk_lo, chunk_hi] (at most
    #                       kv_len), the rest q_len = 1; roles from a seeded permutation

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def paged_layout(w: PagedWorkload):
    """Lengths, cu_seqlens_q, page table and pool size (no activations)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 7])))
    if w.lengths is not None:
        kv_lens = np.asarray(w.lengths, dtype=np.int32)
    else:
        kv_lens = g.integers(w.len_lo, w.len_hi + 1, size=w.num_seqs).astype(np.int32)
    q_lens = np.ones_like(kv_lens) if w.decode else kv_lens.copy()
    if w.mix is not None:
        n_full, n_chunk, lo, hi = w.mix
        roles = g.permutation(len(kv_lens))
        q_lens = np.ones_like(kv_lens)
        q_lens[roles[:n_full]] = kv_lens[roles[:n_full]]
        chunk = roles[n_full:n_full + n_chunk]
        q_lens[chunk] = np.minimum(g.integers(lo, hi + 1, size=len(chunk)), kv_lens[chunk])
    elif w.q_hi > 0:
        q_lens = np.minimum(g.integers(w.q_lo, w.q_hi + 1, size=len(kv_lens)), kv_lens).astype(np.int32)
    cu = np.zeros(len(kv_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    pages_per_seq = (kv_lens + w.page_size - 1) // w.page_size
    num_pages = int(pages_per_seq.sum())
    max_pages = int(max(1, pages_per_seq.max()))
    perm = g.permutation(num_pages).astype(np.int32)
    table = np.full((len(kv_lens), max_pages), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(pages_per_seq):
        table[s, :n] = perm[off:off + n]
        off += n
    return dict(kv_lens=kv_lens, q_lens=q_lens, cu_seqlens_q=cu, page_table=table,
                num_pages=num_pages, max_pages_per_seq=max_pages)


def make_paged(w: PagedWorkload):
    """Returns the layout plus q, k_pages, v_pages (uint16 bf16 bits)."""
    lay = paged_layout(w)
    total_q = int(lay["cu_seqlens_q"][-1])
    P = lay["num_pages"]
    q = normal_bf16(w.seed, (total_q, w.Hq, w.d), 1.0, stream=10)
    kp = normal_bf16(w.seed, (P, w.page_size, w.Hkv, w.d), 1.0, stream=11)
    vp = normal_bf16(w.seed, (P, w.page_size, w.Hkv, w.d), 1.0, stream=12)
    lay.update(q=q, k_pages=kp, v_pages=vp, total_q=total_q)
    return lay


def make_append(w: PagedWorkload):
    """A cache fill: every key/value row of the batch's sequences, packed sequence after sequence,
    to be appended into an empty pool (kv_lens_before = 0). Returns the layout plus k_new, v_new
    (uint16 bf16 bits, [total_new, Hkv, d]), cu_seqlens_new and kv_lens_before."""
    lay = paged_layout(w)
    total = int(lay["kv_lens"].astype(np.int64).sum())
    cu = np.zeros(len(lay["kv_lens"]) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lay["kv_lens"])
    lay.update(k_new=normal_bf16(w.seed, (total, w.Hkv, w.d), 1.0, stream=30),
               v_new=normal_bf16(w.seed, (total, w.Hkv, w.d), 1.0, stream=31),
               cu_seqlens_new=cu, kv_lens_before=np.zeros(len(lay["kv_lens"]), dtype=np.int32), total_new=total)
    return lay


@dataclass
class CascadeWorkload:
    """A decode-style batch whose sequences share one prefix: num_seqs sequences, each with q_len
    query tokens at the end of its own suffix (suffix lengths uniform in [suffix_lo, suffix_hi]),
    all behind the same prefix_len shared keys. One pool holds the prefix pages once and every
    sequence's suffix pages."""

    name: str
    num_seqs: int
    prefix_len: int
    suffix_lo: int
    suffix_hi: int
    q_len: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def make_cascade(w: CascadeWorkload):
    """Cascade inputs plus the same batch laid out flat (each sequence's table lists the shared
    prefix pages, then its own; valid when prefix_len is a multiple of page_size)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 7])))
    kv_lens = g.integers(w.suffix_lo, w.suffix_hi + 1, size=w.num_seqs).astype(np.int32)
    ps = w.page_size
    n_prefix = (w.prefix_len + ps - 1) // ps
    n_suffix = (kv_lens + ps - 1) // ps
    P = int(n_prefix + n_suffix.sum())
    perm = g.permutation(P).astype(np.int32)
    prefix_table = perm[:n_prefix].reshape(1, -1).copy() if n_prefix else np.full((1, 1), -1, np.int32)
    table = np.full((w.num_seqs, max(1, int(n_suffix.max()))), -1, dtype=np.int32)
    off = n_prefix
    for s, n in enumerate(n_suffix):
        table[s, :n] = perm[off:off + n]
        off += n
    q_lens = np.full(w.num_seqs, w.q_len, dtype=np.int32)
    cu = np.zeros(w.num_seqs + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    total_q = int(cu[-1])
    flat = np.full((w.num_seqs, n_prefix + table.shape[1]), -1, dtype=np.int32)
    flat[:, :n_prefix] = prefix_table[0, :n_prefix]
    flat[:, n_prefix:] = table
    return dict(
        q=normal_bf16(w.seed, (total_q, w.Hq, w.d), 1.0, stream=10),
        k_pages=normal_bf16(w.seed, (P, ps, w.Hkv, w.d), 1.0, stream=11),
        v_pages=normal_bf16(w.seed, (P, ps, w.Hkv, w.d), 1.0, stream=12),
        num_pages=P, cu_q_groups=np.array([0, total_q], dtype=np.int32), prefix_page_table=prefix_table,
        prefix_lens=np.array([w.prefix_len], dtype=np.int32), cu_seqlens_q=cu, q_lens=q_lens, page_table=table,
        kv_lens=kv_lens, total_q=total_q, flat_page_table=flat, flat_kv_lens=(kv_lens + w.prefix_len).astype(np.int32))


def paged_allowed_scores(lay, Hq: int, causal: bool) -> int:
    total = 0
    for ql, kl in zip(lay["q_lens"].tolist(), lay["kv_lens"].tolist()):
        if causal:
            # row i sees min(kv, i + kv - ql + 1) keys (bottom-right alignment), at least 0
            off = kl - ql
            for_rows = np.clip(np.arange(ql) + off + 1, 0, kl)
            total += int(for_rows.sum())
        else:
            total += ql * kl
    return total * Hq


# ----------------------------------------------------------------------------- named workloads

WORKLOADS = {
    "dense_noncausal_b1_h2_s256_d64": DenseWorkload(
        "dense_noncausal_b1_h2_s256_d64", B=1, S=256, Hq=2, Hkv=2, d=64, causal=False, seed=1000),
    "causal_prefill_b4_h32_s4096_d128": DenseWorkload(
        "causal_prefill_b4_h32_s4096_d128", B=4, S=4096, Hq=32, Hkv=32, d=128, causal=True, seed=1001),
    # the headline shape at the small workload's head dim (64)
    "causal_prefill_b4_h32_s4096_d64": DenseWorkload(
        "causal_prefill_b4_h32_s4096_d64", B=4, S=4096, Hq=32, Hkv=32, d=64, causal=True, seed=1009),
    "gqa_causal_prefill_b1_hq32_hkv8_s32768_d128": DenseWorkload(
        "gqa_causal_prefill_b1_hq32_hkv8_s32768_d128", B=1, S=32768, Hq=32, Hkv=8, d=128, causal=True,
        seed=1002, act_scale=0.5, outlier_frac=0.01, outlier_gain=8.0),
    "paged_prefill_64seq_512_8192_hq32_hkv8_d128_p16": PagedWorkload(
        "paged_prefill_64seq_512_8192_hq32_hkv8_d128_p16", num_seqs=64, len_lo=512, len_hi=8192,
        Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=False, seed=1003),
    "paged_decode_128seq_1024_16384_hq32_hkv8_d128_p16": PagedWorkload(
        "paged_decode_128seq_1024_16384_hq32_hkv8_d128_p16", num_seqs=128, len_lo=1024,
        len_hi=16384, Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=True, seed=1004),
    # a small decode batch of the same length distribution: too few (sequence, kv head) units to
    # fill the GPU, so the keys are split and the partial states merged by their LSE
    "paged_decode_16seq_1024_16384_hq32_hkv8_d128_p16": PagedWorkload(
        "paged_decode_16seq_1024_16384_hq32_hkv8_d128_p16", num_seqs=16, len_lo=1024,
        len_hi=16384, Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=True, seed=1008),
    # one launch mixing full prefill (16 seqs), chunked prefill (16 seqs, chunks of 1..512 new
    # tokens behind their cached keys) and decode (32 seqs), kv_len 512..8192
    "mixed_paged_64seq_512_8192_hq32_hkv8_d128_p16": PagedWorkload(
        "mixed_paged_64seq_512_8192_hq32_hkv8_d128_p16", num_seqs=64, len_lo=512, len_hi=8192,
        Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=False, seed=1006, mix=(16, 16, 1, 512)),
    # speculative-decoding verification: 2..8 draft tokens per sequence behind 1024..16384 keys
    "verify_paged_128seq_q2_8_kv1024_16384_hq32_hkv8_d128_p16": PagedWorkload(
        "verify_paged_128seq_q2_8_kv1024_16384_hq32_hkv8_d128_p16", num_seqs=128, len_lo=1024,
        len_hi=16384, Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=False, seed=1007, q_lo=2, q_hi=8),
    # 128 decode sequences behind one shared 16384-token prefix, own suffixes of 256..2048 tokens
    "cascade_decode_128seq_prefix16384_suffix256_2048_hq32_hkv8_d128_p16": CascadeWorkload(
        "cascade_decode_128seq_prefix16384_suffix256_2048_hq32_hkv8_d128_p16", num_seqs=128, prefix_len=16384,
        suffix_lo=256, suffix_hi=2048, q_len=1, Hq=32, Hkv=8, d=128, page_size=16, seed=1005),
    # the K/V cache fill of the paged prefill batch above (same lengths and page table)
    "paged_append_64seq_512_8192_hkv8_d128_p16": PagedWorkload(
        "paged_append_64seq_512_8192_hkv8_d128_p16", num_seqs=64, len_lo=512, len_hi=8192,
        Hq=32, Hkv=8, d=128, page_size=16, causal=True, decode=False, seed=1003),
}
