"""Paged KV append oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
module. The product path never imports it.

What it computes: "I/O-Aware Kernels" (datasystem.school, Module 5), section "FlashInfer:
I/O-aware attention for serving" keeps each sequence's keys and values in fixed-size pages of a
shared pool, found through a per-sequence page table. Appending tokens to a sequence means
writing their rows at the positions that follow its current length:

* new token r (counting from 0) of sequence s takes logical position kv_lens_before[s] + r;
* logical position p of sequence s is slot p mod page_size of physical page
  page_table[s][floor(p / page_size)].

This is data movement only (no arithmetic), written as one plain Python loop over tokens.
Pinned in ``tests/test_oracle_append.py`` against the attention oracle's own page addressing,
step-by-step appends and untouched-slot invariants; planted mistakes are caught there too.
"""
from __future__ import annotations

import numpy as np


def paged_append(k_pages, v_pages, page_table, kv_lens_before, cu_seqlens_new, k_new, v_new):
    """Return copies of (k_pages, v_pages) with the new rows written into their slots.

    k_pages, v_pages: [num_pages, page_size, Hkv, d] (any dtype, e.g. uint16 bf16 bits);
    page_table: int [num_seqs, max_pages_per_seq]; kv_lens_before: int [num_seqs];
    cu_seqlens_new: int [num_seqs + 1]; k_new, v_new: [total_new, Hkv, d].
    Raises ValueError when a new row's position falls outside the table or its page id outside
    the pool (the inputs are left untouched).
    """
    k_out = np.array(k_pages, copy=True)
    v_out = np.array(v_pages, copy=True)
    num_pages, page_size = k_out.shape[0], k_out.shape[1]
    num_seqs, max_pages = page_table.shape
    for s in range(num_seqs):
        first, end = int(cu_seqlens_new[s]), int(cu_seqlens_new[s + 1])
        for t in range(first, end):
            pos = int(kv_lens_before[s]) + (t - first)
            logical_page, slot = divmod(pos, page_size)
            if pos < 0 or logical_page >= max_pages:
                raise ValueError(f"sequence {s}: position {pos} is outside its page table")
            page = int(page_table[s, logical_page])
            if not 0 <= page < num_pages:
                raise ValueError(f"sequence {s}: page id {page} is outside the pool")
            k_out[page, slot] = k_new[t]
            v_out[page, slot] = v_new[t]
    return k_out, v_out
