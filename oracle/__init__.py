"""Exact-attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package. The product path (``io_aware_exact_flash_gb300``) never imports it.

The arithmetic lives in ``attn_oracle.c``: the naive attention pipeline of "I/O-Aware Kernels"
(datasystem.school, Module 5, section "Naive attention: materializing the k x k score matrix"),
in fp64, one full score row at a time. This module only compiles that file with gcc, loads it
with ctypes and marshals numpy arrays in and out. Every function can also return the
softmax-weighted mean magnitude of V (``vabs=True``): sum_j p_j |v_jc| per element of O, which the
tests use to bound the effect of bf16-rounded softmax weights.

Parity pins for every function here live in ``tests/test_oracle_pins.py``; none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")


def compile_library(source: str = SOURCE, out: str = LIBRARY) -> str:
    """Compile the oracle's C source into a shared library with gcc; returns its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out, source, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    return out


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str = LIBRARY):
        if path == LIBRARY and (
            not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)
        ):
            compile_library()
        self.path = path
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        i64 = ctypes.c_int64
        dbl = ctypes.c_double
        lib.oracle_dense_rows.argtypes = [p, p, p, i, i, i, i, i, i, i, dbl, p, i64, p, p, p, i]
        lib.oracle_dense_rows.restype = i
        lib.oracle_paged_rows.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, i, dbl, p, i64, p, p, p, i]
        lib.oracle_paged_rows.restype = i
        self._lib = lib

    # ------------------------------------------------------------------ dense
    def dense_rows(self, q, k, v, causal, scale, rows, threads=None, vabs=False):
        """Attention for selected rows of the dense layout.

        q: uint16 bf16 bits [B, Sq, Hq, d]; k, v: [B, Skv, Hkv, d]; rows: int64 [n, 3] of
        (b, i, h). Returns (o [n, d] fp64, lse [n] fp64), and the weighted mean |V| [n, d] when asked.
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        B, Sq, Hq, d = q.shape
        Bk, Skv, Hkv, dk = k.shape
        if Bk != B or dk != d or v.shape != k.shape:
            raise ValueError("shape mismatch between q, k and v")
        n = rows.shape[0]
        o = np.empty((n, d), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        sp = np.empty((n, d), dtype=np.float64) if vabs else None
        rc = self._lib.oracle_dense_rows(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Sq, Skv, Hq, Hkv, d, int(bool(causal)),
            float(scale), rows.ctypes.data, n, o.ctypes.data, lse.ctypes.data,
            sp.ctypes.data if vabs else None, threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_dense_rows failed with code {rc}")
        return (o, lse, sp) if vabs else (o, lse)

    def dense(self, q, k, v, causal, scale, threads=None, vabs=False):
        """All rows: returns (o [B, Sq, Hq, d], lse [B, Sq, Hq]) in fp64, and the weighted
        mean |V| [B, Sq, Hq, d] when asked."""
        B, Sq, Hq, d = q.shape
        b, i, h = np.meshgrid(np.arange(B), np.arange(Sq), np.arange(Hq), indexing="ij")
        rows = np.stack([b.ravel(), i.ravel(), h.ravel()], axis=1)
        r = self.dense_rows(q, k, v, causal, scale, rows, threads, vabs)
        out = (r[0].reshape(B, Sq, Hq, d), r[1].reshape(B, Sq, Hq))
        return out + (r[2].reshape(B, Sq, Hq, d),) if vabs else out

    # ------------------------------------------------------------------ paged
    def paged_rows(self, q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, causal, scale, rows,
                   threads=None, vabs=False):
        """Attention for selected (token, head) rows of the paged, ragged layout.

        q: uint16 [total_q, Hq, d]; k_pages, v_pages: uint16 [num_pages, page_size, Hkv, d];
        page_table: int32 [num_seqs, max_pages_per_seq]; cu_seqlens_q: int32 [num_seqs + 1];
        kv_lens: int32 [num_seqs]; rows: int64 [n, 2] of (t, h). Returns (o [n, d], lse [n]),
        and the weighted mean |V| [n, d] when asked.
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
        v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
        page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        kv_lens = np.ascontiguousarray(kv_lens, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
        total_q, Hq, d = q.shape
        num_pages, page_size, Hkv, dk = k_pages.shape
        num_seqs, max_pages = page_table.shape
        if dk != d or v_pages.shape != k_pages.shape or cu.shape[0] != num_seqs + 1:
            raise ValueError("shape mismatch in paged inputs")
        n = rows.shape[0]
        o = np.empty((n, d), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        sp = np.empty((n, d), dtype=np.float64) if vabs else None
        rc = self._lib.oracle_paged_rows(
            q.ctypes.data, k_pages.ctypes.data, v_pages.ctypes.data, page_table.ctypes.data,
            cu.ctypes.data, kv_lens.ctypes.data, page_size, num_seqs, max_pages, num_pages, Hq, Hkv,
            d, int(bool(causal)), float(scale), rows.ctypes.data, n, o.ctypes.data,
            lse.ctypes.data, sp.ctypes.data if vabs else None, threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_paged_rows failed with code {rc}")
        return (o, lse, sp) if vabs else (o, lse)

    def paged(self, q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, causal, scale,
              threads=None, vabs=False):
        """All rows: returns (o [total_q, Hq, d], lse [total_q, Hq]) in fp64, and the weighted
        mean |V| [total_q, Hq, d] when asked."""
        total_q, Hq, d = q.shape
        t, h = np.meshgrid(np.arange(total_q), np.arange(Hq), indexing="ij")
        rows = np.stack([t.ravel(), h.ravel()], axis=1)
        r = self.paged_rows(q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, causal,
                            scale, rows, threads, vabs)
        out = (r[0].reshape(total_q, Hq, d), r[1].reshape(total_q, Hq))
        return out + (r[2].reshape(total_q, Hq, d),) if vabs else out


_DEFAULT = None


def get() -> Oracle:
    """The oracle built from this package's own source (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
