"""Thin Python binding over the C ABI in ``include/fa.h`` (library ``libfa_gb300.so``).

Every function here only marshals arguments: it checks tensor dtypes, devices and shapes,
allocates outputs with torch when the caller passes none (on the stream the call runs on), and
forwards raw device pointers and the given (or current) CUDA stream to the C entry point of the
same name. All attention arithmetic runs in
the library's sm_103a kernels; there is no other path. If the library is missing, loading fails
with an error that says so.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

import torch

from .buildlib import LIBRARY

FA_OK = 0
_STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
    4: "FA_ERR_WORKSPACE", 5: "FA_ERR_CUDA", 6: "FA_ERR_NO_DEVICE", 7: "FA_ERR_DEVICE_TIMEOUT",
    8: "FA_ERR_DEVICE_BAD_PAGE",
}

EXPORTED = ("fa_status_string", "fa_fwd", "fa_paged_fwd", "fa_paged_workspace_bytes",
            "fa_decode_num_splits", "fa_merge_states", "fa_get_device_status", "fa_paged_decode_noalloc",
            "fa_selftest_wait_timeout", "fa_paged_append", "fa_cascade_fwd", "fa_cascade_workspace_bytes",
            "fa_paged_num_splits")


class FaError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {_STATUS_NAMES.get(code, code)}")


_lib = None


def load_library(path: str = None) -> ctypes.CDLL:
    """Load (once) the compiled library and declare its C signatures. The path defaults to the
    in-tree build; the environment variable FA_GB300_LIBRARY selects another build of it."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = os.environ.get("FA_GB300_LIBRARY", LIBRARY)
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA extension not built: {path} is missing (run __graft_entry__.build() or "
            "python -m io_aware_exact_flash_gb300.buildlib)")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, i, f, vp, vp, vp, sz, i, vp]
    lib.fa_paged_fwd.restype = i
    lib.fa_paged_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i, i]
    lib.fa_paged_workspace_bytes.restype = sz
    lib.fa_paged_num_splits.argtypes = [i] * 9
    lib.fa_paged_num_splits.restype = i
    lib.fa_decode_num_splits.argtypes = [i, i, i, i, i]
    lib.fa_decode_num_splits.restype = i
    lib.fa_merge_states.argtypes = [vp, vp, i, i, i, i, vp, vp, vp]
    lib.fa_merge_states.restype = i
    lib.fa_paged_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, vp, i, vp]
    lib.fa_paged_decode_noalloc.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [i, ctypes.POINTER(i), ctypes.POINTER(i), vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_cascade_workspace_bytes.argtypes = [i] * 12
    lib.fa_cascade_workspace_bytes.restype = sz
    lib.fa_cascade_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, i, i, i, vp, vp, vp, i, i, i, i, vp,
                                   vp, vp, sz, vp]
    lib.fa_cascade_fwd.restype = i
    lib.fa_paged_append.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp]
    lib.fa_paged_append.restype = i
    lib.fa_get_device_status.argtypes = [vp, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.fa_get_device_status.restype = i
    _lib = lib
    return lib


def _check(fn: str, code: int):
    if code != FA_OK:
        raise FaError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _on(stream):
    """Tensors a call allocates (outputs, workspace) belong to the stream the call runs on, so
    the caching allocator does not hand their memory to other work while the call's kernels
    still use it (a workspace is released as soon as the call returns)."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _bf16_cuda(name, t, dim):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if t.dim() != dim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dim}-D tensor")


def _i32_cuda(name, t):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")


def _check_outputs(out, lse, o_shape, like, out_dtype=torch.bfloat16):
    """A caller-given output must have exactly the shape, dtype and device the kernels write: a
    smaller buffer would be written past its end."""
    if out is not None:
        if (not isinstance(out, torch.Tensor) or out.dtype != out_dtype or out.device != like.device
                or tuple(out.shape) != tuple(o_shape) or not out.is_contiguous()):
            raise ValueError(f"out must be a contiguous {out_dtype} tensor of shape {tuple(o_shape)} on {like.device}")
    if lse is not None:
        l_shape = tuple(o_shape[:-1])
        if (not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32 or lse.device != like.device
                or tuple(lse.shape) != l_shape or not lse.is_contiguous()):
            raise ValueError(f"lse must be a contiguous float32 tensor of shape {l_shape} on {like.device}")


def fa_fwd(q, k, v, causal=False, scale=None, out=None, lse=None, return_lse=True, stream=None):
    """Dense attention forward. q: [B, S, Hq, d]; k, v: [B, S, Hkv, d] (bf16, CUDA).

    Returns (o [B, S, Hq, d] bf16, lse [B, S, Hq] fp32 or None)."""
    _bf16_cuda("q", q, 4)
    _bf16_cuda("k", k, 4)
    _bf16_cuda("v", v, 4)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, S, Hkv, d] matching q")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check_outputs(out, lse, q.shape, q)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty((B, S, Hq), dtype=torch.float32, device=q.device)
    lib = load_library()
    code = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, d, int(bool(causal)), scale,
                      _stream(stream))
    _check("fa_fwd", code)
    return out, lse


def fa_paged_workspace_bytes(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d,
                             num_splits=0):
    return int(load_library().fa_paged_workspace_bytes(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq,
                                                       num_pages, Hq, Hkv, d, num_splits))


def fa_paged_num_splits(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d):
    """Key splits fa_paged_fwd plans for these sizes with num_splits = 0 (1 = no split)."""
    return load_library().fa_paged_num_splits(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages,
                                              Hq, Hkv, d)


def fa_decode_num_splits(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv):
    return int(load_library().fa_decode_num_splits(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv))


def fa_paged_fwd(q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, max_q_len, causal=True, scale=None,
                 out=None, lse=None, return_lse=True, workspace=None, num_splits=0, stream=None):
    """Paged, ragged attention forward.

    q: [total_q, Hq, d]; k_pages, v_pages: [num_pages, page_size, Hkv, d] (bf16, CUDA);
    page_table: [num_seqs, max_pages_per_seq], cu_seqlens_q: [num_seqs + 1], kv_lens: [num_seqs]
    (int32, CUDA). max_q_len is a host-side int. Returns (o, lse)."""
    _bf16_cuda("q", q, 3)
    _bf16_cuda("k_pages", k_pages, 4)
    _bf16_cuda("v_pages", v_pages, 4)
    for name, t in (("page_table", page_table), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens)):
        _i32_cuda(name, t)
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_pages.shape
    num_seqs, max_pages = page_table.shape
    if dk != d or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check_outputs(out, lse, q.shape, q)
    need = fa_paged_workspace_bytes(num_seqs, total_q, max_q_len, page_size, max_pages, num_pages, Hq, Hkv, d,
                                    num_splits)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load_library()
    code = lib.fa_paged_fwd(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(cu_seqlens_q),
                            _ptr(kv_lens), num_seqs, total_q, int(max_q_len), page_size, max_pages, num_pages, Hq,
                            Hkv, d, int(bool(causal)), scale, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                            int(num_splits), _stream(stream))
    _check("fa_paged_fwd", code)
    return out, lse


def fa_merge_states(o_parts, lse_parts, out=None, lse=None, return_lse=True, stream=None):
    """Merge partial states: o_parts [P, n, H, d] fp32, lse_parts [P, n, H] fp32 (natural log)."""
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32 or not o_parts.is_cuda:
        raise TypeError("o_parts and lse_parts must be CUDA float32 tensors")
    if not (o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous")
    P, n, H, d = o_parts.shape
    if lse_parts.shape != (P, n, H):
        raise ValueError("lse_parts must be [P, n, H]")
    _check_outputs(out, lse, (n, H, d), o_parts)
    with _on(stream):
        if out is None:
            out = torch.empty((n, H, d), dtype=torch.bfloat16, device=o_parts.device)
        if lse is None and return_lse:
            lse = torch.empty((n, H), dtype=torch.float32, device=o_parts.device)
    code = load_library().fa_merge_states(_ptr(o_parts), _ptr(lse_parts), P, n, H, d, _ptr(out), _ptr(lse),
                                          _stream(stream))
    _check("fa_merge_states", code)
    return out, lse


def fa_cascade_fwd(q, k_pages, v_pages, cu_q_groups, prefix_page_table, prefix_lens, max_group_q_len,
                   cu_seqlens_q, page_table, kv_lens, max_q_len, causal=True, scale=None, out=None, lse=None,
                   return_lse=True, workspace=None, stream=None):
    """Shared-prefix (cascade) attention. Group g of consecutive sequences owns query rows
    [cu_q_groups[g], cu_q_groups[g+1]) and shares prefix_lens[g] keys in prefix_page_table[g];
    sequence s adds kv_lens[s] keys of its own in page_table[s]. The result equals fa_paged_fwd over
    each sequence's prefix ++ suffix keys. Index arrays are int32 CUDA tensors; max_group_q_len and
    max_q_len are host-side ints. Returns (o, lse)."""
    _bf16_cuda("q", q, 3)
    _bf16_cuda("k_pages", k_pages, 4)
    _bf16_cuda("v_pages", v_pages, 4)
    for name, t in (("cu_q_groups", cu_q_groups), ("prefix_page_table", prefix_page_table),
                    ("prefix_lens", prefix_lens), ("cu_seqlens_q", cu_seqlens_q), ("page_table", page_table),
                    ("kv_lens", kv_lens)):
        _i32_cuda(name, t)
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_pages.shape
    num_groups, max_prefix_pages = prefix_page_table.shape
    num_seqs, max_pages = page_table.shape
    if dk != d or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d]")
    if cu_q_groups.shape != (num_groups + 1,) or prefix_lens.shape != (num_groups,):
        raise ValueError("cu_q_groups must be [num_groups + 1] and prefix_lens [num_groups]")
    _check_outputs(out, lse, q.shape, q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = load_library()
    need = lib.fa_cascade_workspace_bytes(num_groups, num_seqs, total_q, int(max_group_q_len), int(max_q_len),
                                          page_size, max_prefix_pages, max_pages, num_pages, Hq, Hkv, d)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    code = lib.fa_cascade_fwd(_ptr(q), _ptr(k_pages), _ptr(v_pages), page_size, num_pages, Hq, Hkv, d, scale,
                              num_groups, _ptr(cu_q_groups), _ptr(prefix_page_table), _ptr(prefix_lens),
                              max_prefix_pages, int(max_group_q_len), num_seqs, _ptr(cu_seqlens_q), _ptr(page_table),
                              _ptr(kv_lens), max_pages, int(max_q_len), int(bool(causal)), total_q, _ptr(out),
                              _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream))
    _check("fa_cascade_fwd", code)
    return out, lse


def fa_cascade_workspace_bytes(num_groups, num_seqs, total_q, max_group_q_len, max_q_len, page_size,
                               max_prefix_pages, max_pages_per_seq, num_pages, Hq, Hkv, d):
    return load_library().fa_cascade_workspace_bytes(num_groups, num_seqs, total_q, max_group_q_len, max_q_len,
                                                     page_size, max_prefix_pages, max_pages_per_seq, num_pages, Hq,
                                                     Hkv, d)


def fa_paged_append(k_new, v_new, cu_seqlens_new, kv_lens_before, page_table, k_pages, v_pages, stream=None):
    """Write new tokens' K/V rows ([total_new, Hkv, d] bf16) into their page slots, in place.

    New row r of sequence s goes to logical position kv_lens_before[s] + r of that sequence, i.e.
    page page_table[s][pos // page_size], slot pos % page_size. cu_seqlens_new ([num_seqs + 1]),
    kv_lens_before ([num_seqs]) and page_table ([num_seqs, max_pages_per_seq]) are int32 CUDA
    tensors; kv_lens_before is not updated. Returns None."""
    _bf16_cuda("k_new", k_new, 3)
    _bf16_cuda("v_new", v_new, 3)
    _bf16_cuda("k_pages", k_pages, 4)
    _bf16_cuda("v_pages", v_pages, 4)
    for name, t in (("cu_seqlens_new", cu_seqlens_new), ("kv_lens_before", kv_lens_before),
                    ("page_table", page_table)):
        _i32_cuda(name, t)
    total_new, Hkv, d = k_new.shape
    num_pages, page_size, Hkv_p, d_p = k_pages.shape
    num_seqs, max_pages = page_table.shape
    if v_new.shape != k_new.shape or v_pages.shape != k_pages.shape or (Hkv_p, d_p) != (Hkv, d):
        raise ValueError("k_new/v_new must be [total_new, Hkv, d] and the pages [num_pages, page_size, Hkv, d]")
    if cu_seqlens_new.shape != (num_seqs + 1,) or kv_lens_before.shape != (num_seqs,):
        raise ValueError("cu_seqlens_new must be [num_seqs + 1] and kv_lens_before [num_seqs]")
    code = load_library().fa_paged_append(_ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_new), _ptr(kv_lens_before),
                                          _ptr(page_table), num_seqs, total_new, page_size, max_pages, num_pages,
                                          Hkv, d, _ptr(k_pages), _ptr(v_pages), _stream(stream))
    _check("fa_paged_append", code)


def fa_get_device_status(stream=None):
    """Returns (code, site) of this GPU's device status word and clears it (synchronises)."""
    code, site = ctypes.c_int(0), ctypes.c_int(0)
    _check("fa_get_device_status",
           load_library().fa_get_device_status(_stream(stream), ctypes.byref(code), ctypes.byref(site)))
    return code.value, site.value


def status_string(code: int) -> str:
    return load_library().fa_status_string(code).decode()


def fa_paged_decode_noalloc(q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, out, lse=None, scale=None,
                            num_splits=0, stream=None):
    """Split-KV decode that uses the library's fixed device scratch instead of a workspace, for
    callers that cannot allocate device memory. Nothing is allocated here either: the caller
    passes `out` ([total_q, Hq, d] bf16) and, optionally, `lse` ([total_q, Hq] fp32)."""
    _bf16_cuda("q", q, 3)
    _bf16_cuda("k_pages", k_pages, 4)
    _bf16_cuda("v_pages", v_pages, 4)
    _bf16_cuda("out", out, 3)
    for name, t in (("page_table", page_table), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens)):
        _i32_cuda(name, t)
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_pages.shape
    num_seqs, max_pages = page_table.shape
    if dk != d or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d]")
    _check_outputs(out, lse, q.shape, q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code = load_library().fa_paged_decode_noalloc(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(cu_seqlens_q), _ptr(kv_lens), num_seqs,
        total_q, page_size, max_pages, num_pages, Hq, Hkv, d, scale, _ptr(out), _ptr(lse), int(num_splits),
        _stream(stream))
    _check("fa_paged_decode_noalloc", code)
    return out, lse


def fa_selftest_wait_timeout(limit_ms=50, stream=None):
    """Runs the device-side timeout diagnostic; returns (code, site) the status word recorded."""
    code, site = ctypes.c_int(0), ctypes.c_int(0)
    _check("fa_selftest_wait_timeout",
           load_library().fa_selftest_wait_timeout(int(limit_ms), ctypes.byref(code), ctypes.byref(site),
                                                   _stream(stream)))
    return code.value, site.value
