"""C-ABI checks that need no GPU: the library loads, exports every function include/fa.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from io_aware_exact_flash_gb300 import buildlib

    if not os.path.exists(buildlib.LIBRARY):
        if shutil.which(buildlib.NVCC) is None and not os.path.exists(buildlib.NVCC):
            pytest.skip("nvcc not available to build the library")
        buildlib.build()
    from io_aware_exact_flash_gb300 import binding

    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_paged_fwd", "fa_paged_workspace_bytes", "fa_merge_states", "fa_get_device_status",
              "fa_status_string", "fa_decode_num_splits"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from io_aware_exact_flash_gb300 import binding

    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fa.h but not exported"
    assert set(binding.EXPORTED) == set(names)


def test_status_strings(lib):
    from io_aware_exact_flash_gb300 import binding

    for code, name in binding._STATUS_NAMES.items():
        assert binding.status_string(code) == name


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced: validation fails first


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=2, S=128, d=128, causal=1, scale=0.1):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse) if lse else None, B, Hq, Hkv, S, d, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(o=0), 1), (dict(B=0), 1), (dict(S=-1), 1), (dict(Hq=3, Hkv=2), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=-1.0), 1),
    (dict(d=96), 2), (dict(d=256), 2),
    (dict(q=FAKE + 8), 3), (dict(v=FAKE + 2), 3), (dict(lse=FAKE + 2), 3),
    (dict(B=1 << 12, S=1 << 20), 2),  # B * S rows past 2^31 - 1
    (dict(B=1 << 10, S=1 << 20, Hq=1 << 10, Hkv=1 << 10), 2),  # elements past 2^40
])
def test_fa_fwd_host_validation(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _paged(lib, **kw):
    a = dict(q=FAKE, kp=FAKE, vp_=FAKE, pt=FAKE, cu=FAKE, kl=FAKE, num_seqs=2, total_q=10, max_q_len=5, ps=16,
             max_pages=4, num_pages=8, Hq=4, Hkv=2, d=128, causal=1, scale=0.1, o=FAKE, lse=None, ws=None, wsb=0,
             splits=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.fa_paged_fwd(vp(a["q"]), vp(a["kp"]), vp(a["vp_"]), vp(a["pt"]), vp(a["cu"]), vp(a["kl"]),
                            a["num_seqs"], a["total_q"], a["max_q_len"], a["ps"], a["max_pages"], a["num_pages"],
                            a["Hq"], a["Hkv"], a["d"], a["causal"], a["scale"], vp(a["o"]),
                            vp(a["lse"]) if a["lse"] else None, vp(a["ws"]) if a["ws"] else None, a["wsb"],
                            a["splits"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(pt=0), 1), (dict(cu=0), 1), (dict(num_seqs=0), 1), (dict(max_q_len=0), 1), (dict(Hq=3), 1),
    (dict(num_pages=0), 1), (dict(splits=-1), 1),
    (dict(ps=8), 2), (dict(ps=48), 2), (dict(d=80), 2),
    (dict(kp=FAKE + 4), 3), (dict(cu=FAKE + 2), 3),
    (dict(max_pages=1 << 26, ps=32), 2),   # a sequence past 2^30 keys
    (dict(num_pages=1 << 27, ps=32), 2),   # a pool past 2^31 - 1 rows
])
def test_fa_paged_fwd_host_validation(lib, kw, code):
    assert _paged(lib, **kw) == code


def test_workspace_query_is_host_only(lib):
    from io_aware_exact_flash_gb300 import binding

    n_prefill = binding.fa_paged_workspace_bytes(64, 300000, 8192, 16, 512, 20000, 32, 8, 128)
    assert n_prefill >= 8 * (300000 // 256 + 64)
    # decode with a GQA group of 4 runs on the tensor-core path: a work list, plus fp32 partial
    # states when the keys are split
    n1 = binding.fa_paged_workspace_bytes(64, 64, 1, 16, 512, 20000, 32, 8, 128, num_splits=1)
    assert 0 < n1 < 64 * 32 * 128 * 4
    n4 = binding.fa_paged_workspace_bytes(64, 64, 1, 16, 512, 20000, 32, 8, 128, num_splits=4)
    assert n4 >= n1 + 4 * 64 * 32 * (128 + 1) * 4
    # MHA decode runs there too (one real row per tile)
    assert binding.fa_paged_workspace_bytes(64, 64, 1, 16, 512, 20000, 8, 8, 128, num_splits=1) > 0


def test_workspace_of_cuda_core_decode():
    """With FA_DECODE_TC=0 decode batches of groups 1/2/4/8 run on the split-KV CUDA-core kernel:
    one split needs no workspace, more need the partials (the switch is read once per process)."""
    import subprocess
    import sys

    code = ("from io_aware_exact_flash_gb300 import binding as b\n"
            "print(b.fa_paged_workspace_bytes(64, 64, 1, 16, 512, 20000, 8, 8, 128, num_splits=1),"
            " b.fa_paged_workspace_bytes(64, 64, 1, 16, 512, 20000, 8, 8, 128, num_splits=4))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, FA_DECODE_TC="0"))
    assert r.returncode == 0, r.stderr
    n1, n4 = map(int, r.stdout.split())
    assert n1 == 0 and n4 >= 4 * 64 * 8 * (128 + 1) * 4


def test_merge_host_validation(lib):
    vp = ctypes.c_void_p
    assert lib.fa_merge_states(None, vp(FAKE), 2, 4, 8, 128, vp(FAKE), None, None) == 1
    assert lib.fa_merge_states(vp(FAKE), vp(FAKE), 0, 4, 8, 128, vp(FAKE), None, None) == 1
    assert lib.fa_merge_states(vp(FAKE), vp(FAKE), 2, 4, 8, 100, vp(FAKE), None, None) == 2
    assert lib.fa_merge_states(vp(FAKE + 4), vp(FAKE), 2, 4, 8, 128, vp(FAKE), None, None) == 3


def _append(lib, **kw):
    a = dict(kn=FAKE, vn=FAKE, cu=FAKE, kl=FAKE, pt=FAKE, num_seqs=2, total_new=10, ps=16, max_pages=4,
             num_pages=8, Hkv=2, d=128, kp=FAKE, vp_=FAKE)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.fa_paged_append(vp(a["kn"]), vp(a["vn"]), vp(a["cu"]), vp(a["kl"]), vp(a["pt"]), a["num_seqs"],
                               a["total_new"], a["ps"], a["max_pages"], a["num_pages"], a["Hkv"], a["d"],
                               vp(a["kp"]), vp(a["vp_"]), None)


@pytest.mark.parametrize("kw,code", [
    (dict(kn=0), 1), (dict(pt=0), 1), (dict(vp_=0), 1), (dict(num_seqs=0), 1), (dict(total_new=-1), 1),
    (dict(num_pages=0), 1), (dict(Hkv=0), 1), (dict(max_pages=0), 1),
    (dict(d=96), 2), (dict(ps=24), 2), (dict(ps=256), 2),
    (dict(kn=FAKE + 8), 3), (dict(kp=FAKE + 4), 3), (dict(cu=FAKE + 2), 3), (dict(kl=FAKE + 1), 3),
])
def test_fa_paged_append_host_validation(lib, kw, code):
    assert _append(lib, **kw) == code


def test_fa_paged_append_empty_rows_may_be_null(lib):
    # nothing to append: NULL row buffers pass validation (the call then needs a device)
    assert _append(lib, kn=0, vn=0, total_new=0) != 1
    assert _append(lib, kn=0, total_new=1) == 1


def test_key_split_plan_is_host_only():
    """The automatic key-split count (host planning, no GPU needed). A decode batch that fills
    the GPU three times over is not split. A small decode batch is split with at least 8 key tiles
    per split. A shared prefix read by 128 query rows (16 compute-bound units over 128 key tiles)
    gets the count that fits one wave of this part's SMs, not the three-wave count."""
    from io_aware_exact_flash_gb300 import binding

    big_decode = binding.fa_paged_num_splits(128, 128, 1, 16, 1024, 70000, 32, 8, 128)
    assert big_decode == 1
    small_decode = binding.fa_paged_num_splits(4, 4, 1, 16, 1024, 70000, 32, 8, 128)
    assert 2 <= small_decode <= (1024 * 16 // 128) // 8
    prefix = binding.fa_paged_num_splits(1, 128, 128, 16, 1024, 70000, 32, 8, 128)
    assert 2 <= prefix <= 16 and 16 * prefix <= 148  # one wave (148 or 152 SMs), each split >= 8 tiles
    # no split when a pass has more units than three waves, whatever the key length
    assert binding.fa_paged_num_splits(64, 64 * 512, 512, 16, 1024, 70000, 32, 8, 128) == 1


def _noalloc(lib, **kw):
    a = dict(q=FAKE, kp=FAKE, vp_=FAKE, pt=FAKE, cu=FAKE, kl=FAKE, num_seqs=4, total_q=4, ps=16, max_pages=64,
             num_pages=256, Hq=32, Hkv=8, d=128, scale=0.1, o=FAKE, lse=None, splits=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.fa_paged_decode_noalloc(vp(a["q"]), vp(a["kp"]), vp(a["vp_"]), vp(a["pt"]), vp(a["cu"]), vp(a["kl"]),
                                       a["num_seqs"], a["total_q"], a["ps"], a["max_pages"], a["num_pages"], a["Hq"],
                                       a["Hkv"], a["d"], a["scale"], vp(a["o"]), vp(a["lse"]) if a["lse"] else None,
                                       a["splits"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(num_seqs=0), 1), (dict(total_q=5), 1), (dict(Hq=12), 1), (dict(splits=-1), 1),
    (dict(num_seqs=70000, total_q=70000), 2), (dict(Hq=48, Hkv=3), 2), (dict(d=96), 2), (dict(ps=8), 2),
    (dict(o=FAKE + 8), 3),
    # 64 splits x 1024 sequences x 32 heads x 129 floats: far above the 16 MiB scratch
    (dict(num_seqs=1024, total_q=1024, splits=64), 4),
])
def test_fa_paged_decode_noalloc_host_validation(lib, kw, code):
    """Rows beyond one per sequence, grids the decode kernel cannot launch and split counts whose
    partials do not fit the fixed scratch are refused on the host, before anything is enqueued."""
    assert _noalloc(lib, **kw) == code


def test_fa_paged_decode_noalloc_caps_splits_before_the_scratch_check(lib):
    """64 splits of 4-page sequences are capped at 4, which fit (4 x 128 sequences x 32 heads x 129
    floats): validation passes (the call then needs a device, so on a machine without one it fails
    later, with another code). Uncapped, the same 64 splits would not fit."""
    assert _noalloc(lib, num_seqs=128, total_q=128, max_pages=64, splits=64) == 4
    assert _noalloc(lib, num_seqs=128, total_q=128, max_pages=4, splits=64) not in (1, 2, 3, 4)
