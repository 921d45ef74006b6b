"""Calls from several host threads at once, each on its own CUDA stream (the C ABI promises
reentrant calls; ctypes releases the GIL during each call). Every thread runs dense and paged
forwards from a fresh process state, so the first-call set-up (device probe, kernel attribute
caches) also races; results must equal those of the same calls made one at a time, bit for bit
(the kernels are deterministic), and the device status word must stay clear."""
import math
import threading

import numpy as np
import pytest

from io_aware_exact_flash_gb300.workloads import normal_bf16
from tests.helpers import i32_dev, to_dev
from tests.test_parity_paged import build_case

pytestmark = pytest.mark.gpu

N_THREADS = 4


def _inputs(i):
    q = to_dev(normal_bf16(900 + i, (1, 700, 8, 128), stream=0))
    k = to_dev(normal_bf16(900 + i, (1, 700, 2, 128), stream=1))
    v = to_dev(normal_bf16(900 + i, (1, 700, 2, 128), stream=2))
    t = build_case([300, 1, 900, 57], 8, 2, 128, 16, i % 2 == 1, 950 + i, poison=False)
    paged = (to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"]), i32_dev(t["page_table"]),
             i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"]), int(t["q_lens"].max()))
    return (q, k, v), paged


def _run(fa, dense, paged, stream):
    import torch

    q, k, v = dense
    o1, l1 = fa.fa_fwd(q, k, v, causal=True, scale=1 / math.sqrt(128), stream=stream)
    o2, l2 = fa.fa_paged_fwd(*paged[:6], max_q_len=paged[6], causal=True, scale=0.09, stream=stream)
    stream.synchronize()
    return [t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
            for t in (o1, l1, o2, l2)]


def concurrent_then_serial():
    """Runs in a fresh process: the threads' first calls are the process's first library calls."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    inputs = [_inputs(i) for i in range(N_THREADS)]
    streams = [torch.cuda.Stream() for _ in range(N_THREADS)]
    results = [None] * N_THREADS
    errors = []
    start = threading.Barrier(N_THREADS)

    def worker(i):
        try:
            start.wait()
            out = None
            for _ in range(5):
                out = _run(fa, *inputs[i], streams[i])
            results[i] = out
        except Exception as e:  # reported below, in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(N_THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert fa.fa_get_device_status() == (0, 0)
    for i in range(N_THREADS):
        serial = _run(fa, *inputs[i], streams[0])
        for a, b in zip(results[i], serial):
            assert np.array_equal(a, b), f"thread {i}: a concurrent result differs from the serial one"


def test_concurrent_calls_match_serial_calls():
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", "from tests.test_threads import concurrent_then_serial as f; f()"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
