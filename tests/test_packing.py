"""Path choices of the paged entry point, forced both ways for the whole paged and cascade parity
suites (their smaller cases), so every shape there is checked against the oracle on each path:
GQA packing of the tensor-core path (a tile's rows = token x head of one kv head's query heads)
on and off, and decode batches on the split-KV CUDA-core kernel instead of the tensor cores."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("env", [{"FA_PAGED_PACK": "1"}, {"FA_PAGED_PACK": "0"}, {"FA_DECODE_TC": "0"}],
                         ids=["always_pack", "never_pack", "decode_on_cuda_cores"])
def test_paged_parity_with_forced_paths(env):
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not full_size",
                        "-p", "no:cacheprovider", "tests/test_parity_paged.py", "tests/test_cascade.py"],
                       env=dict(os.environ, **env), cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
