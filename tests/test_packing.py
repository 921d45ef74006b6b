"""Path choices of the entry points, forced the other way for the parity suites (their smaller
cases), so every shape there is checked against the oracle on each path: GQA packing of the
tensor-core path (a tile's rows = token x head of one kv head's query heads) off, decode batches
on the split-KV CUDA-core kernel instead of the tensor cores, decode and verify batches on the
packed prefill kernel instead of the key-row kernel, and the prefill launch modes. The seeded random shapes of test_fuzz.py run
under each of them too (the default paths run in the suites themselves)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("env", [{"FA_PAGED_PACK": "0"}, {"FA_DECODE_TC": "0"}, {"FA_DECODE_KEY_ROWS": "0"}],
                         ids=["never_pack", "decode_on_cuda_cores", "decode_on_packed_tiles"])
def test_paged_parity_with_forced_paths(env):
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not full_size",
                        "-p", "no:cacheprovider", "tests/test_parity_paged.py", "tests/test_cascade.py",
                        "tests/test_fuzz.py"],
                       env=dict(os.environ, **env), cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


@pytest.mark.parametrize("env", [{"FA_PREFILL_TAKE_OVER": "0"}, {"FA_PREFILL_PERSISTENT": "1"},
                                 {"FA_PREFILL_PERSISTENT": "0"}],
                         ids=["no_take_over", "persistent", "one_cta_per_unit"])
def test_launch_modes(env):
    """The prefill launch modes other than the default take-over: dense CTAs that exit after their
    own item with a persistent paged grid, a persistent grid everywhere, and one CTA per unit.
    Each runs the dense, paged, cascade and random-shape parity suites (their smaller cases)."""
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not full_size",
                        "-p", "no:cacheprovider", "tests/test_parity_dense.py", "tests/test_parity_paged.py",
                        "tests/test_cascade.py", "tests/test_fuzz.py"],
                       env=dict(os.environ, **env), cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
