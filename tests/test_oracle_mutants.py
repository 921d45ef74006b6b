"""Plant plausible mistakes in a copy of the oracle's C source and check that the pins catch
every one of them (CPU only; the real oracle file is never modified)."""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import oracle_pins

# (name, text in the oracle source, replacement): each is a mistake a careful reader could make
MUTANTS = [
    ("dropped_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("wrong_exp_sign", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("lse_without_max", "*lse = m + log(sum);", "*lse = log(sum);"),
    ("causal_off_by_one", "long n = i + (kv_len - q_len) + 1;", "long n = i + (kv_len - q_len);"),
    ("top_left_causal", "long n = i + (kv_len - q_len) + 1;", "long n = i + 1;"),
    ("gqa_modulo_map", "const int64_t hk = h / group;", "const int64_t hk = h % J->Hkv;"),
    ("values_from_keys", "V[j * d + c] = bf16_to_double(J->v[at]);", "V[j * d + c] = bf16_to_double(J->k[at]);"),
    ("reversed_feature_index", "acc += q[c] * K[j * d + c];", "acc += q[c] * K[j * d + (d - 1 - c)];"),
    ("wrong_page_slot", "const long slot = j % J->page_size;", "const long slot = (j + 1) % J->page_size;"),
    ("unnormalised_p", "double p = s[j] / sum;", "double p = s[j];"),
    ("max_not_updated", "if (s[j] > m) m = s[j];", "if (s[j] > m) m = m;"),
    ("vabs_without_abs", "vabs[c] += p * fabs(V[j * d + c]);", "vabs[c] += p * V[j * d + c];"),
    ("vabs_unweighted", "vabs[c] += p * fabs(V[j * d + c]);", "vabs[c] += fabs(V[j * d + c]);"),
    ("vabs_centered_on_o", "vabs[c] += p * fabs(V[j * d + c]);", "vabs[c] += p * fabs(V[j * d + c] - o[c]);"),
]


def _count(text, needle):
    return text.count(needle)


@pytest.fixture(scope="module")
def source_text():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, source_text, name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    assert _count(source_text, old) >= 1, f"mutation site for {name} not found in the oracle source"
    src = tmp_path / f"{name}.c"
    src.write_text(source_text.replace(old, new))
    lib = oracle.compile_library(str(src), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
