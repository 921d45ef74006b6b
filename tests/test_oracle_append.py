"""The paged KV append oracle against facts that do not depend on its own formula (CPU only):

* filling an empty cache and then attending through the page table (the attention oracle's own
  page addressing, itself pinned against the dense layout) equals dense attention over the new
  rows taken in order;
* appending in several steps (a prefill chunk, then single decode tokens, each step starting at
  the length the previous one left) equals appending everything at once;
* no slot outside the new rows' positions changes, and positions outside the table are refused.

Planted mistakes in a copy of the oracle's source must each fail at least one of these."""
import inspect
import types

import numpy as np
import pytest

import oracle
from oracle import kv_append

NAN_BITS = np.uint16(0x7FC0)


def _layout(seed, lengths, page_size, spare_pages=3):
    """Page table with a seeded permutation of physical pages (plus unreferenced spares)."""
    rng = np.random.default_rng(seed)
    npages = [(L + page_size - 1) // page_size for L in lengths]
    P = sum(npages) + spare_pages
    perm = rng.permutation(P).astype(np.int32)
    table = np.full((len(lengths), max(1, max(npages))), -1, np.int32)
    off = 0
    for s, n in enumerate(npages):
        table[s, :n] = perm[off:off + n]
        off += n
    return table, P


def _rows(seed, n, Hkv, d):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def pin_fill_then_attend(append):
    lengths, ps, Hkv, Hq, d = [1, 16, 17, 40, 5], 16, 2, 4, 8
    table, P = _layout(31, lengths, ps)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    k_new, v_new = _rows(1, int(cu[-1]), Hkv, d), _rows(2, int(cu[-1]), Hkv, d)
    empty = np.full((P, ps, Hkv, d), NAN_BITS, np.uint16)
    kp, vp = append(empty, empty, table, np.zeros(len(lengths), np.int32), cu, k_new, v_new)
    q = _rows(3, int(cu[-1]), Hq, d)
    orc = oracle.get()
    o, lse = orc.paged(q, kp, vp, table, cu, np.asarray(lengths, np.int32), True, 0.3, threads=2)
    for s in range(len(lengths)):
        sl = slice(cu[s], cu[s + 1])
        od, ld = orc.dense(q[sl][None], k_new[sl][None], v_new[sl][None], True, 0.3, threads=1)
        assert np.array_equal(o[sl], od[0]) and np.array_equal(lse[sl], ld[0]), f"sequence {s}"


def pin_steps_equal_once(append):
    ps, Hkv, d = 16, 2, 8
    final = [37, 16, 3, 64]
    table, P = _layout(32, final, ps)
    rng = np.random.default_rng(4)
    base_k = _rows(5, P * ps, Hkv, d).reshape(P, ps, Hkv, d)
    base_v = _rows(6, P * ps, Hkv, d).reshape(P, ps, Hkv, d)
    cu_all = np.concatenate([[0], np.cumsum(final)]).astype(np.int32)
    k_all, v_all = _rows(7, int(cu_all[-1]), Hkv, d), _rows(8, int(cu_all[-1]), Hkv, d)
    once_k, once_v = append(base_k, base_v, table, np.zeros(4, np.int32), cu_all, k_all, v_all)
    # steps: a prefill chunk of random size, then one token at a time
    done = np.asarray([rng.integers(0, L + 1) for L in final], np.int32)
    kk, vv = append(base_k, base_v, table, np.zeros(4, np.int32),
                    np.concatenate([[0], np.cumsum(done)]).astype(np.int32),
                    np.concatenate([k_all[cu_all[s]:cu_all[s] + done[s]] for s in range(4)]),
                    np.concatenate([v_all[cu_all[s]:cu_all[s] + done[s]] for s in range(4)]))
    while (done < final).any():
        n = (done < final).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        idx = [cu_all[s] + done[s] for s in range(4) if n[s]]
        kk, vv = append(kk, vv, table, done, cu, k_all[idx], v_all[idx])
        done = done + n
    assert np.array_equal(kk, once_k) and np.array_equal(vv, once_v)


def pin_untouched_slots_and_bounds(append):
    ps, Hkv, d = 16, 1, 8
    before = [5, 16, 0]
    new = [12, 1, 20]
    table, P = _layout(33, [b + n for b, n in zip(before, new)], ps)
    kp = _rows(9, P * ps, Hkv, d).reshape(P, ps, Hkv, d)
    vp = _rows(10, P * ps, Hkv, d).reshape(P, ps, Hkv, d)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    k_new = np.full((int(cu[-1]), Hkv, d), 0x3F80, np.uint16)  # 1.0, differs from every old value
    v_new = np.full((int(cu[-1]), Hkv, d), 0x4000, np.uint16)  # 2.0
    k2, v2 = append(kp, vp, table, np.asarray(before, np.int32), cu, k_new, v_new)
    changed_k = (k2 != kp).any(axis=(2, 3))
    changed_v = (v2 != vp).any(axis=(2, 3))
    expect = np.zeros((P, ps), bool)
    for s in range(3):
        for r in range(new[s]):
            pos = before[s] + r
            expect[table[s, pos // ps], pos % ps] = True
    assert int(expect.sum()) == sum(new)
    assert np.array_equal(changed_k, expect) and np.array_equal(changed_v, expect)
    assert (k2[expect] == 0x3F80).all() and (v2[expect] == 0x4000).all()
    try:  # one row past the table of sequence 1 must be refused
        append(kp, vp, table, np.asarray([0, table.shape[1] * ps, 0], np.int32),
               np.asarray([0, 0, 1, 1], np.int32), k_new[:1], v_new[:1])
    except ValueError:
        pass
    else:
        raise AssertionError("a position past the page table was accepted")


PINS = [pin_fill_then_attend, pin_steps_equal_once, pin_untouched_slots_and_bounds]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_append_pin(pin):
    pin(kv_append.paged_append)


MUTANTS = [
    ("one_past_length", "pos = int(kv_lens_before[s]) + (t - first)", "pos = int(kv_lens_before[s]) + (t - first) + 1"),
    ("ignores_cached_length", "pos = int(kv_lens_before[s]) + (t - first)", "pos = (t - first)"),
    ("global_row_index", "pos = int(kv_lens_before[s]) + (t - first)", "pos = int(kv_lens_before[s]) + t"),
    ("page_slot_swapped", "logical_page, slot = divmod(pos, page_size)", "slot, logical_page = divmod(pos, page_size)"),
    ("values_from_keys", "v_out[page, slot] = v_new[t]", "v_out[page, slot] = k_new[t]"),
    ("last_row_dropped", "for t in range(first, end):", "for t in range(first, end - 1):"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new):
    src = inspect.getsource(kv_append)
    assert src.count(old) == 1, f"mutation site for {name} not found"
    mod = types.ModuleType(f"kv_append_{name}")
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), mod.__dict__)
    caught = []
    for pin in PINS:
        try:
            pin(mod.paged_append)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
