"""The paged work list, read back from the workspace after a call, against a numpy restatement of
its definition. Sequences are ordered by key-tile count, longest first, with equal counts in index
order (a stable sort). Each sequence's (sequence, tile-pair) items are contiguous, heaviest tile
pair first under causal masking. Both planner forms are covered: one sequence per thread (up to
1024 sequences) and the chunked form for larger batches. The layout read here is the library's
internal one: the item count at byte 0, then int2 items from byte 256."""
import math

import numpy as np
import pytest

from tests.helpers import i32_dev, to_dev
from tests.test_parity_paged import build_case

pytestmark = pytest.mark.gpu


def expected_work(kv_lens, q_lens, pack, causal, max_pages_per_seq, page_size):
    max_kv_tiles = (max_pages_per_seq * page_size + 127) // 128
    buckets = min(max_kv_tiles, 8192)
    cost = np.minimum((np.asarray(kv_lens) + 127) // 128, buckets)
    order = np.argsort(-cost, kind="stable")
    work = []
    for s in order:
        q = int(q_lens[s])
        n = (q * pack + 255) // 256 if q > 0 else 0
        work += [(int(s), n - 1 - it if causal else it) for it in range(n)]
    return work


@pytest.mark.parametrize("n_seqs,causal,decode", [(700, True, False), (700, False, False), (3000, True, False),
                                                  (2500, True, True)])
def test_work_list_order(n_seqs, causal, decode):
    import torch

    import io_aware_exact_flash_gb300 as fa

    rng = np.random.default_rng(400 + n_seqs)
    lengths = rng.integers(0, 1200, size=n_seqs)
    lengths[rng.random(n_seqs) < 0.3] = 384  # many equal counts: the sort must keep index order
    lengths = lengths.tolist()
    q_lens = None if decode else [min(L, int(rng.integers(1, 300))) for L in lengths]
    t = build_case(lengths, 8, 2, 64, 16, decode, 401, q_lens=q_lens, poison=False)
    max_q = max(1, int(t["q_lens"].max()))
    num_pages, page_size = t["k_pages"].shape[:2]
    need = fa.fa_paged_workspace_bytes(n_seqs, int(t["total_q"]), max_q, page_size, t["page_table"].shape[1],
                                       num_pages, 8, 2, 64, 1)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    fa.fa_paged_fwd(to_dev(t["q"]), to_dev(t["k_pages"]), to_dev(t["v_pages"]), i32_dev(t["page_table"]),
                    i32_dev(t["cu_seqlens_q"]), i32_dev(t["kv_lens"]), max_q_len=max_q, causal=causal,
                    scale=1 / math.sqrt(64), workspace=ws, num_splits=1)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (0, 0)
    raw = ws.cpu().numpy()
    count = int(raw[:4].view(np.int32)[0])
    items = raw[256:256 + 8 * count].view(np.int32).reshape(-1, 2)
    pack = 4  # group 4 packs
    want = expected_work(t["kv_lens"], t["q_lens"], pack, causal, t["page_table"].shape[1], page_size)
    assert count == len(want)
    assert [tuple(x) for x in items.tolist()] == want
