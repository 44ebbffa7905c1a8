"""kvattn_combine (the split-KV log-sum-exp merge) against the oracle's merge.

The merge of split partials follows "MLA：为什么一份 Latent 可以代替多头 KV Cache",
section "FlashMLA 解决的不是模型公式本身" (each split's local max and normaliser,
then a stable merge); the oracle's lse_combine is pinned in test_oracle.py.
"""
import numpy as np
import pytest
import torch

import kv_cache_decode_paged_gb300 as kv

pytestmark = pytest.mark.gpu


def _case(rng, counts, rows, dv, empty_rows=()):
    """Partials of len(counts) units, unit u split counts[u] ways."""
    first = np.zeros(len(counts), dtype=np.int32)
    first[1:] = np.cumsum(counts)[:-1]
    n_slots = int(sum(counts))
    part_o = rng.standard_normal((max(n_slots, 1), rows, dv)).astype(np.float32)
    part_l = (rng.standard_normal((max(n_slots, 1), rows)) * 4.0).astype(np.float32)
    for slot, r in empty_rows:  # a split with no valid token for this row
        part_l[slot, r] = -np.inf
        part_o[slot, r] = 0.0
    return first, np.asarray(counts, dtype=np.int32), part_o, part_l


def _run(first, count, part_o, part_l, rows, dv):
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    n = len(count)
    out = torch.full((n, rows, dv), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((n, rows), float("nan"), dtype=torch.float32, device=dev)
    kv.kvattn_combine(t(part_o), t(part_l), t(first), t(count), rows, dv, out, lse)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("counts,rows,dv", [
    ([1, 2, 3, 0, 5], 8, 16),        # one split, several, none
    ([18] * 16, 32, 128),            # many splits per unit, GQA-like rows
    ([40, 1, 7], 128, 512),          # MLA-like rows
])
def test_combine_matches_oracle(oracle, counts, rows, dv):
    rng = np.random.default_rng(sum(counts) + rows + dv)
    empty = [(0, 1), (1, 0)] if sum(counts) > 1 else []
    first, count, part_o, part_l = _case(rng, counts, rows, dv, empty)
    out, lse = _run(first, count, part_o, part_l, rows, dv)
    for u, c in enumerate(counts):
        if c == 0:
            assert (out[u] == 0).all() and np.isneginf(lse[u]).all()
            continue
        sl = slice(first[u], first[u] + c)
        want_o, want_l = oracle.lse_combine(part_o[sl], part_l[sl])
        np.testing.assert_allclose(out[u], want_o, rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(lse[u], want_l, rtol=1e-5, atol=1e-5)


def test_combine_all_splits_empty_row(oracle):
    # every split of unit 0 has no valid token for row 2: zeros and -inf
    rng = np.random.default_rng(7)
    first, count, part_o, part_l = _case(rng, [3, 2], 4, 8, [(0, 2), (1, 2), (2, 2)])
    out, lse = _run(first, count, part_o, part_l, 4, 8)
    assert (out[0, 2] == 0).all() and np.isneginf(lse[0, 2])
    want_o, want_l = oracle.lse_combine(part_o[3:5], part_l[3:5])
    np.testing.assert_allclose(out[1], want_o, rtol=1e-4, atol=1e-5)
