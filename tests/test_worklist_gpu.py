"""The tensor-core attention's work list, built on the device and read back (test aid).

Checked against what the list must be, from the lengths alone (DFlash KV Injection
Walkthrough, Step 7: the cache grows by the injected context rows, then the block follows
them; a query sees the whole prefix or, under a sliding window of W, the last W positions):
every (sequence, KV head) key range is covered once, in order, by items of whole 128-key
tiles, cut into no more than max_splits pieces; each CTA's items are a contiguous run of the
list; the pairs the combine writes are exactly the split and the refused ones; and the
CTAs' costs (8 per tile plus item_cost per item) stay within a tile and two item headers of
an equal share.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_dflash_gb300 import dflash as D

pytestmark = pytest.mark.gpu

TK = 128
TILE_COST = 8


def _case(batch, n_kv, capacity, lens, counts, window=0, paged=False, bs=16, n_h=None):
    n_h = n_h or 4 * n_kv
    dims = D.make_dims(256, n_h, n_kv, 128, 1, bs, 1e-6, "bf16")
    cache = D.KVCache(1, batch, n_kv, capacity, 128, "bf16", "cuda", paged=paged, seed=1)
    cache.lens.copy_(torch.tensor(np.asarray(lens, np.int32)[None, :], device="cuda"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    M = int(np.sum(counts))
    ws = torch.empty(D.dflash_workspace_bytes(dims, batch, capacity, max(M, batch * bs, 1)),
                     dtype=torch.uint8, device="cuda")
    wl = D.dflash_test_attn_worklist(dims, cache, 0, cu, M, window, ws)
    return dims, wl


def _expected_ranges(lens, counts, capacity, bs, window, n_kv, align):
    """Per pair (sequence-major): (lo, end) of its keys, or None for a refused sequence."""
    out = []
    for L, n in zip(lens, counts):
        if not (L >= 0 and L + n <= capacity):
            n = 0  # an inject that does not fit appends nothing
        start = L + n
        end = start + bs
        lo = max(0, start - window + 1) if window > 0 else 0
        lo -= lo % align
        ok = start >= 0 and end <= capacity
        out += [(lo, end) if ok else None] * n_kv
    return out


def _check(wl, ranges):
    n_ctas, max_splits, B = wl["n_ctas"], wl["max_splits"], wl["item_cost"]
    first, items, splits = wl["first"], wl["items"], wl["splits"]
    n_items = int(first[n_ctas])
    assert len(items) == n_ctas + n_items
    lst = items[n_ctas:]
    # each CTA a contiguous run of the list; its first slot holds the run's last item
    assert first[0] == 0 and np.all(np.diff(first) >= 0)
    owner = np.full(n_items, -1)
    for c in range(n_ctas):
        run = lst[first[c]:first[c + 1]]
        owner[first[c]:first[c + 1]] = c
        if len(run):
            assert np.array_equal(items[c], run[-1])
        else:
            assert items[c][0] == -1
    assert np.all(owner >= 0)
    # every pair covered once, in order, by whole tiles
    by_pair = {}
    for it in lst:
        by_pair.setdefault(int(it[0]), []).append(it)
    for pr, rng in enumerate(ranges):
        its = sorted(by_pair.get(pr, []), key=lambda x: x[1])
        if rng is None:
            assert splits[pr] == 0 and not its
            continue
        lo, end = rng
        n = len(its)
        assert n == splits[pr] and 1 <= n <= max_splits
        assert its[0][1] == lo and its[-1][2] == end
        for a, b in zip(its, its[1:]):
            assert a[2] == b[1] and (b[1] - lo) % TK == 0
        for it in its:
            assert it[2] > it[1]
        assert [int(it[3]) for it in its] == ([-1] if n == 1 else list(range(n)))
    # the combine's pairs: split or refused, with their item counts
    want = {pr | (int(splits[pr]) << 20) for pr in range(len(ranges)) if splits[pr] != 1}
    assert set(int(v) for v in wl["merge_list"]) == want and len(wl["merge_list"]) == len(want)
    # balance of the cost stream (only where ranges may be cut)
    if max_splits >= 2:
        tiles = (lst[:, 2] - lst[:, 1] + TK - 1) // TK
        cost = np.zeros(n_ctas)
        np.add.at(cost, owner, TILE_COST * tiles + B)
        used = cost > 0
        W = sum(B + TILE_COST * -(-(e - lo) // TK) for r in ranges if r is not None for lo, e in [r])
        share = W / used.sum()
        # a CTA's tile centres fall in its share; its cut ends add up to two item headers
        assert cost.max() <= share + TILE_COST + 2 * B + 1, (cost.max(), share)
        return cost[used]
    return None


def test_serving_lengths():
    rng = np.random.default_rng(0)
    lens = rng.integers(256, 4097, 32)
    counts = np.full(32, 16)
    _, wl = _case(32, 8, 4160, lens, counts)
    ranges = _expected_ranges(lens, counts, 4160, 16, 0, 8, 1)
    cost = _check(wl, ranges)
    # every SM has a share of the serving workload
    assert wl["n_ctas"] == int((cost > 0).sum())


@pytest.mark.parametrize("window", [64, 2048])
def test_sliding_windows(window):
    rng = np.random.default_rng(1)
    lens = rng.integers(0, 8200, 64)
    counts = rng.integers(1, 17, 64)
    _, wl = _case(64, 8, 8256, lens, counts, window=window)
    _check(wl, _expected_ranges(lens, counts, 8256, 16, window, 8, 1))


def test_long_context_ranges_stay_within_max_splits():
    lens = np.array([32768, 30000, 1000, 16])
    counts = np.array([16, 16, 16, 16])
    _, wl = _case(4, 8, 32832, lens, counts)
    _check(wl, _expected_ranges(lens, counts, 32832, 16, 0, 8, 1))


def test_batch_one_uses_few_ctas():
    lens, counts = np.array([1024]), np.array([16])
    _, wl = _case(1, 8, 1088, lens, counts)
    cost = _check(wl, _expected_ranges(lens, counts, 1088, 16, 0, 8, 1))
    assert len(cost) < wl["n_ctas"]  # shares of at least two tiles


def test_paged_cache_ranges_start_on_pages():
    rng = np.random.default_rng(2)
    lens = rng.integers(0, 1900, 12)
    counts = rng.integers(0, 17, 12)
    _, wl = _case(12, 2, 2048, lens, counts, window=300, paged=True)
    _check(wl, _expected_ranges(lens, counts, 2048, 16, 300, 2, 128))


def test_refused_sequences_and_injects_that_do_not_fit():
    # sequence 1: the block does not fit (refused); sequence 3: its inject does not fit
    # (nothing appended), but the block does
    lens = np.array([100, 1020, 0, 1000, 513])
    counts = np.array([16, 0, 5, 40, 16])
    _, wl = _case(5, 2, 1024, lens, counts)
    ranges = _expected_ranges(lens, counts, 1024, 16, 0, 2, 1)
    assert ranges[2] is None and ranges[6] is not None
    _check(wl, ranges)


def test_ranges_are_never_cut_with_one_item_per_range():
    # capacity <= 512: one item per range at most; each range goes whole to one CTA
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 480, 40)
    counts = rng.integers(0, 17, 40)
    _, wl = _case(40, 4, 512, lens, counts)
    assert wl["max_splits"] == 1
    _check(wl, _expected_ranges(lens, counts, 512, 16, 0, 4, 1))
