"""dflash_accept against the oracle's round bookkeeping, bit for bit (integers).

Token ids are seeded; each sequence's accepted length is drawn first and the posterior
is built to match exactly that many leading positions, so every length 0 .. bs-1 occurs.
"""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


def _case(batch, bs, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    block = rng.integers(0, 1000, size=(batch, bs), dtype=np.int64)
    post = rng.integers(0, 1000, size=(batch, bs), dtype=np.int64)
    a = rng.integers(0, bs, size=batch)
    for b in range(batch):
        post[b, :a[b]] = block[b, 1:a[b] + 1]
        if a[b] < bs - 1 and post[b, a[b]] == block[b, a[b] + 1]:
            post[b, a[b]] = (block[b, a[b] + 1] + 1) % 1000    # force the first miss
    ctx = rng.integers(0, 5000, size=batch, dtype=np.int64)
    return block, post, ctx


def _device(block, post, ctx):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()  # noqa: E731
    B = block.shape[0]
    bt, pt, ct = dev(block), dev(post), dev(ctx)
    if B == 0:
        bt = torch.zeros((0, block.shape[1]), dtype=torch.int32, device="cuda")
        pt = bt.clone()
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    cu = torch.full((B + 1,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    anc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    D.dflash_accept(bt, pt, ct, acc, cu, nxt, anc)
    torch.cuda.synchronize()
    return [t.cpu().numpy().tolist() for t in (acc, cu, nxt, anc)]


@pytest.mark.parametrize("batch,bs,seed", [(1, 4, 0), (37, 16, 1), (3000, 16, 2), (5, 1, 3),
                                           (64, 5, 4), (1025, 2, 5)])
def test_accept_matches_oracle(batch, bs, seed):
    block, post, ctx = _case(batch, bs, seed)
    got = _device(block, post, ctx)
    want = O.round_bookkeeping(block.tolist(), post.tolist(), ctx.tolist())
    assert got[0] == list(want[0])
    assert got[1] == list(want[1])
    assert got[2] == list(want[2])
    assert got[3] == list(want[3])


def test_accept_walkthrough_example():
    """["on", "the", "mat", "."] against ["the", "mat", "in", <next>]: a = 2, start 3 -> 6."""
    ids = {"on": 1, "the": 2, "mat": 3, ".": 4, "in": 5, "<next>": 6}
    block = np.array([[ids[t] for t in ("on", "the", "mat", ".")]])
    post = np.array([[ids[t] for t in ("the", "mat", "in", "<next>")]])
    acc, cu, nxt, anc = _device(block, post, np.array([3]))
    assert acc == [2] and cu == [0, 3] and nxt == [6] and anc == [ids["in"]]


def test_accept_empty_batch():
    block = np.zeros((0, 4), dtype=np.int64)
    acc, cu, nxt, anc = _device(block, block, np.zeros(0, dtype=np.int64))
    assert cu == [0] and acc == [] and nxt == [] and anc == []
