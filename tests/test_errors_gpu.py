"""Device-side error paths: capacity overflow, crop beyond the length, empty inputs."""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_dflash_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(w, **kw):
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload
    return DeviceWorkload(w, **kw)


def _tiny(kv="bf16"):
    return synth.WORKLOADS["serve_b32"].replace(
        name="tiny", d=512, n_h=4, n_kv=2, k=1, batch=3, n_layers=1, windows=(0,),
        prefill_lo=10, prefill_hi=60, rounds=1, seed=9, kv=kv)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_capacity_overflow_skips_sequence_and_flags(layer_mode, kv):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = _tiny(kv)
    L0 = synth.prefill_lens(w)
    cap = int(L0.max()) + 10          # the longest sequence cannot take its 16 context rows
    dev = _dev(w, capacity=cap)
    assert D.dflash_status_get() == 0
    x = dev.round_inputs(1, L0)
    dev.run_round(x, crop=False, fused_layer=layer_mode)
    st = D.dflash_status_get()
    assert st & D.DEV_CAPACITY
    lens = dev.cache.lens.cpu().numpy()[0]
    n_refused = 0
    for b in range(w.batch):
        after_inject = L0[b] + 16 if L0[b] + 16 <= cap else L0[b]
        block_ok = after_inject + 16 <= cap
        assert lens[b] == after_inject + (16 if block_ok else 0)
        if not block_ok:
            n_refused += 1
            assert torch.all(dev.out[0][b] == 0)         # skipped rows are zero
    assert n_refused >= 1
    assert D.dflash_status_get() == 0                    # read clears the word


def test_crop_beyond_length_refused():
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = _tiny()
    dev = _dev(w)
    L0 = synth.prefill_lens(w)
    bad = torch.tensor(L0 + np.array([1, 0, -1]), dtype=torch.int32, device="cuda")
    D.dflash_cache_crop(dev.cache, bad)
    st = D.dflash_status_get()
    assert st == D.DEV_CROP
    lens = dev.cache.lens.cpu().numpy()[0]
    assert lens.tolist() == [L0[0], L0[1], L0[2] - 1]
    neg = torch.tensor([-1, 0, 0], dtype=torch.int32, device="cuda")
    D.dflash_cache_crop(dev.cache, neg)
    assert D.dflash_status_get() == D.DEV_CROP
    assert dev.cache.lens.cpu().numpy()[0].tolist() == [L0[0], 0, 0]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_rope_table_too_short_flags(layer_mode, kv):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = _tiny(kv)
    dev = _dev(w)
    L0 = synth.prefill_lens(w)
    x = dev.round_inputs(1, L0)
    dev.table_len = int(L0.min()) + 8     # positions beyond the table for every sequence
    dev.run_round(x, crop=False, fused_layer=layer_mode)
    assert D.dflash_status_get() & D.DEV_ROPE
    assert dev.cache.lens.cpu().numpy()[0].tolist() == L0.tolist()


def test_empty_inject_is_noop():
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = _tiny()
    dev = _dev(w)
    before = dev.cache.lens.clone()
    cu = torch.zeros(w.batch + 1, dtype=torch.int32, device="cuda")
    D.dflash_kv_inject(dev.dims, dev.cache, 0, dev.C, cu, 0, dev.W_K[0], dev.W_V[0], dev.g_k[0],
                       dev.rope, dev.table_len, dev.ws)
    torch.cuda.synchronize()
    assert torch.equal(before, dev.cache.lens)
    assert D.dflash_status_get() == 0


def test_ragged_inject_with_empty_sequences():
    """A sequence with no new rows keeps its length; rows land after each sequence's length."""
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    import harness
    from oracle import dflash_oracle as O
    w = _tiny()
    dev = _dev(w)
    L0 = synth.prefill_lens(w)
    counts = np.array([0, 5, 2])
    x = dev.round_inputs(1, L0, counts=counts)
    C = dev.C[:x.M]
    D.dflash_ctx_project(dev.dims, x.hidden, x.M, dev.W_fc, dev.g_h, C, dev.ws)
    D.dflash_kv_inject(dev.dims, dev.cache, 0, C, x.cu_rows, x.M, dev.W_K[0], dev.W_V[0],
                       dev.g_k[0], dev.rope, dev.table_len, dev.ws)
    assert D.dflash_status_get() == 0
    lens = dev.cache.lens.cpu().numpy()[0]
    assert lens.tolist() == (L0 + counts).tolist()
    Cref = O.ctx_project(synth.hidden_states(w, 1, counts), synth.W_fc(w), synth.gamma_h(w), w.eps)
    harness.check_close(C.float().cpu().numpy(), Cref, w.dtype, "C")
    cu = synth.cu_rows(counts)
    for b in range(w.batch):
        if counts[b] == 0:
            continue
        K, V = O.kv_project(Cref[cu[b]:cu[b + 1]], synth.W_K(w, 0), synth.W_V(w, 0),
                            synth.gamma_k(w, 0), w.n_kv, w.d_h, w.eps,
                            L0[b] + np.arange(counts[b]), w.theta)
        gk = dev.cache.rows("k", 0, b, L0[b], L0[b] + counts[b]).float().cpu().numpy()
        gv = dev.cache.rows("v", 0, b, L0[b], L0[b] + counts[b]).float().cpu().numpy()
        harness.check_close(gk, K, w.dtype, f"K seq {b}")
        harness.check_close(gv, V, w.dtype, f"V seq {b}")


def test_fp8_refused_rows_leave_cache_untouched():
    """A refused append writes no code: the fp8 cache bytes past a refused sequence's
    length keep their previous content (the zeros the cache was created with)."""
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = _tiny("fp8")
    L0 = synth.prefill_lens(w)
    cap = int(L0.max()) + 10
    dev = _dev(w, capacity=cap)
    x = dev.round_inputs(1, L0)
    dev.run_round(x, crop=False)
    assert D.dflash_status_get() & D.DEV_CAPACITY
    b = int(np.argmax(L0))
    tail = dev.cache.k[0, b, :, int(L0[b]):]
    assert torch.all(tail == 0)


def test_pipeline_wait_that_runs_out_returns_with_status():
    """A pipeline wait that runs out: with the test aid's limit at 1 ns, the context
    projection's GEMM (16 rows: single-CTA tiles, nine K-splits) gives up at its first
    stage wait. Each CTA drains the copies and MMAs it issued, frees its tensor memory and
    returns; the status word reports DFLASH_DEV_TIMEOUT. With the default limit back, the
    next calls on the same GPU (the projection again, then a whole round) are correct."""
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    import harness
    from oracle import dflash_oracle as O
    w = synth.WORKLOADS["qwen3_8b_b1"]
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    M = 16
    counts = np.full(1, M, dtype=np.int64)
    hid_np = synth.hidden_states(w, 1, counts)
    hid = [torch.from_numpy(h).to("cuda", torch.bfloat16) for h in hid_np]
    W_fc = torch.from_numpy(synth.W_fc(w)).to("cuda", torch.bfloat16)
    g_h = torch.from_numpy(synth.gamma_h(w)).to("cuda", torch.bfloat16)
    C = torch.empty((M, w.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(D.dflash_workspace_bytes(dims, 1, 64, M), dtype=torch.uint8, device="cuda")
    assert D.dflash_status_get() == 0
    st = 0
    try:
        D.dflash_test_wait_limit(1)
        for _ in range(3):               # the first stage of some CTA takes more than 1 ns
            D.dflash_ctx_project(dims, hid, M, W_fc, g_h, C, ws)
            st |= D.dflash_status_get()
            if st & D.DEV_TIMEOUT:
                break
    finally:
        D.dflash_test_wait_limit(0)
    assert st & D.DEV_TIMEOUT
    C.fill_(float("nan"))
    D.dflash_ctx_project(dims, hid, M, W_fc, g_h, C, ws)
    assert D.dflash_status_get() == 0
    ref = O.ctx_project(hid_np, synth.W_fc(w), synth.gamma_h(w), w.eps)
    harness.check_close(C.float().cpu().numpy(), ref, w.dtype, "C after a timed-out launch")
    # a whole draft round (grouped projections, attention, combine) on the same GPU
    t = _tiny()
    seqs = list(range(t.batch))
    dev_res, _ = harness.device_rounds(t, seqs)
    harness.compare(t, dev_res, harness.oracle_rounds(t, seqs), seqs)
