"""Device (C ABI) against the float64 oracle, element by element, on seeded inputs.

Small workloads run every sequence through the oracle; the full-size workloads
run the same launch configuration as the benchmark and check a seeded sample
of sequences (every output row depends on its own sequence only).
"""
import numpy as np
import pytest

from speculative_decoding_draft_dflash_gb300 import synth
import harness

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

SMALL = {
    # G = 4, two layers (one windowed at 64), several 256-key chunks with ragged tails,
    # an empty cache (length 0) among them, random gammas.
    "small_gqa_bf16": W["serve_b32"].replace(
        name="small_gqa_bf16", d=512, n_h=8, n_kv=2, k=2, batch=4, n_layers=2, windows=(0, 64),
        prefill_lo=0, prefill_hi=700, seed=3, random_gamma=True),
    # G = 1 (MHA), odd block size, prefill by projection + inject of real rows.
    "small_mha_bf16": W["qwen3_8b_b1"].replace(
        name="small_mha_bf16", d=256, n_h=4, n_kv=4, k=1, bs=5, batch=2, prefill_lo=300,
        prefill_hi=300, new_ctx=7, rounds=2, seed=4, random_gamma=True),
    # G = 8, block of 16 -> 128 stacked query rows; block size 1 in the f32 variant below.
    "small_g8_bf16": W["serve_b32"].replace(
        name="small_g8_bf16", d=256, n_h=16, n_kv=2, k=3, batch=3, n_layers=1, windows=(16,),
        prefill_lo=1, prefill_hi=513, seed=5),
    # One sequence at a width whose K allows four splits: each layer's two projections run
    # as one split-K launch (layer modes "split" and the default); the prefill by
    # projection + inject (200 rows, more than that launch takes) as two calls; round 2
    # injects a_i rows
    "small_b1_bf16": W["qwen3_8b_b1"].replace(
        name="small_b1_bf16", d=1024, n_h=8, n_kv=2, k=2, batch=1, n_layers=2, windows=(0, 64),
        prefill_lo=200, prefill_hi=200, rounds=2, seed=10, random_gamma=True),
    # One sequence injecting 100 context rows: the split-K grouping with more context rows
    # than block rows (both within one 128-row tile)
    "small_b1_inject100_bf16": W["qwen3_8b_b1"].replace(
        name="small_b1_inject100_bf16", d=1024, n_h=8, n_kv=2, k=2, batch=1, n_layers=1,
        windows=(0,), prefill_lo=300, prefill_hi=300, prefill_inject=False, new_ctx=100,
        rounds=1, seed=12),
    "small_gqa_f32": W["walkthrough_f32"].replace(
        name="small_gqa_f32", d=96, n_h=6, n_kv=2, d_h=32, k=2, bs=3, batch=3, n_layers=2,
        windows=(0, 5), prefill_lo=0, prefill_hi=600, new_ctx=4, rounds=2, seed=6,
        random_gamma=True),
    # 20 sequences: 320 block rows and 320 context rows in round 1, so the projections run
    # on CTA pairs (three 128-row tiles: the second pair's odd CTA holds no rows); round 2
    # injects a_i rows, a ragged M
    "small_pairs_bf16": W["serve_b32"].replace(
        name="small_pairs_bf16", d=256, n_h=4, n_kv=2, k=2, batch=20, n_layers=1, windows=(0,),
        prefill_lo=0, prefill_hi=400, seed=8, random_gamma=True),
    "small_bs1_f32": W["walkthrough_f32"].replace(
        name="small_bs1_f32", d=64, n_h=2, n_kv=1, d_h=64, k=1, bs=1, batch=2, n_layers=1,
        windows=(0,), prefill_lo=255, prefill_hi=257, new_ctx=1, rounds=2, seed=7),
}


def _run(w, seqs, fused_layer=True, paged=False):
    dev_res, dev = harness.device_rounds(w, seqs, fused_layer=fused_layer, paged=paged)
    ora_res = harness.oracle_rounds(w, seqs)
    return harness.compare(w, dev_res, ora_res, seqs)


def test_walkthrough_f32():
    """The walkthrough's example end to end: lengths 0 -> 3 -> 7 -> 3 -> 6 -> 10 -> 6."""
    w = W["walkthrough_f32"]
    _run(w, [0])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workloads(name, layer_mode):
    w = SMALL[name]
    _run(w, list(range(w.batch)), fused_layer=layer_mode)


@pytest.mark.parametrize("name", sorted(n for n in SMALL if SMALL[n].dtype == "bf16"))
def test_small_workloads_paged(name, layer_mode):
    """The same schedules on a paged cache: 128-row pages in a seeded permutation."""
    w = SMALL[name]
    _run(w, list(range(w.batch)), fused_layer=layer_mode, paged=True)


def _sample(w, n, seed=11):
    L = synth.prefill_lens(w)
    picks = {int(np.argmin(L)), int(np.argmax(L))}
    rng = np.random.default_rng(seed)
    while len(picks) < min(n, w.batch):
        picks.add(int(rng.integers(0, w.batch)))
    return sorted(picks)


@pytest.mark.slow
@pytest.mark.parametrize("name,n", [("qwen3_8b_b1", 1), ("serve_b32", 4), ("long_ctx_b4", 2),
                                    ("hybrid_swa_b64", 3)])
def test_full_size(name, n):
    w = W[name]
    _run(w, _sample(w, n))


@pytest.mark.slow
@pytest.mark.parametrize("name,n", [("serve_b32", 3), ("hybrid_swa_b64", 2)])
def test_full_size_paged(name, n):
    w = W[name]
    _run(w, _sample(w, n, seed=12), paged=True)


# fp8 (E4M3) cache: the GQA (NARROW tile) case with a window, the MHA case with an odd
# block and a prefill by projection + inject, the G = 8 case (128 query rows, WIDE), and
# the one-sequence case
FP8 = {n.replace("bf16", "fp8"): SMALL[n].replace(name=n.replace("bf16", "fp8"), kv="fp8")
       for n in ("small_gqa_bf16", "small_mha_bf16", "small_g8_bf16", "small_b1_bf16")}


@pytest.mark.parametrize("name", sorted(FP8))
def test_small_workloads_fp8(name, layer_mode):
    w = FP8[name]
    _run(w, list(range(w.batch)), fused_layer=layer_mode)


@pytest.mark.parametrize("name", sorted(FP8))
def test_small_workloads_fp8_paged(name):
    w = FP8[name]
    _run(w, list(range(w.batch)), paged=True)


@pytest.mark.slow
@pytest.mark.parametrize("name,n,paged", [("serve_b32", 3, False), ("long_ctx_b4", 1, False),
                                          ("hybrid_swa_b64", 2, True)])
def test_full_size_fp8(name, n, paged):
    w = W[name].replace(kv="fp8")
    _run(w, _sample(w, n, seed=13), paged=paged)



@pytest.mark.parametrize("name", ["small_gqa_bf16", "small_g8_bf16"])
def test_output_16_byte_aligned(name):
    """Output buffers that are 16-byte but not 32-byte aligned (all the API asks for) take
    the attention's 16-byte store path for whole-range rows: same results."""
    import torch
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload
    w = SMALL[name]
    dev = DeviceWorkload(w)
    n = w.batch * w.bs * w.n_h * w.d_h
    views = []
    for _ in range(w.n_layers):
        buf = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
        v = buf[8:8 + n].view(w.batch, w.bs, w.n_h * w.d_h)
        assert v.data_ptr() % 32 == 16
        views.append(v)
    dev.out = views
    seqs = list(range(w.batch))
    dev_res, _ = harness.device_rounds(w, seqs, dev=dev)
    harness.compare(w, dev_res, harness.oracle_rounds(w, seqs), seqs)


@pytest.mark.parametrize("pairs", ["0", "1"])
def test_single_and_paired_projection_tiles(pairs, monkeypatch):
    """The projections on single-CTA tiles (DFLASH_PAIR_GEMM=0) and on CTA pairs give the
    same results at shapes where both apply (M > 128 rows)."""
    monkeypatch.setenv("DFLASH_PAIR_GEMM", pairs)
    w = SMALL["small_pairs_bf16"]
    _run(w, list(range(w.batch)))


@pytest.mark.parametrize("fused", ["0", "1"])
@pytest.mark.parametrize("name", ["small_pairs_bf16", "small_gqa_bf16"])
def test_fused_and_separate_hidden_norm(name, fused, monkeypatch):
    """hidden_norm in the fc epilogue (DFLASH_FUSED_NORM=1, where the launch fits) and as a
    separate pass over the split partials (the default): the same C and round results, on
    CTA pairs with 2 K-splits (320 rows) and on single CTAs with 4 splits (64 rows)."""
    monkeypatch.setenv("DFLASH_FUSED_NORM", fused)
    w = SMALL[name]
    _run(w, list(range(w.batch)))


def test_fused_hidden_norm_at_serving_and_prefill_widths(monkeypatch):
    """The fused norm at full width (d = 4096, k = 5): 512 rows on CTA pairs with 2 K-splits
    and 1024 rows with one split, against the oracle row by row on a sample of rows."""
    import torch
    from oracle import dflash_oracle as O
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    monkeypatch.setenv("DFLASH_FUSED_NORM", "1")
    w = W["qwen3_8b_b1"]
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    W_fc_np, g_np = synth.W_fc(w), synth.gamma_h(w)
    W_fc = torch.from_numpy(W_fc_np).to("cuda", torch.bfloat16)
    g_h = torch.from_numpy(g_np).to("cuda", torch.bfloat16)
    for M in (512, 1024):
        hid_np = synth.hidden_states(w, 3, np.full(1, M, dtype=np.int64))
        hid = [torch.from_numpy(h).to("cuda", torch.bfloat16) for h in hid_np]
        C = torch.full((M, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(D.dflash_workspace_bytes(dims, 1, 64, M), dtype=torch.uint8,
                         device="cuda")
        D.dflash_ctx_project(dims, hid, M, W_fc, g_h, C, ws)
        assert D.dflash_status_get() == 0
        rows = np.unique(np.r_[0, 127, 128, M - 1, np.random.default_rng(M).integers(0, M, 12)])
        ref = O.ctx_project([h[rows] for h in hid_np], W_fc_np, g_np, w.eps)
        harness.check_close(C.float().cpu().numpy()[rows], ref, w.dtype, f"C rows, M={M}")
