"""dflash_layer_out and dflash_rms_norm against the float64 oracle, element by element.

The residual stream, stand-in attention rows and all weights come from the seeded
generators (already rounded to the storage type); the oracle runs on the same values.
A chained case feeds dflash_block_attn's output rows into the layer output.
"""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from speculative_decoding_draft_dflash_gb300 import synth
import harness

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

CASES = {
    # bf16: 3 sequences x 16 rows (48 rows, one partial M tile), random gammas
    "bf16_small": W["serve_b32"].replace(name="lo_bf16_small", d=256, n_h=4, n_kv=2, k=1,
                                         batch=3, n_layers=1, windows=(0,), d_ff=384, seed=31,
                                         random_gamma=True),
    # bf16: 10 sequences (160 rows: two M tiles, the second ragged), wider layer
    "bf16_wide": W["serve_b32"].replace(name="lo_bf16_wide", d=1024, n_h=8, n_kv=2, k=1,
                                        batch=10, n_layers=1, windows=(0,), d_ff=3072, seed=32),
    # f32: the walkthrough-sized layer
    "f32": W["walkthrough_f32"].replace(name="lo_f32", batch=2, d_ff=40, seed=33,
                                        random_gamma=True),
}


def _dev(a, w):
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dt)


def _run_layer_out(w, attn, x, layer=0, alias=False):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    M = attn.shape[0]
    args = [_dev(a, w) for a in (synth.W_O(w, layer), synth.gamma_post(w, layer),
                                 synth.W_gate(w, layer), synth.W_up(w, layer),
                                 synth.W_down(w, layer))]
    ta, tx = _dev(attn, w), _dev(x, w)
    out = tx if alias else torch.empty_like(tx)
    ws = torch.empty(D.dflash_layer_out_workspace_bytes(dims, M, w.ffn), dtype=torch.uint8,
                     device="cuda")
    D.dflash_layer_out(dims, M, ta, tx, args[0], args[1], w.ffn, args[2], args[3], args[4], out, ws)
    assert D.dflash_status_get() == 0
    return out.float().cpu().numpy()


def _oracle(w, attn, x, layer=0):
    return O.layer_output(x, attn, synth.W_O(w, layer), synth.gamma_post(w, layer),
                          synth.W_gate(w, layer), synth.W_up(w, layer), synth.W_down(w, layer),
                          w.eps)


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_out_matches_oracle(name):
    w = CASES[name]
    attn = synth.attn_rows(w, 1, 0)
    x = synth.residual(w, 1, 0)
    got = _run_layer_out(w, attn, x)
    harness.check_close(got, _oracle(w, attn, x), w.dtype, f"{name} layer output")


def test_layer_out_in_place():
    """x_out may be x: the residual is read before the output is written."""
    w = CASES["bf16_small"]
    attn, x = synth.attn_rows(w, 2, 0), synth.residual(w, 2, 0)
    got = _run_layer_out(w, attn, x, alias=True)
    harness.check_close(got, _oracle(w, attn, x), w.dtype, "in-place layer output")


def test_layer_out_after_block_attention():
    """Chained: the block attention's output rows feed the layer output."""
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload
    w = CASES["bf16_small"]
    L0 = synth.prefill_lens(w)
    res, dev = harness.device_rounds(w, list(range(w.batch)), rounds=1)
    ref = harness.oracle_rounds(w, list(range(w.batch)), rounds=1)
    attn_dev = dev.out[0].float().cpu().numpy().reshape(w.batch * w.bs, -1)
    attn_ref = np.concatenate([ref[0]["out"][0][b] for b in range(w.batch)], axis=0)
    x = synth.residual(w, 1, 0)
    got = _run_layer_out(w, attn_dev, x)
    harness.check_close(got, _oracle(w, attn_ref.reshape(w.batch * w.bs, -1), x), w.dtype,
                        "chained layer output")


@pytest.mark.parametrize("name", ["bf16_small", "f32"])
def test_rms_norm_matches_oracle(name):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = CASES[name]
    x = synth.residual(w, 3, 0)
    g = synth.gamma_post(w, 0)
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    tx, tg = _dev(x, w), _dev(g, w)
    out = torch.empty_like(tx)
    D.dflash_rms_norm(dims, x.shape[0], tx, tg, out)
    torch.cuda.synchronize()
    harness.check_close(out.float().cpu().numpy(), O.rms_norm(x, g, w.eps), w.dtype, "rms_norm")
